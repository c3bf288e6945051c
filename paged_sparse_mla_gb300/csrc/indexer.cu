// smla_index_scores: indexer scores of each query token over its visible context.
//
// [AgentX "DeepSeek V4"]: the indexer has 64 heads but yields a single global
// top-k selection per token.  [GLM-5.3 "What is new"]: the indexer scans the
// whole context (quadratic cost) to choose 2,048 tokens.
//
//   I[t, j] = s_I[j] * sum_h w[t, h] * ReLU(q_I[t, h] . k_I[j])
//
// Design (sm_103a, one persistent CTA per SM):
//   * a work item is (sequence b, group g of <= 4 query tokens of b, key chunk c
//     of 2048 keys); the valid items are enumerated densely (prefix sums over
//     the sequences, in shared memory) and dealt round-robin to the CTAs, so
//     every CTA gets the same number of tiles to within one item, and CTAs that
//     run at the same time work on neighbouring sequences (prefix-shared blocks
//     are read once from HBM and then from L2);
//   * the contraction is one FP8 tcgen05.mma per 32 key dims with the 128 keys
//     of a tile as M (TMEM lane = key) and the group's query heads as N
//     (<= 4 tokens x 64 heads = 256), accumulated in fp32 in tensor memory,
//     double-buffered;
//   * warps 0-15 (epilogue; warp w reads TMEM lanes 32*(w%4).. for query token
//     w/4) hold their token's head weights in registers for the whole item and
//     reduce sum_h w * ReLU(.) per key in registers -- no cross-thread
//     reduction -- then scale by s_I[j] and store the fp32 score;
//   * warp 16 (producer) moves data with the tensor-memory-access unit: one 3-D
//     tensor-map load per block of the indexer-key region (block ids from the
//     block table, the MMA's swizzle applied by the copy, blocks beyond the
//     context loaded out of bounds as zeros), a bulk copy of the block's key
//     scales, and per item a 2-D tensor-map load of the group's query rows and a
//     bulk copy of its weights; completion is counted in transaction bytes on
//     the stage's mbarrier;
//   * warp 17 issues the MMAs and owns the tensor-memory allocation.
//
// FP4 keys ([AgentX "Hybrid KV cache management"]: the FP4 indexer shrinks the
// packed block): the pool holds each key as 128 packed E2M1 codes (64 bytes).
// The key copy uses the tensor map's 4-bit unpacking type, which places every
// 16 codes (8 bytes) at the start of a 16-byte shared-memory chunk, the other
// 8 bytes being padding -- the layout tcgen05.mma.kind::f8f6f4 reads 4-bit
// operands in -- so
// the key tile keeps the 128-byte rows and swizzle of the E4M3 tile, and the
// MMA takes E2M1 keys (A) times E4M3 queries (B) at the FP8 rate while the key
// stream from HBM is halved.
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kTile = 128;         // keys per tile (MMA M)
constexpr int kGroup = 4;          // query tokens per item (MMA N = kGroup * n_idx_heads)
constexpr int kStages = 8;         // key-tile ring
constexpr int kChunkTiles = 16;    // tiles per work item (2048 keys)
constexpr int kEpiWarps = 16;      // four warps per TMEM sub-partition, one query token each
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = 32 * (kEpiWarps + 4);  // warpgroup 4: producer, MMA issuer, two idle warps
// Register split: the launch gives every thread kLaunchRegs (five warps per SM sub-partition);
// setmaxnreg then moves registers from warpgroup 4 to the epilogue warpgroups.
constexpr int kLaunchRegs = 96;
constexpr int kEpiRegs = 104;
constexpr int kOtherRegs = 56;
static_assert(32 * kEpiWarps * kEpiRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs, "register split exceeds the launch");
constexpr int kMaxN = 256;         // MMA N limit
// Transaction bytes a 4-bit-unpacking key copy completes on its mbarrier: the packed bytes it
// reads from global memory (half of the shared-memory bytes it fills; measured on GB300).  The
// padding half of each 16-byte chunk is left as it was; the MMA does not read it.
constexpr bool kUnpackTxIsSmemBytes = false;
// Instruction-descriptor operand formats of kind::f8f6f4.
constexpr int kFmtE4M3 = 0;
constexpr int kFmtE2M1 = 5;
constexpr int kMaxSeqSmem = 1024;  // batches up to this size are scheduled densely

struct __align__(1024) IdxSmem {
  uint8_t keys[kStages][kTile * 128];   // 16 KB per stage, 1024-aligned
  uint8_t q[2][kMaxN * 128];            // 32 KB per buffer
  float kscale[kStages][kTile];         // s_I of the tile's keys, loaded with the keys
  float4 w[2][kGroup * 64 / 4];         // weights of the item whose q is in q[i]
  int seq_meta[2 * kMaxSeqSmem + 1];     // query_start_loc[0..B], then seq_lens[0..B)
  int item_off[kMaxSeqSmem + 1];         // first dense work item of each sequence (prefix sum)
  int chunks[kMaxSeqSmem];               // key chunks of each sequence's last query group
  uint64_t key_full[kStages], key_empty[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t final_bar;
  uint32_t tmem_slot;
  int abort;
};

struct Item {
  int valid;
  int b;          // sequence
  int t0;         // first query token (absolute row)
  int n_grp;      // tokens in the group
  int p_first;    // position of the first token of the group
  int key_begin;  // first key of the chunk
  int key_end;    // one past the last key needed (p_last + 1, chunk-bounded)
  int n_tiles;
};

struct IdxArgs {
  KernelLayout L;
  int n_idx_heads, layer;
  const uint8_t* pool;
  const float* w;
  const int32_t* block_table;
  int bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int batch, tok_begin, tok_end, n_groups, n_chunks;
  float* scores;
  int64_t scores_stride;
  unsigned* err;
};


// Shared-memory matrix descriptor for K-major rows of kD bytes: the 128-byte
// swizzle for 128-byte rows, the 32-byte swizzle for 32-byte rows; 8-row groups.
template <int kD>
__device__ __forceinline__ uint64_t key_desc(uint32_t addr) {
  if constexpr (kD == 128) {
    return sw128_desc(addr, 16, 1024);
  } else {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1) << 16;              // leading offset (unused for swizzled K-major)
    d |= static_cast<uint64_t>((8 * kD) >> 4) << 32;  // 8 rows of kD bytes
    d |= static_cast<uint64_t>(1) << 46;              // descriptor version for tcgen05
    d |= static_cast<uint64_t>(6) << 61;              // 32-byte swizzle
    return d;
  }
}

// ---------------------------------------------------------------------------
// Work items
// ---------------------------------------------------------------------------
__device__ __forceinline__ Item make_item(const IdxArgs& A, int b, int g, int c, int q0, int q1, int len_b) {
  Item it;
  it.valid = 0;
  const int r0 = max(q0, A.tok_begin), r1 = min(q1, A.tok_end);  // this call's rows of sequence b
  const int first = r0 + g * kGroup;
  if (first >= r1) return it;
  const int n_grp = min(kGroup, r1 - first);
  const int p_first = len_b - (q1 - q0) + (first - q0);
  const int p_last = p_first + n_grp - 1;
  const int key_begin = c * kChunkTiles * kTile;
  if (p_last < 0 || key_begin > p_last) return it;
  const int key_end = min(key_begin + kChunkTiles * kTile, p_last + 1);
  it.valid = 1;
  it.b = b;
  it.t0 = first;
  it.n_grp = n_grp;
  it.p_first = p_first;
  it.key_begin = key_begin;
  it.key_end = key_end;
  it.n_tiles = (key_end - key_begin + kTile - 1) / kTile;
  return it;
}

// Sparse enumeration for large batches: item = (c * batch + b) * n_groups + g.
__device__ __forceinline__ Item decode_sparse(const IdxArgs& A, int item) {
  const int g = item % A.n_groups;
  const int rest = item / A.n_groups;
  const int b = rest % A.batch;
  const int c = rest / A.batch;
  return make_item(A, b, g, c, __ldg(A.qsl + b), __ldg(A.qsl + b + 1), __ldg(A.seq_lens + b));
}

// Dense enumeration (batches up to kMaxSeqSmem): sequence b owns items
// item_off[b] .. item_off[b+1]-1 = (group g, chunk c), c fastest, c < chunks[b].
__device__ __forceinline__ Item decode_dense(const IdxArgs& A, const IdxSmem& sm, int item) {
  int lo = 0, hi = A.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.item_off[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int local = item - sm.item_off[b];
  const int nc = sm.chunks[b];
  return make_item(A, b, local / nc, local % nc, sm.seq_meta[b], sm.seq_meta[b + 1], sm.seq_meta[A.batch + 1 + b]);
}

__device__ __forceinline__ int seq_items(const IdxArgs& A, const int* meta, int b, int& nc) {
  const int q0 = meta[b], q1 = meta[b + 1];
  const int r0 = max(q0, A.tok_begin), r1 = min(q1, A.tok_end);
  const int rows = max(0, r1 - r0);
  const int p_last = meta[A.batch + 1 + b] - (q1 - q0) + (r1 - 1 - q0);
  nc = (rows > 0 && p_last >= 0) ? (p_last + kChunkTiles * kTile) / (kChunkTiles * kTile) : 0;
  return ((rows + kGroup - 1) / kGroup) * nc;
}

// Items per sequence and their prefix sum (one warp).
__device__ void build_item_table(const IdxArgs& A, IdxSmem& sm) {
  const int lane = threadIdx.x & 31;
  const int per = (A.batch + 31) / 32;
  const int b0 = min(A.batch, lane * per), b1 = min(A.batch, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    int nc;
    local += seq_items(A, sm.seq_meta, b, nc);
    sm.chunks[b] = max(nc, 1);
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - local;
  for (int b = b0; b < b1; ++b) {
    sm.item_off[b] = run;
    int nc;
    run += seq_items(A, sm.seq_meta, b, nc);
  }
  if (lane == 31) sm.item_off[A.batch] = incl;
}

// Four heads of one key: acc0 += (v0 + |v0|, v1 + |v1|) * w01 and acc1 += (v2 + |v2|, v3 + |v3|) * w23,
// with packed fp32 pairs.  v + |v| is exactly 2 ReLU(v), so both accumulators carry twice the
// ReLU-weighted sum (a factor of two commutes with rounding) and the caller halves the total.
// Each ReLU pair is one packed add whose second operand is the pair's absolute value.
__device__ __forceinline__ void relu_fma4(uint64_t& acc0, uint64_t& acc1, uint32_t v0, uint32_t v1, uint32_t v2,
                                          uint32_t v3, uint64_t w01, uint64_t w23) {
  asm("{\n\t.reg .f32 a0, a1, b0, b1;\n\t.reg .b64 p, q, pa, qa;\n\t"
      "abs.f32 a0, %2;\n\t"
      "abs.f32 a1, %3;\n\t"
      "abs.f32 b0, %4;\n\t"
      "abs.f32 b1, %5;\n\t"
      "mov.b64 p, {%2, %3};\n\t"
      "mov.b64 q, {%4, %5};\n\t"
      "mov.b64 pa, {a0, a1};\n\t"
      "mov.b64 qa, {b0, b1};\n\t"
      "add.rn.f32x2 p, p, pa;\n\t"
      "add.rn.f32x2 q, q, qa;\n\t"
      "fma.rn.f32x2 %0, p, %6, %0;\n\t"
      "fma.rn.f32x2 %1, q, %7, %1;\n\t}"
      : "+l"(acc0), "+l"(acc1)
      : "r"(v0), "r"(v1), "r"(v2), "r"(v3), "l"(w01), "l"(w23));
}

// mbar_wait's bound for a wait that is usually far from complete and off the critical path (a
// producer several stages ahead of its consumer): a non-blocking test, then a sleep of kSleepNs,
// so that the waiting warp takes few issue slots from the warps of its SM sub-partition.
template <uint32_t kSleepNs>
__device__ __forceinline__ bool mbar_wait_lazy(uint64_t* bar, uint32_t parity, unsigned* err, volatile int* abort) {
  const uint32_t addr = smem_u32(bar);
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    if (ok) return true;
    __nanosleep(kSleepNs);
    if ((i & 15u) == 15u) {
      if (*abort) return false;
      const uint64_t t = globaltimer_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > kWaitLimitNs) {
        latch_error(err, SMLA_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ float pair_sum(uint64_t p) {
  return __uint_as_float(static_cast<uint32_t>(p)) + __uint_as_float(static_cast<uint32_t>(p >> 32));
}

__device__ __forceinline__ int mma_n(int n_grp, int heads) {
  const int n = n_grp * heads;
  return max(16, (n + 15) & ~15);
}

template <int kH, int kD, int kBS, bool kFP4>
__global__ void __launch_bounds__(kThreads, 1)
    index_scores_kernel(const IdxArgs A, const __grid_constant__ CUtensorMap key_map,
                        const __grid_constant__ CUtensorMap q_map) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base, formed by pointer arithmetic on the shared array so that accesses stay shared-space
  IdxSmem& sm = *reinterpret_cast<IdxSmem*>(
      smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u));
  // warp index broadcast from lane 0: the compiler then treats it (and the roles, TMEM addresses
  // and branches derived from it) as warp-uniform
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  constexpr int H = kH;
  constexpr int kBlocks = kTile / kBS;  // blocks per tile
  static_assert(kTile % kBS == 0 && kBlocks <= 32 && kBS % 4 == 0, "tile geometry");
  static_assert(H % 4 == 0 && H * kGroup <= kMaxN, "head geometry");
  static_assert(!kFP4 || kD == 128, "FP4 keys are built for 128-dim keys (128-byte unpacked rows)");
  // shared-memory bytes of one key tile; with FP4 keys the copy reads half of them from global memory
  constexpr uint32_t kKeyTileTx = (kFP4 && !kUnpackTxIsSmemBytes) ? kTile * kD / 2 : kTile * kD;
  const bool dense = A.batch <= kMaxSeqSmem;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.key_full[s], 1);               // producer arrive + transaction bytes
      mbar_init(&sm.key_empty[s], 1 + kEpiWarps);  // MMA done + every epilogue warp read the scales
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1 + kEpiWarps);    // MMA done + every epilogue warp holds its weights
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], kEpiWarps);      // one arrive per epilogue warp
    }
    mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  if (dense) {
    for (int i = threadIdx.x; i <= A.batch; i += kThreads) sm.seq_meta[i] = __ldg(A.qsl + i);
    for (int i = threadIdx.x; i < A.batch; i += kThreads) sm.seq_meta[A.batch + 1 + i] = __ldg(A.seq_lens + i);
    __syncthreads();
    if (warp == 0) build_item_table(A, sm);
  }
  if (warp == kMmaWarp) tmem_alloc(&sm.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  volatile int* abort = &sm.abort;
  const int n_items = dense ? sm.item_off[A.batch] : A.n_chunks * A.batch * A.n_groups;
  const auto item_at = [&](int item) { return dense ? decode_dense(A, sm, item) : decode_sparse(A, item); };

  if (warp == kProducerWarp) {
    // ------------------------------ producer (TMA) ------------------------------
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    const int64_t layer_off = static_cast<int64_t>(A.layer) * A.L.layer_stride;
    // Block-table entries of a whole item (kItemBlocks blocks) are fetched one item ahead:
    // lane l holds the entries of the item's blocks l, l + 32, ... (blocks past the item's
    // last key are not read).  Each tile then takes its kBlocks entries from the owning lanes.
    constexpr int kItemBlocks = kChunkTiles * kBlocks;
    constexpr int kPer = (kItemBlocks + 31) / 32;
    static_assert(32 % kBlocks == 0, "a tile's block entries sit in one register slot");
    const auto fetch_bt = [&](const Item& it, int (&dst)[kPer]) {
      const int32_t* bt = A.block_table + static_cast<int64_t>(it.b) * A.bt_stride;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int key0 = it.key_begin + (lane + 32 * i) * kBS;
        dst[i] = key0 < it.key_end ? __ldg(bt + key0 / kBS) : -1;
      }
    };
    const auto next_valid = [&](int item, Item& it) {
      for (; item < n_items; item += gridDim.x) {
        it = item_at(item);
        if (it.valid) return item;
      }
      return n_items;
    };
    uint32_t k = 0, nq = 0;  // key tiles and query loads issued
    Item cur, nxt;
    int bt_cur[kPer], bt_nxt[kPer];
    int item = next_valid(blockIdx.x, cur);
    if (item < n_items) fetch_bt(cur, bt_cur);
    while (item < n_items && !*abort) {
      const int item_n = next_valid(item + gridDim.x, nxt);
      if (item_n < n_items) fetch_bt(nxt, bt_nxt);  // in flight while this item's tiles are issued
      {
        const int qb = nq & 1;
        if (!mbar_wait(&sm.q_empty[qb], ((nq >> 1) & 1) ^ 1, A.err, abort)) break;
        if (lane == 0) {
          const uint32_t wbytes = static_cast<uint32_t>(cur.n_grp * H * 4);
          mbar_arrive_expect_tx(&sm.q_full[qb], kGroup * H * kD + wbytes);
          tma_load_2d(smem_u32(sm.q[qb]), &q_map, 0, cur.t0 * H, &sm.q_full[qb]);
          bulk_load(smem_u32(&sm.w[qb][0]), A.w + static_cast<int64_t>(cur.t0) * H, wbytes, &sm.q_full[qb]);
        }
        ++nq;
        __syncwarp();
      }
      bool ok = true;
      for (int tile = 0; tile < cur.n_tiles; ++tile, ++k) {
        const int s = k % kStages;
        // lane b < kBlocks: physical block of the tile's b-th block; num_blocks loads zeros
        const int e = tile * kBlocks + (lane % kBlocks);
        const int slot = (tile * kBlocks) / 32;
        int mine_v = bt_cur[0];
#pragma unroll
        for (int i = 1; i < kPer; ++i) mine_v = slot == i ? bt_cur[i] : mine_v;
        const int v = __shfl_sync(0xffffffffu, mine_v, e % 32);
        int blk = static_cast<int>(A.L.num_blocks);
        bool have = false;
        if (lane < kBlocks && cur.key_begin + tile * kTile + lane * kBS < cur.key_end) {
          if (v < 0 || v >= A.L.num_blocks) {
            latch_error(A.err, SMLA_ERR_BAD_INDEX);
          } else {
            blk = v;
            have = true;
          }
        }
        const uint32_t n_have = __popc(__ballot_sync(0xffffffffu, have));
        // the producer runs up to kStages tiles ahead: its wait for a free stage sleeps between tests
        if (!mbar_wait_lazy<256>(&sm.key_empty[s], ((k / kStages) & 1) ^ 1, A.err, abort)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&sm.key_full[s], kKeyTileTx + n_have * kBS * 4);
        __syncwarp();
        if (lane < kBlocks) {
          tma_load_3d(smem_u32(sm.keys[s]) + lane * kBS * kD, &key_map, 0, 0, blk, &sm.key_full[s]);
          if (have)
            bulk_load(smem_u32(&sm.kscale[s][lane * kBS]),
                      A.pool + static_cast<int64_t>(blk) * A.L.block_stride + layer_off + A.L.idx_scale_off,
                      kBS * 4, &sm.key_full[s]);
        }
      }
      if (!ok) break;
      item = item_n;
      cur = nxt;
#pragma unroll
      for (int i = 0; i < kPer; ++i) bt_cur[i] = bt_nxt[i];
    }
    // Leave only after the copies issued last have landed (they have, unless a wait timed out).
    if (lane == 0) {
      for (uint32_t i = 0; i < kStages && i < k; ++i) {
        const uint32_t kk = k - 1 - i;
        mbar_drain(&sm.key_full[kk % kStages], (kk / kStages) & 1);
      }
      for (uint32_t i = 0; i < 2 && i < nq; ++i) {
        const uint32_t qq = nq - 1 - i;
        mbar_drain(&sm.q_full[qq & 1], (qq >> 1) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ------------------------------
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (lane == 0) {
      uint32_t k = 0, nitem = 0, a = 0;
      bool issued = false;
      for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
        const Item it = item_at(item);
        if (!it.valid) continue;
        const int qb = nitem & 1;
        if (!mbar_wait(&sm.q_full[qb], (nitem >> 1) & 1, A.err, abort)) break;
        const int n = mma_n(it.n_grp, H);
        const uint32_t idesc = make_idesc(128, n, kFP4 ? kFmtE2M1 : kFmtE4M3, kFmtE4M3, 0, 0);
        const uint32_t qaddr = smem_u32(sm.q[qb]);
        bool ok = true;
        for (int tile = 0; tile < it.n_tiles; ++tile, ++k, ++a) {
          const int s = k % kStages;
          const int ab = a & 1;
          if (!mbar_wait(&sm.key_full[s], (k / kStages) & 1, A.err, abort) ||
              !mbar_wait(&sm.acc_empty[ab], ((a >> 1) & 1) ^ 1, A.err, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kaddr = smem_u32(sm.keys[s]);
#pragma unroll
          for (int kk = 0; kk < kD / 32; ++kk) {
            mma_f8(tmem + ab * 256, key_desc<kD>(kaddr + kk * 32), key_desc<kD>(qaddr + kk * 32), idesc, kk > 0);
          }
          issued = true;
          mma_commit(&sm.key_empty[s]);
          mma_commit(&sm.acc_full[ab]);
        }
        if (!ok) break;
        mma_commit(&sm.q_empty[qb]);
        ++nitem;
      }
      if (issued) {
        mma_commit(&sm.final_bar);
        mbar_drain(&sm.final_bar, 0);
      }
    }
  } else if (warp >= kEpiWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));  // idle
  } else {
    // ------------------------------ epilogue (warps 0-15) ------------------------------
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
    static_assert(kEpiWarps / 4 == kGroup, "one epilogue warp per query token of the group");
    const int row = (warp & 3) * 32 + lane;  // TMEM lane == key within the tile
    const int tok = warp >> 2;               // query token of the group handled by this warp
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t a = 0, nitem = 0;
    for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
      const Item it = item_at(item);
      if (!it.valid) continue;
      const int qb = nitem & 1;
      if (!mbar_wait(&sm.q_full[qb], (nitem >> 1) & 1, A.err, abort)) break;
      // this warp's token weights stay in registers for the whole item, as packed pairs
      uint64_t wp[H / 2];
      {
        const float* wf = reinterpret_cast<const float*>(sm.w[qb]) + min(tok, it.n_grp - 1) * H;
#pragma unroll
        for (int x = 0; x < H; x += 4) {
          const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(wf + x);
          wp[x / 2] = v.x;
          wp[x / 2 + 1] = v.y;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&sm.q_empty[qb]);  // the weights are in registers now
      const bool mine = tok < it.n_grp;
      // keys j < j_end of this token's row are stored (causal bound and chunk bound)
      const int j_end = min(it.p_first + tok + 1, it.key_end);
      float* srow = A.scores + static_cast<int64_t>(it.t0 + tok - A.tok_begin) * A.scores_stride;
      const int n_tiles = it.n_tiles;
      int j = it.key_begin + row;
      bool ok = true;
      for (int tile = 0; tile < n_tiles; ++tile, ++a, j += kTile) {
        const int ab = a & 1;
        if (!mbar_wait(&sm.acc_full[ab], (a >> 1) & 1, A.err, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = a % kStages;  // the MMA consumed global tile a from stage a % kStages
        const float s_key = sm.kscale[st][row];
        if (mine) {
          // head h goes to element h % 2 of acc0 (h % 4 < 2) or of acc1 (h % 4 >= 2); every term doubled
          // 16-column TMEM loads, the next one in flight while the current one is reduced
          uint64_t acc0 = 0, acc1 = 0;
          const uint32_t tbase = tmem + lane_base + ab * 256 + tok * H;
          uint32_t v[2][16];
          tmem_ld16(tbase, v[0]);
          tmem_ld_wait(v[0]);
#pragma unroll
          for (int c = 0; c < (H + 15) / 16; ++c) {
            const bool more = (c + 1) * 16 < H;
            if (more) tmem_ld16(tbase + (c + 1) * 16, v[(c + 1) & 1]);
#pragma unroll
            for (int x = 0; x < 16 && c * 16 + x < H; x += 4)
              relu_fma4(acc0, acc1, v[c & 1][x], v[c & 1][x + 1], v[c & 1][x + 2], v[c & 1][x + 3],
                        wp[(c * 16 + x) / 2], wp[(c * 16 + x) / 2 + 1]);
            if (more) tmem_ld_wait(v[(c + 1) & 1]);
          }
          const float total = 0.5f * (pair_sum(acc0) + pair_sum(acc1));
          if (j < j_end) srow[j] = total * s_key;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_relaxed(&sm.acc_empty[ab]);   // TMEM reads are complete (wait::ld)
          mbar_arrive_relaxed(&sm.key_empty[st]);   // the key scales were consumed above
        }
      }
      if (!ok) break;
      ++nitem;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
template <int kH, int kD, int kBS, bool kFP4>
smla_status_t launch_shape(const IdxArgs& A, const uint8_t* q_idx, int n_token_rows, int grid, cudaStream_t stream) {
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return SMLA_ERR_CUDA;
  const CUtensorMapSwizzle swz = kD == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B;
  CUtensorMap key_map, q_map;
  {
    // keys: [num_blocks][block_size][kD elements] of one layer's indexer-key region: kD bytes per key
    // (E4M3), or kD / 2 bytes of packed E2M1 codes unpacked to 16-byte chunks by the copy
    void* base = const_cast<uint8_t*>(A.pool) + static_cast<int64_t>(A.layer) * A.L.layer_stride + A.L.idx_key_off;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(kBS),
                                static_cast<cuuint64_t>(A.L.num_blocks)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kFP4 ? kD / 2 : kD),
                                   static_cast<cuuint64_t>(A.L.block_stride)};
    const cuuint32_t box[3] = {kD, kBS, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType kt = kFP4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (enc(&key_map, kt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SMLA_ERR_CUDA;
  }
  {
    // query rows: [tokens * heads][kD] bytes; one box = the kGroup tokens of a work item
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(n_token_rows) * kH};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD)};
    const cuuint32_t box[2] = {kD, kGroup * kH};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&q_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q_idx), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SMLA_ERR_CUDA;
  }
  const size_t smem = sizeof(IdxSmem) + 1024;
  static std::atomic<bool> attr_set[kMaxDeviceSlots] = {};
  const int dev = current_device_index();
  if (dev < 0) return SMLA_ERR_CUDA;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(index_scores_kernel<kH, kD, kBS, kFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SMLA_ERR_CUDA;
    // setmaxnreg.inc can only draw on the registers the CTA was launched with;
    // refuse to launch if the compiled allocation does not cover the split.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, index_scores_kernel<kH, kD, kBS, kFP4>) != cudaSuccess) return SMLA_ERR_CUDA;
    if (fa.numRegs < kLaunchRegs) return SMLA_ERR_UNSUPPORTED;
    attr_set[dev].store(true, std::memory_order_release);
  }
  index_scores_kernel<kH, kD, kBS, kFP4><<<grid, kThreads, smem, stream>>>(A, key_map, q_map);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace

EncodeTiledFn encode_tiled() {
  static std::atomic<EncodeTiledFn> cached{nullptr};  // the driver's entry point, one per process
  EncodeTiledFn fn = cached.load(std::memory_order_acquire);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// Shapes built into the library: (indexer heads, key dims, block size) with E4M3 keys; FP4 (E2M1)
// keys with 64 heads of 128 dims.
bool index_shape_supported(const KernelLayout& L, int n_idx_heads) {
  const bool deepseek = n_idx_heads == 64 && L.d_index == 128 && (L.block_size == 64 || L.block_size == 16);
  if (L.key_format == SMLA_KEY_E2M1) return deepseek;
  return L.key_format == SMLA_KEY_E4M3 && (deepseek || (n_idx_heads == 4 && L.d_index == 32 && L.block_size == 16));
}

smla_status_t launch_index_scores(const KernelLayout& L, int n_idx_heads, const void* pool, int layer,
                                  const uint8_t* q_idx, const float* w, const int32_t* block_table, int bt_stride,
                                  const int32_t* seq_lens, const int32_t* query_start_loc, int batch, int tok_begin,
                                  int tok_end, int max_q, int max_ctx, float* scores, int64_t scores_stride,
                                  cudaStream_t stream, unsigned* err) {
  if (tok_end <= tok_begin || max_ctx <= 0) return SMLA_OK;
  if (!index_shape_supported(L, n_idx_heads)) return SMLA_ERR_UNSUPPORTED;
  IdxArgs A;
  A.L = L;
  A.n_idx_heads = n_idx_heads;
  A.layer = layer;
  A.pool = static_cast<const uint8_t*>(pool);
  A.w = w;
  A.block_table = block_table;
  A.bt_stride = bt_stride;
  A.seq_lens = seq_lens;
  A.qsl = query_start_loc;
  A.batch = batch;
  A.tok_begin = tok_begin;
  A.tok_end = tok_end;
  const int rows = tok_end - tok_begin;
  A.n_groups = (min(max_q, rows) + kGroup - 1) / kGroup;
  A.n_chunks = (max_ctx + kChunkTiles * kTile - 1) / (kChunkTiles * kTile);
  A.scores = scores;
  A.scores_stride = scores_stride;
  A.err = err;
  const long long items = static_cast<long long>(A.n_chunks) * batch * A.n_groups;
  if (items <= 0) return SMLA_OK;
  const long long sms = device_sm_count();
  const int grid = static_cast<int>(items < sms ? items : sms);
  // Query rows are addressed by absolute token (token t -> rows t*heads ..), so the map spans every
  // token below tok_end; the box of a group near the end reads past it as zeros.
  const bool fp4 = L.key_format == SMLA_KEY_E2M1;
  if (n_idx_heads == 64 && L.d_index == 128 && L.block_size == 64)
    return fp4 ? launch_shape<64, 128, 64, true>(A, q_idx, tok_end, grid, stream)
               : launch_shape<64, 128, 64, false>(A, q_idx, tok_end, grid, stream);
  if (n_idx_heads == 64 && L.d_index == 128 && L.block_size == 16)
    return fp4 ? launch_shape<64, 128, 16, true>(A, q_idx, tok_end, grid, stream)
               : launch_shape<64, 128, 16, false>(A, q_idx, tok_end, grid, stream);
  if (n_idx_heads == 4 && L.d_index == 32 && L.block_size == 16 && !fp4)
    return launch_shape<4, 32, 16, false>(A, q_idx, tok_end, grid, stream);
  return SMLA_ERR_UNSUPPORTED;
}

}  // namespace smla
