// smla_index_scores: indexer scores of each query token over its visible context.
//
// [AgentX "DeepSeek V4"]: the indexer has 64 heads but yields a single global
// top-k selection per token.  [GLM-5.3 "What is new"]: the indexer scans the
// whole context (quadratic cost) to choose 2,048 tokens.
//
//   I[t, j] = s_I[j] * sum_h w[t, h] * ReLU(q_I[t, h] . k_I[j])
//
// Design (sm_103a, one persistent CTA per SM):
//   * a work item is (key chunk c, sequence b, group g of <= 4 query tokens of b);
//     items are ordered chunk-major so CTAs working at the same time read the
//     same key chunk of neighbouring sequences (prefix-shared blocks hit L2);
//   * the contraction is one FP8 tcgen05.mma per 32 key dims with the 128 keys
//     of a tile as M (TMEM lane = key) and the group's query heads as N
//     (<= 4 tokens x 64 heads = 256), accumulated in fp32 in tensor memory;
//   * warps 0-15 (epilogue; warp w reads TMEM lanes 32*(w%4).. for query token
//     w/4 of the group) read a key's row of head dot products from TMEM and
//     reduce sum_h w * ReLU(.) per token in registers -- no cross-thread
//     reduction -- then scale by s_I[j] and store the fp32 score;
//   * warps 16-19 (producers) stream 128-key tiles of the indexer-key region of
//     each block through the block table with 16-byte cp.async into 128-byte
//     swizzled stages (one warp per tile, four tiles in flight per CTA);
//   * warp 20 issues the MMAs and owns the tensor-memory allocation.
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kTile = 128;         // keys per tile (MMA M)
constexpr int kGroup = 4;          // query tokens per item (MMA N = kGroup * n_idx_heads)
constexpr int kStages = 8;         // key-tile ring
constexpr int kChunkTiles = 16;    // tiles per work item (2048 keys)
constexpr int kEpiWarps = 16;      // four warps per TMEM sub-partition, one query token each
constexpr int kProducers = 4;      // producer warps
constexpr int kMmaWarp = kEpiWarps + kProducers;
constexpr int kThreads = 32 * (kEpiWarps + kProducers + 1);
constexpr int kMaxN = 256;         // MMA N limit
constexpr int kMaxSeqSmem = 1024;  // batches up to this size keep their metadata in shared memory

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
  const uint8_t* q_idx;
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

__device__ __forceinline__ Item decode_item(const IdxArgs& A, const int* meta, int item) {
  Item it;
  it.valid = 0;
  const int g = item % A.n_groups;
  const int rest = item / A.n_groups;
  const int b = rest % A.batch;
  const int c = rest / A.batch;
  const bool in_smem = A.batch <= kMaxSeqSmem;
  const int q0 = in_smem ? meta[b] : __ldg(A.qsl + b);
  const int q1 = in_smem ? meta[b + 1] : __ldg(A.qsl + b + 1);
  const int r0 = max(q0, A.tok_begin), r1 = min(q1, A.tok_end);  // this call's rows of sequence b
  const int first = r0 + g * kGroup;
  if (first >= r1) return it;
  const int n_grp = min(kGroup, r1 - first);
  const int n_q = q1 - q0;
  const int p_first = (in_smem ? meta[A.batch + 1 + b] : __ldg(A.seq_lens + b)) - n_q + (first - q0);
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

// Dense work items (batches up to kMaxSeqSmem): sequence b owns items
// item_off[b] .. item_off[b+1]-1, enumerating (query group g, key chunk c) with
// c fastest, c < chunks[b]; consecutive items are consecutive chunks, so the
// CTAs running at the same time share sequences (and prefix-shared blocks).
__device__ __forceinline__ Item decode_dense(const IdxArgs& A, const int* meta, const int* item_off,
                                             const int* chunks, int item) {
  int lo = 0, hi = A.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (item_off[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int local = item - item_off[b];
  const int nc = chunks[b];
  const int g = local / nc, c = local % nc;
  Item it;
  it.valid = 0;
  const int q0 = meta[b], q1 = meta[b + 1];
  const int r0 = max(q0, A.tok_begin), r1 = min(q1, A.tok_end);
  const int first = r0 + g * kGroup;
  if (first >= r1) return it;
  const int n_grp = min(kGroup, r1 - first);
  const int p_first = meta[A.batch + 1 + b] - (q1 - q0) + (first - q0);
  const int p_last = p_first + n_grp - 1;
  const int key_begin = c * kChunkTiles * kTile;
  if (p_last < 0 || key_begin > p_last) return it;  // an early group of a long chunk list
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

// Items per sequence and their prefix sum (one warp).
__device__ void build_item_table(const IdxArgs& A, const int* meta, int* item_off, int* chunks) {
  const int lane = threadIdx.x & 31;
  const int per = (A.batch + 31) / 32;
  const int b0 = min(A.batch, lane * per), b1 = min(A.batch, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    const int q0 = meta[b], q1 = meta[b + 1];
    const int r0 = max(q0, A.tok_begin), r1 = min(q1, A.tok_end);
    const int rows = max(0, r1 - r0);
    const int p_last = meta[A.batch + 1 + b] - (q1 - q0) + (r1 - 1 - q0);
    const int nc = (rows > 0 && p_last >= 0) ? (p_last + kChunkTiles * kTile) / (kChunkTiles * kTile) : 0;
    chunks[b] = max(nc, 1);
    local += ((rows + kGroup - 1) / kGroup) * nc;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - local;
  for (int b = b0; b < b1; ++b) {
    item_off[b] = run;
    const int q0 = meta[b], q1 = meta[b + 1];
    const int rows = max(0, min(q1, A.tok_end) - max(q0, A.tok_begin));
    const int p_last = meta[A.batch + 1 + b] - (q1 - q0) + (min(q1, A.tok_end) - 1 - q0);
    const int nc = (rows > 0 && p_last >= 0) ? (p_last + kChunkTiles * kTile) / (kChunkTiles * kTile) : 0;
    run += ((rows + kGroup - 1) / kGroup) * nc;
  }
  if (lane == 31) item_off[A.batch] = incl;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%1, %2};\n\tmov.b64 rb, {%3, %4};\n\tmov.b64 rc, {%5, %6};\n\t"
      "fma.rn.f32x2 %0, ra, rb, rc;\n\t}"
      : "=l"(d)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return make_float2(__uint_as_float(static_cast<uint32_t>(d)), __uint_as_float(static_cast<uint32_t>(d >> 32)));
}

__device__ __forceinline__ int mma_n(int n_grp, int heads) {
  const int n = n_grp * heads;
  return max(16, (n + 15) & ~15);
}

template <int kH, int kD, int kBS>
__global__ void __launch_bounds__(kThreads, 1) index_scores_kernel(const IdxArgs A) {
  extern __shared__ uint8_t smem_raw[];
  IdxSmem& sm = *reinterpret_cast<IdxSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool dense = A.batch <= kMaxSeqSmem;
  constexpr int H = kH;
  constexpr int D = kD;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.key_full[s], 1);               // one arrive per producer warp
      mbar_init(&sm.key_empty[s], 1 + kEpiWarps);  // MMA done + every epilogue warp read the scales
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1 + kEpiWarps);  // MMA done + every epilogue warp done with the weights
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
    if (warp == 0) build_item_table(A, sm.seq_meta, sm.item_off, sm.chunks);
  }
  if (warp == kMmaWarp) tmem_alloc(&sm.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  volatile int* abort = &sm.abort;
  const int n_items = dense ? sm.item_off[A.batch] : A.n_chunks * A.batch * A.n_groups;
  const auto item_at = [&](int item) {
    return dense ? decode_dense(A, sm.seq_meta, sm.item_off, sm.chunks, item) : decode_item(A, sm.seq_meta, item);
  };

  if (warp >= kEpiWarps && warp < kMmaWarp) {
    // ------------------------------ producers ------------------------------
    // Lane l always copies 16-byte chunk (l % kCh) of rows l / kCh + i * kRowStep;
    // a tile spans kTile / kBS blocks whose bases lanes 0.. load once per tile.
    constexpr int kCh = kD / 16;
    constexpr int kRowStep = 32 / kCh;
    constexpr int kIters = kTile / kRowStep;
    constexpr int kBlocks = kTile / kBS;
    static_assert(kTile % kBS == 0 && kBS % kRowStep == 0 && kBlocks <= 32 && kBS % 4 == 0, "tile geometry");
    const int pw = warp - kEpiWarps;
    const int ch = lane % kCh, r0 = lane / kCh;
    const int64_t layer_off = static_cast<int64_t>(A.layer) * A.L.layer_stride;
    uint32_t k = 0, nitem = 0;
    for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
      const Item it = item_at(item);
      if (!it.valid) continue;
      const int32_t* bt = A.block_table + static_cast<int64_t>(it.b) * A.bt_stride;
      if (pw == 0) {
        const int qb = nitem & 1;
        if (!mbar_wait(&sm.q_empty[qb], ((nitem >> 1) & 1) ^ 1, A.err, abort)) break;
        const int rows = it.n_grp * H;
        const uint32_t qbase = smem_u32(sm.q[qb]);
        const uint8_t* qsrc = A.q_idx + static_cast<int64_t>(it.t0) * H * kD + ch * 16;
        for (int r = r0; r < rows; r += kRowStep) cp_async16(qbase + sw128_off(r, ch), qsrc + r * kD, 16);
        // the group's weights (n_grp * H floats, contiguous rows of w) ride along with q
        const float* wsrc = A.w + static_cast<int64_t>(it.t0) * H;
        for (int i = lane; i < rows / 4; i += 32) cp_async16(smem_u32(&sm.w[qb][i]), wsrc + 4 * i, 16);
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.q_full[qb]);
      }
      for (int tile = 0; tile < it.n_tiles; ++tile, ++k) {
        if (static_cast<int>(k % kProducers) != pw) continue;
        const int s = k % kStages;
        const int j0 = it.key_begin + tile * kTile;
        unsigned long long kbase = 0;  // lane b < kBlocks: base of block b of the tile (0 = skip)
        if (lane < kBlocks && j0 + lane * kBS < it.key_end) {
          const int blk = __ldg(bt + (j0 + lane * kBS) / kBS);
          if (blk < 0 || blk >= A.L.num_blocks) {
            latch_error(A.err, SMLA_ERR_BAD_INDEX);
          } else {
            kbase = reinterpret_cast<unsigned long long>(A.pool + static_cast<int64_t>(blk) * A.L.block_stride + layer_off);
          }
        }
        if (!mbar_wait(&sm.key_empty[s], ((k / kStages) & 1) ^ 1, A.err, abort)) break;
        const uint32_t base = smem_u32(sm.keys[s]);
#pragma unroll
        for (int i = 0; i < kIters; ++i) {
          const int r = r0 + i * kRowStep;
          const unsigned long long b = __shfl_sync(0xffffffffu, kbase, (i * kRowStep) / kBS);
          const bool ok = b != 0 && j0 + r < it.key_end;
          const uint8_t* src = ok ? reinterpret_cast<const uint8_t*>(b) + A.L.idx_key_off + (r % kBS) * kD + ch * 16
                                  : A.pool;
          cp_async16(base + sw128_off(r, ch), src, ok ? 16u : 0u);
        }
        {
          // key scales: lane l copies keys 4l..4l+3 (never straddling a block)
          const unsigned long long b = __shfl_sync(0xffffffffu, kbase, (4 * lane) / kBS);
          const bool ok = b != 0 && j0 + 4 * lane < it.key_end;
          const uint8_t* src =
              ok ? reinterpret_cast<const uint8_t*>(b) + A.L.idx_scale_off + ((4 * lane) % kBS) * 4 : A.pool;
          cp_async16(smem_u32(&sm.kscale[s][4 * lane]), src, ok ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.key_full[s]);
      }
      ++nitem;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      uint32_t k = 0, nitem = 0, a = 0;
      bool issued = false;
      for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
        const Item it = item_at(item);
        if (!it.valid) continue;
        const int qb = nitem & 1;
        if (!mbar_wait(&sm.q_full[qb], (nitem >> 1) & 1, A.err, abort)) break;
        const int n = mma_n(it.n_grp, H);
        const uint32_t idesc = make_idesc(128, n, 0, 0, 0, 0);
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
          for (int kk = 0; kk < D / 32; ++kk) {
            mma_f8(tmem + ab * 256, sw128_desc(kaddr + kk * 32, 16, 1024), sw128_desc(qaddr + kk * 32, 16, 1024),
                   idesc, kk > 0);
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
        mbar_wait(&sm.final_bar, 0, A.err, abort);
      }
    }
  } else {
    // ------------------------------ epilogue (warps 0-15) ------------------------------
    const int row = (warp & 3) * 32 + lane;  // TMEM lane == key within the tile
    const int tok = warp >> 2;               // query token of the group handled by this warp
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t a = 0, nitem = 0;
    for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
      const Item it = item_at(item);
      if (!it.valid) continue;
      const int qb = nitem & 1;
      if (!mbar_wait(&sm.q_full[qb], (nitem >> 1) & 1, A.err, abort)) break;
      const float4* wq = sm.w[qb];
      bool ok = true;
      for (int tile = 0; tile < it.n_tiles; ++tile, ++a) {
        const int j = it.key_begin + tile * kTile + row;
        const int ab = a & 1;
        if (!mbar_wait(&sm.acc_full[ab], (a >> 1) & 1, A.err, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = a % kStages;  // the MMA consumed global tile a from stage a % kStages
        const float s_key = sm.kscale[st][row];
        for (int i = tok; i < it.n_grp; i += kEpiWarps / 4) {
          // two packed accumulator pairs: head h goes to lane h % 4 of (acc01, acc23)
          float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
#pragma unroll
          for (int h0 = 0; h0 < H; h0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + ab * 256 + i * H + h0, v);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32 && h0 + x < H; x += 4) {
              const float4 wv = wq[(i * H + h0 + x) / 4];
              const float2 r01 = make_float2(fmaxf(__uint_as_float(v[x]), 0.f), fmaxf(__uint_as_float(v[x + 1]), 0.f));
              const float2 r23 =
                  make_float2(fmaxf(__uint_as_float(v[x + 2]), 0.f), fmaxf(__uint_as_float(v[x + 3]), 0.f));
              acc01 = ffma2(r01, make_float2(wv.x, wv.y), acc01);
              acc23 = ffma2(r23, make_float2(wv.z, wv.w), acc23);
            }
          }
          const float total = (acc01.x + acc01.y) + (acc23.x + acc23.y);
          if (j <= it.p_first + i && j < it.key_end) {
            A.scores[static_cast<int64_t>(it.t0 + i - A.tok_begin) * A.scores_stride + j] = total * s_key;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_relaxed(&sm.acc_empty[ab]);   // TMEM reads are complete (wait::ld)
          mbar_arrive_relaxed(&sm.key_empty[st]);   // the key scales were consumed above
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&sm.q_empty[qb]);  // this warp is done with the item's weights
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

template <int kH, int kD, int kBS>
smla_status_t launch_shape(const IdxArgs& A, int grid, cudaStream_t stream) {
  const size_t smem = sizeof(IdxSmem) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(index_scores_kernel<kH, kD, kBS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SMLA_ERR_CUDA;
    attr_set = true;
  }
  index_scores_kernel<kH, kD, kBS><<<grid, kThreads, smem, stream>>>(A);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace

smla_status_t launch_index_scores(const KernelLayout& L, int n_idx_heads, const void* pool, int layer,
                                  const uint8_t* q_idx, const float* w, const int32_t* block_table, int bt_stride,
                                  const int32_t* seq_lens, const int32_t* query_start_loc, int batch, int tok_begin,
                                  int tok_end, int max_q, int max_ctx, float* scores, int64_t scores_stride,
                                  cudaStream_t stream, unsigned* err) {
  if (tok_end <= tok_begin || max_ctx <= 0) return SMLA_OK;
  if (n_idx_heads * kGroup > kMaxN || n_idx_heads > 64 || L.d_index % 32 != 0 || L.d_index > 128)
    return SMLA_ERR_UNSUPPORTED;
  IdxArgs A;
  A.L = L;
  A.n_idx_heads = n_idx_heads;
  A.layer = layer;
  A.pool = static_cast<const uint8_t*>(pool);
  A.q_idx = q_idx;
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
  // Shapes built into the library: (indexer heads, key dims, block size).
  if (n_idx_heads == 64 && L.d_index == 128 && L.block_size == 64) return launch_shape<64, 128, 64>(A, grid, stream);
  if (n_idx_heads == 64 && L.d_index == 128 && L.block_size == 16) return launch_shape<64, 128, 16>(A, grid, stream);
  if (n_idx_heads == 4 && L.d_index == 32 && L.block_size == 16) return launch_shape<4, 32, 16>(A, grid, stream);
  return SMLA_ERR_UNSUPPORTED;
}

}  // namespace smla
