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
//   * warps 0-3 (epilogue) read a key's row of head dot products from TMEM and
//     reduce sum_h w * ReLU(.) per token in registers -- no cross-thread
//     reduction -- then scale by s_I[j] and store the fp32 score (coalesced);
//   * warps 4-7 (producers) stream 128-key tiles of the indexer-key region of
//     each block through the block table with 16-byte cp.async into 128-byte
//     swizzled stages (one warp per tile, four tiles in flight per CTA);
//   * warp 8 issues the MMAs and owns the tensor-memory allocation.
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kTile = 128;         // keys per tile (MMA M)
constexpr int kGroup = 4;          // query tokens per item (MMA N = kGroup * n_idx_heads)
constexpr int kStages = 8;         // key-tile ring
constexpr int kChunkTiles = 16;    // tiles per work item (2048 keys)
constexpr int kProducers = 4;      // producer warps
constexpr int kThreads = 32 * (4 + kProducers + 1);
constexpr int kMaxN = 256;         // MMA N limit

struct __align__(1024) IdxSmem {
  uint8_t keys[kStages][kTile * 128];   // 16 KB per stage, 1024-aligned
  uint8_t q[2][kMaxN * 128];            // 32 KB per buffer
  float w[kGroup * 64];                 // epilogue-owned weights of the current item
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

__device__ __forceinline__ Item decode_item(const IdxArgs& A, int item) {
  Item it;
  it.valid = 0;
  const int g = item % A.n_groups;
  const int rest = item / A.n_groups;
  const int b = rest % A.batch;
  const int c = rest / A.batch;
  const int q0 = __ldg(A.qsl + b), q1 = __ldg(A.qsl + b + 1);
  const int r0 = max(q0, A.tok_begin), r1 = min(q1, A.tok_end);  // this call's rows of sequence b
  const int first = r0 + g * kGroup;
  if (first >= r1) return it;
  const int n_grp = min(kGroup, r1 - first);
  const int n_q = q1 - q0;
  const int p_first = __ldg(A.seq_lens + b) - n_q + (first - q0);
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

__device__ __forceinline__ int mma_n(int n_grp, int heads) {
  const int n = n_grp * heads;
  return max(16, (n + 15) & ~15);
}

__global__ void __launch_bounds__(kThreads, 1) index_scores_kernel(const IdxArgs A) {
  extern __shared__ uint8_t smem_raw[];
  IdxSmem& sm = *reinterpret_cast<IdxSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = A.n_chunks * A.batch * A.n_groups;
  const int H = A.n_idx_heads;
  const int D = A.L.d_index;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.key_full[s], 32);
      mbar_init(&sm.key_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 32);
      mbar_init(&sm.q_empty[i], 1);
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], 128);
    }
    mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  if (warp == 8) tmem_alloc(&sm.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  volatile int* abort = &sm.abort;

  if (warp >= 4 && warp < 4 + kProducers) {
    // ------------------------------ producers ------------------------------
    const int pw = warp - 4;
    uint32_t k = 0, nitem = 0;
    const int chunks_per_row = D / 16;
    for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
      const Item it = decode_item(A, item);
      if (!it.valid) continue;
      const int32_t* bt = A.block_table + static_cast<int64_t>(it.b) * A.bt_stride;
      if (pw == 0) {
        const int qb = nitem & 1;
        if (!mbar_wait(&sm.q_empty[qb], ((nitem >> 1) & 1) ^ 1, A.err, abort)) break;
        const int rows = it.n_grp * H;
        const uint32_t qbase = smem_u32(sm.q[qb]);
        for (int u = lane; u < rows * chunks_per_row; u += 32) {
          const int r = u / chunks_per_row, ch = u % chunks_per_row;
          const uint8_t* src = A.q_idx + (static_cast<int64_t>(it.t0) * H + r) * D + ch * 16;
          cp_async16(qbase + sw128_off(r, ch), src, 16);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async();
        mbar_arrive(&sm.q_full[qb]);
      }
      for (int tile = 0; tile < it.n_tiles; ++tile, ++k) {
        if (static_cast<int>(k % kProducers) != pw) continue;
        const int s = k % kStages;
        if (!mbar_wait(&sm.key_empty[s], ((k / kStages) & 1) ^ 1, A.err, abort)) break;
        const uint32_t base = smem_u32(sm.keys[s]);
        const int j0 = it.key_begin + tile * kTile;
        for (int u = lane; u < kTile * chunks_per_row; u += 32) {
          const int r = u / chunks_per_row, ch = u % chunks_per_row;
          const int j = j0 + r;
          const uint8_t* src = A.pool;
          uint32_t bytes = 0;
          if (j < it.key_end) {
            int blk = __ldg(bt + j / A.L.block_size);
            if (blk < 0 || blk >= A.L.num_blocks) {
              latch_error(A.err, SMLA_ERR_BAD_INDEX);
            } else {
              src = A.pool + static_cast<int64_t>(blk) * A.L.block_stride +
                    static_cast<int64_t>(A.layer) * A.L.layer_stride + A.L.idx_key_off +
                    static_cast<int64_t>(j % A.L.block_size) * D + ch * 16;
              bytes = 16;
            }
          }
          cp_async16(base + sw128_off(r, ch), src, bytes);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async();
        mbar_arrive(&sm.key_full[s]);
      }
      ++nitem;
    }
  } else if (warp == 8) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      uint32_t k = 0, nitem = 0, a = 0;
      bool issued = false;
      for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
        const Item it = decode_item(A, item);
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
    // ------------------------------ epilogue (warps 0-3) ------------------------------
    const int row = threadIdx.x;  // TMEM lane == key within the tile
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    uint32_t a = 0;
    for (int item = blockIdx.x; item < n_items && !*abort; item += gridDim.x) {
      const Item it = decode_item(A, item);
      if (!it.valid) continue;
      named_bar_sync(1, 128);
      for (int i = row; i < it.n_grp * H; i += 128) sm.w[i] = __ldg(A.w + static_cast<int64_t>(it.t0) * H + i);
      named_bar_sync(1, 128);
      const int32_t* bt = A.block_table + static_cast<int64_t>(it.b) * A.bt_stride;
      bool ok = true;
      for (int tile = 0; tile < it.n_tiles; ++tile, ++a) {
        const int j = it.key_begin + tile * kTile + row;
        float s_key = 0.f;
        if (j < it.key_end) {
          const int blk = __ldg(bt + j / A.L.block_size);
          if (blk >= 0 && blk < A.L.num_blocks) {
            s_key = __ldg(reinterpret_cast<const float*>(A.pool + static_cast<int64_t>(blk) * A.L.block_stride +
                                                         static_cast<int64_t>(A.layer) * A.L.layer_stride +
                                                         A.L.idx_scale_off) +
                          (j % A.L.block_size));
          }
        }
        const int ab = a & 1;
        if (!mbar_wait(&sm.acc_full[ab], (a >> 1) & 1, A.err, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int i = 0; i < it.n_grp; ++i) {
          float acc = 0.f;
          for (int h0 = 0; h0 < H; h0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + ab * 256 + i * H + h0, v);
            tmem_ld_wait();
            const int hn = min(32, H - h0);
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              if (x < hn) acc = fmaf(fmaxf(__uint_as_float(v[x]), 0.f), sm.w[i * H + h0 + x], acc);
            }
          }
          if (j <= it.p_first + i && j < it.key_end) {
            A.scores[static_cast<int64_t>(it.t0 + i - A.tok_begin) * A.scores_stride + j] = acc * s_key;
          }
        }
        tc_fence_before();
        mbar_arrive(&sm.acc_empty[ab]);
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
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
  const size_t smem = sizeof(IdxSmem) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(index_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SMLA_ERR_CUDA;
    attr_set = true;
  }
  const long long sms = device_sm_count();
  const int grid = static_cast<int>(items < sms ? items : sms);
  index_scores_kernel<<<grid, kThreads, smem, stream>>>(A);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
