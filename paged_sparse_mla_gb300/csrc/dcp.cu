// Split-context (DCP-style) decode on one GPU: candidate merge and log-sum-exp merge.
//
// [AgentX "Kimi K3"]: decode context parallelism spreads one long context over
// ranks; each rank attends over its own part and the partial outputs are
// merged with their log-sum-exp statistics.  [GLM-5.3 "What is new"]: DCP8 for
// decode.  With N shards holding the positions j = N i + r round-robin, every
// shard scores its own positions and keeps its local top-k (smla_index_scores,
// smla_topk on the shard); the two kernels here are the exchange steps:
//
//   * smla_dcp_topk_merge: the union of the shards' (score, global position)
//     candidates is reduced to the k highest by (score desc, position asc) --
//     the unsharded selection -- and each shard receives its selected local
//     positions in ascending order (one CTA per query token; the candidates are
//     sorted in shared memory as 64-bit (order-preserving score key, ~position)
//     words, so every candidate is distinct and the k-th word is the cut);
//   * smla_lse_merge: out = sum_r exp(lse_r - lse) out_r, lse = ln sum_r
//     exp(lse_r), fp32 arithmetic, bf16 out (one warp per query head, 16-byte
//     loads and stores).
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kMergeThreads = 512;
constexpr int kMaxCand = 16384;  // shards x top_k handled by one CTA
constexpr int kMaxMergeK = 4096; // top_k of the merge (the merged-position sort buffer)

__device__ __forceinline__ uint32_t order_key32(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// In-place bitonic sort, descending, of m (a power of two) 64-bit words in shared memory.
__device__ void bitonic_desc(unsigned long long* a, int m) {
  for (int size = 2; size <= m; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < m / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long x = a[lo], y = a[hi];
        if (desc ? (x < y) : (x > y)) {
          a[lo] = y;
          a[hi] = x;
        }
      }
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const float* __restrict__ scores, int64_t shard_stride,
                                                                 int64_t row_stride, const int32_t* __restrict__ topk,
                                                                 int n_shards, int n_tokens, int k,
                                                                 int32_t* __restrict__ shard_sel,
                                                                 int32_t* __restrict__ merged) {
  extern __shared__ unsigned long long cand[];  // [m] sort buffer, then [k] merged positions (as words)
  __shared__ unsigned long long cut;
  __shared__ int n_valid;
  const int t = blockIdx.x;
  const int total = n_shards * k;
  int m = 1;
  while (m < total) m <<= 1;
  if (threadIdx.x == 0) n_valid = 0;
  __syncthreads();
  // candidate (r, i) -> (key << 32) | ~j with j = loc * n_shards + r; empty slots are 0 (below any key)
  int local_valid = 0;
  for (int c = threadIdx.x; c < m; c += blockDim.x) {
    unsigned long long w = 0;
    if (c < total) {
      const int r = c / k, i = c % k;
      const int loc = __ldg(topk + (static_cast<int64_t>(r) * n_tokens + t) * k + i);
      if (loc >= 0) {
        const float s = __ldg(scores + r * shard_stride + static_cast<int64_t>(t) * row_stride + loc);
        const uint32_t j = static_cast<uint32_t>(loc) * static_cast<uint32_t>(n_shards) + static_cast<uint32_t>(r);
        w = (static_cast<unsigned long long>(order_key32(s)) << 32) | static_cast<uint32_t>(~j);
        ++local_valid;
      }
    }
    cand[c] = w;
  }
  atomicAdd(&n_valid, local_valid);
  __syncthreads();
  const int nv = n_valid;
  // the k-th largest word is the cut: a candidate is kept iff its word >= cut
  unsigned long long* sorted = cand;
  bitonic_desc(sorted, m);
  if (threadIdx.x == 0) cut = nv >= k ? sorted[k - 1] : 1ull;
  __syncthreads();
  const unsigned long long c_word = cut;
  const int kept = nv < k ? nv : k;
  // merged global positions, ascending: the first `kept` words hold them; sort them by position
  if (merged != nullptr) {
    unsigned long long* pos = cand + m;  // [mk] scratch after the sort buffer
    int mk = 1;
    while (mk < k) mk <<= 1;
    for (int i = threadIdx.x; i < mk; i += blockDim.x)
      pos[i] = i < kept ? static_cast<unsigned long long>(~static_cast<uint32_t>(sorted[i] & 0xFFFFFFFFull)) : 0ull;
    bitonic_desc(pos, mk);  // positions descending (padding zeros last); written back reversed
    for (int i = threadIdx.x; i < k; i += blockDim.x)
      merged[static_cast<int64_t>(t) * k + i] = i < kept ? static_cast<int32_t>(pos[kept - 1 - i]) : -1;
  }
  // each shard's kept local positions, in the order of its (ascending) top-k list
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_warps = blockDim.x >> 5;
  for (int r = warp; r < n_shards; r += n_warps) {
    const int32_t* row = topk + (static_cast<int64_t>(r) * n_tokens + t) * k;
    const float* srow = scores + r * shard_stride + static_cast<int64_t>(t) * row_stride;
    int32_t* out = shard_sel + (static_cast<int64_t>(r) * n_tokens + t) * k;
    int written = 0;
    for (int i0 = 0; i0 < k; i0 += 32) {
      const int i = i0 + lane;
      bool keep = false;
      int loc = -1;
      if (i < k) {
        loc = __ldg(row + i);
        if (loc >= 0) {
          const uint32_t j = static_cast<uint32_t>(loc) * static_cast<uint32_t>(n_shards) + static_cast<uint32_t>(r);
          const unsigned long long w =
              (static_cast<unsigned long long>(order_key32(__ldg(srow + loc))) << 32) | static_cast<uint32_t>(~j);
          keep = w >= c_word;
        }
      }
      const uint32_t mask = __ballot_sync(0xffffffffu, keep);
      if (keep) out[written + __popc(mask & ((1u << lane) - 1u))] = loc;
      written += __popc(mask);
    }
    for (int i = written + lane; i < k; i += 32) out[i] = -1;
  }
}

// One warp per (token, head): 8 bf16 per lane per step, n_shards partials.
__global__ void lse_merge_kernel(const __nv_bfloat16* __restrict__ parts, const float* __restrict__ parts_lse,
                                 int n_shards, int64_t rows, int d, __nv_bfloat16* __restrict__ out,
                                 float* __restrict__ lse) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int r = 0; r < n_shards; ++r) mx = fmaxf(mx, __ldg(parts_lse + r * rows + row));
  float z = 0.f;
  for (int r = 0; r < n_shards; ++r) {
    const float l = __ldg(parts_lse + r * rows + row);
    z += (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
  }
  const float inv_z = z > 0.f ? 1.f / z : 0.f;
  for (int d0 = 8 * lane; d0 < d; d0 += 8 * 32) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int r = 0; r < n_shards; ++r) {
      const float l = __ldg(parts_lse + r * rows + row);
      if (mx == -INFINITY || l == -INFINITY) continue;
      const float wr = expf(l - mx) * inv_z;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(parts + (r * rows + row) * d + d0));
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        acc[2 * x] += wr * __uint_as_float(vw[x] << 16);
        acc[2 * x + 1] += wr * __uint_as_float(vw[x] & 0xFFFF0000u);
      }
    }
    *reinterpret_cast<uint4*>(out + row * d + d0) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
  }
  if (lane == 0) lse[row] = z > 0.f ? mx + logf(z) : -INFINITY;
}

}  // namespace
}  // namespace smla

using namespace smla;

extern "C" {

smla_status_t smla_dcp_topk_merge(const float* shard_scores, int64_t shard_stride, int64_t row_stride,
                                  const int32_t* shard_topk, int n_shards, int n_tokens, int top_k,
                                  int32_t* shard_sel, int32_t* merged, void* stream) {
  if (n_tokens < 0 || n_shards <= 0 || top_k <= 0) return SMLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return SMLA_OK;
  if (!shard_scores || !shard_topk || !shard_sel || row_stride <= 0 || shard_stride < row_stride * n_tokens)
    return SMLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_shards) * top_k > kMaxCand || top_k > kMaxMergeK) return SMLA_ERR_UNSUPPORTED;
  int m = 1;
  while (m < n_shards * top_k) m <<= 1;
  int mk = 1;
  while (mk < top_k) mk <<= 1;
  const size_t smem = static_cast<size_t>(m + (merged ? mk : 0)) * sizeof(unsigned long long);
  static bool attr_set = false;  // the largest dynamic size any call can ask for, set once
  if (!attr_set) {
    if (cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>((kMaxCand + kMaxMergeK) * sizeof(unsigned long long))) != cudaSuccess)
      return SMLA_ERR_UNSUPPORTED;
    attr_set = true;
  }
  topk_merge_kernel<<<n_tokens, kMergeThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      shard_scores, shard_stride, row_stride, shard_topk, n_shards, n_tokens, top_k, shard_sel, merged);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

smla_status_t smla_lse_merge(const void* parts_out, const float* parts_lse, int n_shards, int n_tokens, int n_heads,
                             int d, void* out, float* lse, void* stream) {
  if (n_shards <= 0 || n_tokens < 0 || n_heads <= 0 || d <= 0) return SMLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return SMLA_OK;
  if (!parts_out || !parts_lse || !out || !lse) return SMLA_ERR_INVALID_ARG;
  if (d % 8 != 0 || (reinterpret_cast<uintptr_t>(parts_out) & 15) != 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0)
    return SMLA_ERR_UNSUPPORTED;
  const int64_t rows = static_cast<int64_t>(n_tokens) * n_heads;
  const int warps = 8;
  const int64_t grid = (rows + warps - 1) / warps;
  lse_merge_kernel<<<static_cast<unsigned>(grid), 32 * warps, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(parts_out), parts_lse, n_shards, rows, d, static_cast<__nv_bfloat16*>(out),
      lse);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // extern "C"
