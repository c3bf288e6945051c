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
//     64-bit (order-preserving score key, ~position) words in shared memory, so
//     every candidate is distinct; a radix select finds the k-th word, each
//     shard's kept positions are compacted in list order, and the merged
//     positions are placed by rank);
//   * smla_lse_merge: out = sum_r exp(lse_r - lse) out_r, lse = ln sum_r
//     exp(lse_r), fp32 arithmetic, bf16 out (one warp per query head, 16-byte
//     loads and stores).
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kMergeThreads = 512;
constexpr int kMaxCand = 16384;  // shards x top_k handled by one CTA

__device__ __forceinline__ uint32_t order_key32(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the CTA (kMergeThreads threads); returns this thread's prefix and the total.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kMergeThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kMergeThreads / 32) warp_sums[lane] = w;
  }
  __syncthreads();
  total = warp_sums[kMergeThreads / 32 - 1];
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  __syncthreads();
  return before + x - v;
}

struct MergeSmem {
  unsigned long long word[kMaxCand];  // candidate c = r * k + i, in the shards' list order
  int sel[kMaxCand];                  // shard r's kept local positions at [r * k ...]
  int hist[256];
  int warp_sums[32];
  int kept[64];                       // kept count per shard
  unsigned long long prefix;
  int remaining;
};

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const float* __restrict__ scores, int64_t shard_stride,
                                                                 int64_t row_stride, const int32_t* __restrict__ topk,
                                                                 int n_shards, int n_tokens, int k,
                                                                 int32_t* __restrict__ shard_sel,
                                                                 int32_t* __restrict__ merged) {
  extern __shared__ __align__(16) uint8_t merge_smem_raw[];
  MergeSmem& sm = *reinterpret_cast<MergeSmem*>(merge_smem_raw);
  const int t = blockIdx.x;
  const int total = n_shards * k;
  // candidate (r, i) -> (key << 32) | ~j, j = loc * n_shards + r; empty slots are 0 (below any key).
  // In rounds of 8 per thread: top-k entries first, then the scores they point at, so each
  // thread's loads are in flight together.
  constexpr int kRound = 8;
  int nv = 0;
  for (int c0 = 0; c0 < total; c0 += kRound * kMergeThreads) {
    int loc[kRound];
    float sv[kRound];
#pragma unroll
    for (int x = 0; x < kRound; ++x) {
      const int c = c0 + threadIdx.x + x * kMergeThreads;
      loc[x] = c < total ? __ldg(topk + (static_cast<int64_t>(c / k) * n_tokens + t) * k + c % k) : -1;
    }
#pragma unroll
    for (int x = 0; x < kRound; ++x) {
      const int c = c0 + threadIdx.x + x * kMergeThreads;
      sv[x] = loc[x] >= 0 ? __ldg(scores + (c / k) * shard_stride + static_cast<int64_t>(t) * row_stride + loc[x])
                          : 0.f;
    }
#pragma unroll
    for (int x = 0; x < kRound; ++x) {
      const int c = c0 + threadIdx.x + x * kMergeThreads;
      if (c < total) {
        unsigned long long w = 0;
        if (loc[x] >= 0) {
          const uint32_t j = static_cast<uint32_t>(loc[x]) * static_cast<uint32_t>(n_shards) +
                             static_cast<uint32_t>(c / k);
          w = (static_cast<unsigned long long>(order_key32(sv[x])) << 32) | static_cast<uint32_t>(~j);
          ++nv;
        }
        sm.word[c] = w;
      }
    }
  }
  int n_valid;
  cta_exclusive_scan(nv, sm.warp_sums, n_valid);
  // the k-th largest word (all words distinct): radix select, 8 bits a pass from the top
  unsigned long long cut = 1ull;  // fewer than k candidates: keep every valid one
  if (n_valid > k) {
    if (threadIdx.x == 0) {
      sm.prefix = 0ull;
      sm.remaining = k;
    }
    unsigned long long mask = 0ull;
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kMergeThreads) sm.hist[i] = 0;
      __syncthreads();
      const unsigned long long pre = sm.prefix;
      for (int c = threadIdx.x; c < total; c += kMergeThreads) {
        const unsigned long long w = sm.word[c];
        if ((w & mask) == pre) atomicAdd(&sm.hist[(w >> shift) & 0xFF], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {  // highest bin whose suffix count reaches `remaining`
        const int lane = threadIdx.x;
        int cnt[8], sum = 0;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          cnt[x] = sm.hist[255 - (lane * 8 + x)];
          sum += cnt[x];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int need = sm.remaining;
        int above = incl - sum;
        const bool here = above < need && incl >= need;
        if (here) {
          for (int x = 0; x < 8; ++x) {
            if (above + cnt[x] >= need) {
              sm.prefix = pre | (static_cast<unsigned long long>(255 - (lane * 8 + x)) << shift);
              sm.remaining = need - above;
              break;
            }
            above += cnt[x];
          }
        }
      }
      mask |= 0xFFull << shift;
      __syncthreads();
    }
    cut = sm.prefix;  // every word is distinct, so exactly k words are >= the k-th one
  }
  // each shard's kept local positions in list order (ascending), compacted by a CTA scan
  for (int r = 0; r < n_shards; ++r) {
    int base = 0;
    for (int i0 = 0; i0 < k; i0 += kMergeThreads) {
      const int i = i0 + threadIdx.x;
      const unsigned long long w = i < k ? sm.word[r * k + i] : 0ull;
      const bool keep = i < k && w != 0ull && w >= cut;
      int tot;
      const int pos = cta_exclusive_scan(keep ? 1 : 0, sm.warp_sums, tot);
      if (keep) sm.sel[r * k + base + pos] = static_cast<int>((~static_cast<uint32_t>(w & 0xFFFFFFFFull) -
                                                                static_cast<uint32_t>(r)) /
                                                               static_cast<uint32_t>(n_shards));
      base += tot;
    }
    if (threadIdx.x == 0) sm.kept[r] = base;
  }
  __syncthreads();
  for (int r = 0; r < n_shards; ++r) {
    int32_t* out = shard_sel + (static_cast<int64_t>(r) * n_tokens + t) * k;
    for (int i = threadIdx.x; i < k; i += kMergeThreads) out[i] = i < sm.kept[r] ? sm.sel[r * k + i] : -1;
  }
  // merged global positions, ascending: an element's rank is the number of kept positions
  // below it in every shard (binary search in each shard's ascending list)
  if (merged != nullptr) {
    int n_kept = 0;
    for (int r = 0; r < n_shards; ++r) n_kept += sm.kept[r];
    int32_t* mrow = merged + static_cast<int64_t>(t) * k;
    for (int c = threadIdx.x; c < total; c += kMergeThreads) {
      const int r = c / k, i = c % k;
      if (i >= sm.kept[r]) continue;
      const long long j = static_cast<long long>(sm.sel[c]) * n_shards + r;
      int rank = i;
      for (int r2 = 0; r2 < n_shards; ++r2) {
        if (r2 == r) continue;
        // kept local positions l of shard r2 with l * N + r2 < j
        int lo = 0, hi = sm.kept[r2];
        const int* list = sm.sel + r2 * k;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (static_cast<long long>(list[mid]) * n_shards + r2 < j) lo = mid + 1; else hi = mid;
        }
        rank += lo;
      }
      mrow[rank] = static_cast<int32_t>(j);
    }
    for (int i = n_kept + threadIdx.x; i < k; i += kMergeThreads) mrow[i] = -1;
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
  if (static_cast<int64_t>(n_shards) * top_k > kMaxCand) return SMLA_ERR_UNSUPPORTED;
  if (n_shards > 64) return SMLA_ERR_UNSUPPORTED;
  const size_t smem = sizeof(MergeSmem);
  static std::atomic<bool> attr_set[kMaxDeviceSlots] = {};
  const int dev = current_device_index();
  if (dev < 0) return SMLA_ERR_CUDA;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return SMLA_ERR_UNSUPPORTED;
    attr_set[dev].store(true, std::memory_order_release);
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
