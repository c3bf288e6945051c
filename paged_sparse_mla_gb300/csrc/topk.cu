// smla_topk: exact top-k of each query token's scores, ties to the lower position.
//
// [GLM-5.3 "What is new"]: the indexer keeps 2,048 tokens per query token.
// [AgentX "DeepSeek V4"]: one global top-k per token; [AgentX "Closing the
// loop: kernels"] names a dedicated top-k path among the kernels that matter.
//
// One CTA per query row.  Scores map to order-preserving 32-bit keys
// (-0 folded onto +0).  A radix select over the key bits (12, 12, then 8 bits,
// each pass a shared-memory histogram of the elements that still match the
// bits fixed so far, with warp-aggregated increments) finds the k-th largest
// key T and how many elements equal to T are still needed.  The selection pass
// then gives each thread a contiguous segment of the row: counts of "> T" and
// "== T" per segment, two block scans (tie rank, output slot), and a second
// read of the segment writes the kept positions in ascending order.
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the CTA; returns the prefix and writes the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kWarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) warp_tot[lane] = t;  // inclusive
  }
  __syncthreads();
  total = warp_tot[kWarps - 1];
  return x - v + (warp > 0 ? warp_tot[warp - 1] : 0);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(int k, const float* __restrict__ scores, int64_t stride,
                                                        const int32_t* __restrict__ seq_lens,
                                                        const int32_t* __restrict__ qsl, int batch, int tok_begin,
                                                        int32_t* __restrict__ out) {
  __shared__ int hist[kBins];
  __shared__ int warp_tot[32];
  __shared__ int sel_bin, sel_above;
  const int row = blockIdx.x;
  const int t = tok_begin + row;
  const int b = seq_of_token(qsl, batch, t);
  const int q0 = __ldg(qsl + b), n_q = __ldg(qsl + b + 1) - q0;
  const int n = __ldg(seq_lens + b) - n_q + (t - q0) + 1;  // positions 0..p
  const float* s = scores + static_cast<int64_t>(row) * stride;
  int32_t* o = out + static_cast<int64_t>(row) * k;

  if (n <= k) {
    for (int i = threadIdx.x; i < k; i += kThreads) o[i] = i < n ? i : -1;
    return;
  }

  // ---- radix select of the k-th largest key ----
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const uint32_t bmask = (1u << widths[pass]) - 1u;
    const int nb = 1 << widths[pass];
    for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kThreads) {
      const int j = base + threadIdx.x;
      bool hit = false;
      uint32_t bin = 0;
      if (j < n) {
        const uint32_t key = order_key(__ldg(s + j));
        hit = (key & mask) == prefix;
        bin = (key >> shift) & bmask;
      }
      const uint32_t active = __ballot_sync(0xffffffffu, hit);
      if (hit) {
        const uint32_t peers = __match_any_sync(active, bin);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
    }
    __syncthreads();
    // bins are scanned from the top: find B with count(> B) < remaining <= count(>= B)
    const int per = nb / kThreads > 0 ? nb / kThreads : 1;
    int local = 0;
    const int hi_bin = nb - 1 - threadIdx.x * per;  // this thread's bins: hi_bin down to hi_bin-per+1
    if (threadIdx.x * per < nb)
      for (int x = 0; x < per; ++x) local += hist[hi_bin - x];
    int total;
    const int before = block_exclusive_scan(threadIdx.x * per < nb ? local : 0, warp_tot, total);
    if (threadIdx.x * per < nb && before < remaining && before + local >= remaining) {
      int acc = before;
      for (int x = 0; x < per; ++x) {
        const int c = hist[hi_bin - x];
        if (acc + c >= remaining) {
          sel_bin = hi_bin - x;
          sel_above = acc;
          break;
        }
        acc += c;
      }
    }
    __syncthreads();
    const int bin = sel_bin;
    remaining -= sel_above;
    prefix |= static_cast<uint32_t>(bin) << shift;
    mask |= bmask << shift;
    const bool exact = hist[bin] == remaining;  // every element of this bin is kept
    __syncthreads();
    if (exact) break;
  }

  // ---- ordered selection ----
  const int seg = (n + kThreads - 1) / kThreads;
  const int lo = min(n, threadIdx.x * seg), hi = min(n, lo + seg);
  int gt = 0, eq = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(__ldg(s + j)) & mask;
    gt += key > prefix;
    eq += key == prefix;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, warp_tot, tot);
  const int eq_take = max(0, min(eq, remaining - eq_before));
  const int out_before = block_exclusive_scan(gt + eq_take, warp_tot, tot);
  int pos = out_before, eq_seen = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(__ldg(s + j)) & mask;
    bool keep = key > prefix;
    if (key == prefix) {
      keep = eq_seen < eq_take;
      ++eq_seen;
    }
    if (keep) o[pos++] = j;
  }
}

}  // namespace

smla_status_t launch_topk(int top_k, const float* scores, int64_t scores_stride, const int32_t* seq_lens,
                          const int32_t* query_start_loc, int batch, int tok_begin, int tok_end, int32_t* topk_idx,
                          cudaStream_t stream, unsigned* err) {
  (void)err;
  const int rows = tok_end - tok_begin;
  if (rows <= 0) return SMLA_OK;
  topk_kernel<<<rows, kThreads, 0, stream>>>(top_k, scores, scores_stride, seq_lens, query_start_loc, batch,
                                             tok_begin, topk_idx);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
