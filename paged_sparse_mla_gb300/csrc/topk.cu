// smla_topk: exact top-k of each query token's scores, ties to the lower position.
//
// [GLM-5.3 "What is new"]: the indexer keeps 2,048 tokens per query token.
// [AgentX "DeepSeek V4"]: one global top-k per token; [AgentX "Closing the
// loop: kernels"] names a dedicated top-k path among the kernels that matter.
//
// One CTA per query row; scores map to order-preserving 32-bit keys (-0 folded
// onto +0).  Fast path, one coalesced read of the row:
//   1. an 8,192-element sample (256 runs of 32 consecutive positions, whole
//      128-byte lines of an aligned row, evenly spread) is radix-selected (top 24
//      key bits) in shared memory to a threshold T whose rank in the sample
//      leaves a safety margin above k/n of the sample; the radix histograms count
//      with plain shared-memory atomics;
//   2. warp w scans its own contiguous segment of the row and appends every
//      element with key >= T, as a 64-bit (key, ~position) pair, to its own list
//      in shared memory, in position order (16 keys per lane per iteration, the
//      next 16 in flight; one warp scan per iteration places the hits).  Bulk
//      L2 prefetches run 4 KB ahead of each warp.  (Prefetching the start of
//      each segment before the sample was measured: those lines were evicted
//      before use and read again, +64 MB per launch and slower.)
// If at least k were collected and no list overflowed, a radix select over the
// lists gives the exact k-th largest key; keys above it are kept and ties keep
// their lowest positions.  If some list overflowed but all the hits fit the
// buffer (they cluster in a few warps' segments, as the highest scores of a real
// row cluster on recent positions), the row is collected once more with every
// warp's hits packed after those of the warps before it, and selected from there.  Because the lists are position-ordered and the
// segments increase with the warp index, every warp writes its kept positions
// straight to their output slots from per-warp prefix counts: the output is in
// ascending order without a sort.  Rows with at most `capacity` positions take
// every position as a candidate.  Otherwise the row falls back to a radix select
// over all 32 key bits (three histogram passes) and an index-ordered selection.
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;
constexpr int kCap = 8192;     // candidate capacity of the fast path (power of two)
constexpr int kSample = 8192;  // sample size for the threshold (runs of 32)
constexpr int kMaxK = 4096;    // largest k of the fast path (power of two)
constexpr int kWarpCap = kCap / kWarps;  // candidates per warp list (512)
constexpr int kSpan = 32 * 16;           // positions a warp scans per iteration (16 per lane)
constexpr int kPrefetchAhead = 1024;     // positions each warp keeps requested into L2 ahead of its scan

struct TopkSmem {
  int hist[kBins];
  unsigned long long cand[kCap];
  int warp_tot[32];
  int sel_bin, sel_above;
  int wcnt[kWarps], wgt[kWarps], weq[kWarps];  // per-warp candidate lists: length, > T, == T
  int woff[kWarps];                             // packed lists (select_packed): start of each in cand
  // where the row's selection goes besides the output row (see RowOut), kept here rather than in
  // registers, which the collection pass needs
  int pos_base;
  const int32_t* map;
  float* score_out;
};

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

// Histogram of ((key >> shift) & bmask) over elements with (key & mask) == prefix.
__device__ __forceinline__ void add_to_hist(int* hist, uint32_t key, bool in_row, uint32_t mask, uint32_t prefix,
                                            int shift, uint32_t bmask) {
  const bool hit = in_row && (key & mask) == prefix;
  const uint32_t bin = (key >> shift) & bmask;
  if (hit) atomicAdd(&hist[bin], 1);
}

// Visit every element of the row (float4 loads when the row is 16-byte aligned).
template <typename F>
__device__ __forceinline__ void for_row(const float* s, int n, F&& f) {
  if ((reinterpret_cast<uintptr_t>(s) & 15) == 0) {
    const int n4 = n & ~3;
    for (int base = threadIdx.x * 4; base < ((n + 4 * kThreads - 1) / (4 * kThreads)) * 4 * kThreads;
         base += 4 * kThreads) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (base < n4) {
        v = __ldg(reinterpret_cast<const float4*>(s + base));
      } else if (base < n) {
        v.x = __ldg(s + base);
        if (base + 1 < n) v.y = __ldg(s + base + 1);
        if (base + 2 < n) v.z = __ldg(s + base + 2);
      }
      f(base, v.x, base < n);
      f(base + 1, v.y, base + 1 < n);
      f(base + 2, v.z, base + 2 < n);
      f(base + 3, v.w, base + 3 < n);
    }
  } else {
    for (int base = 0; base < n; base += kThreads) {
      const int j = base + threadIdx.x;
      f(j, j < n ? __ldg(s + j) : 0.f, j < n);
    }
  }
}

// Pick the bin B (scanning from the top) with count(> B) < remaining <= count(>= B).
__device__ __forceinline__ void find_bin(TopkSmem& sm, int nb, int remaining) {
  const int per = nb / kThreads > 0 ? nb / kThreads : 1;
  const bool owns = threadIdx.x * per < nb;
  const int hi_bin = nb - 1 - threadIdx.x * per;
  int local = 0;
  if (owns)
    for (int x = 0; x < per; ++x) local += sm.hist[hi_bin - x];
  int total;
  const int before = block_exclusive_scan(owns ? local : 0, sm.warp_tot, total);
  if (owns && before < remaining && before + local >= remaining) {
    int acc = before;
    for (int x = 0; x < per; ++x) {
      const int c = sm.hist[hi_bin - x];
      if (acc + c >= remaining) {
        sm.sel_bin = hi_bin - x;
        sm.sel_above = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// The want-th largest of n keys in shared memory (radix select on 12, 12, 8
// bits; `passes` < 3 stops early and returns the prefix of the decided bits).  `rem`
// returns how many keys equal to the result are within the top
// `want` (1 <= rem <= count of that key).
__device__ uint32_t radix_select(TopkSmem& sm, const uint32_t* keys, int n, int want, int& rem, int passes = 3) {
  uint32_t prefix = 0, mask = 0;
  int remaining = want;
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = shifts[pass];
    const uint32_t bmask = (1u << widths[pass]) - 1u;
    const int nb = 1 << widths[pass];
    for (int i = threadIdx.x; i < nb; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + threadIdx.x;
      add_to_hist(sm.hist, i < n ? keys[i] : 0u, i < n, mask, prefix, shift, bmask);
    }
    __syncthreads();
    find_bin(sm, nb, remaining);
    remaining -= sm.sel_above;
    prefix |= static_cast<uint32_t>(sm.sel_bin) << shift;
    mask |= bmask << shift;
    __syncthreads();
  }
  rem = remaining;
  return prefix;
}

// The k-th largest key among the per-warp candidate lists (warp w's list is
// cand[w * kWarpCap .. + wcnt[w])).
// `mask_out` gives the key bits the result decides: compare (key & mask_out) with it.
template <bool kPacked>
__device__ uint32_t radix_select_lists(TopkSmem& sm, int k, int& rem, uint32_t& mask_out) {
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const uint32_t bmask = (1u << widths[pass]) - 1u;
    const int nb = 1 << widths[pass];
    for (int i = threadIdx.x; i < nb; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    {  // each warp histograms its own list
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
      const int cnt = sm.wcnt[warp];
      const unsigned long long* list = sm.cand + (kPacked ? sm.woff[warp] : warp * kWarpCap);
      for (int j0 = 0; j0 < cnt; j0 += 32) {
        const int j = j0 + lane;
        const bool in = j < cnt;
        const uint32_t key = in ? static_cast<uint32_t>(list[j] >> 32) : 0u;
        add_to_hist(sm.hist, key, in, mask, prefix, shift, bmask);
      }
    }
    __syncthreads();
    find_bin(sm, nb, remaining);
    remaining -= sm.sel_above;
    prefix |= static_cast<uint32_t>(sm.sel_bin) << shift;
    mask |= bmask << shift;
    const bool exact = sm.hist[sm.sel_bin] == remaining;
    __syncthreads();
    if (exact) break;  // every key of the bin is taken: the prefix already separates them
  }
  rem = remaining;
  mask_out = mask;
  return prefix;
}

// Output slot i of the row (o) receives position j.  kPlain: as j.  Otherwise as
// sm.pos_base + j (or sm.map[j]), and sm.score_out[i] receives the score s[j] when it is set;
// only `o` travels in registers.
template <bool kPlain>
__device__ __forceinline__ void emit(const TopkSmem& sm, int32_t* o, const float* s, int i, int j) {
  if constexpr (kPlain) {
    o[i] = j;
  } else {
    const int32_t* map = sm.map;
    o[i] = map ? __ldg(map + j) : sm.pos_base + j;
    if (float* so = sm.score_out) so[i] = __ldg(s + j);
  }
}
template <bool kPlain>
__device__ __forceinline__ void emit_pad(const TopkSmem& sm, int32_t* o, int i) {
  o[i] = -1;
  if constexpr (!kPlain) {
    if (float* so = sm.score_out) so[i] = -INFINITY;
  }
}

template <bool kPlain>
__device__ void topk_slow(TopkSmem& sm, const float* s, int n, int k, int32_t* o) {
  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const uint32_t bmask = (1u << widths[pass]) - 1u;
    const int nb = 1 << widths[pass];
    for (int i = threadIdx.x; i < nb; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for_row(s, n, [&](int, float x, bool in) { add_to_hist(sm.hist, order_key(x), in, mask, prefix, shift, bmask); });
    __syncthreads();
    find_bin(sm, nb, remaining);
    const int bin = sm.sel_bin;
    remaining -= sm.sel_above;
    prefix |= static_cast<uint32_t>(bin) << shift;
    mask |= bmask << shift;
    const bool exact = sm.hist[bin] == remaining;
    __syncthreads();
    if (exact) break;
  }
  const int seg = (n + kThreads - 1) / kThreads;
  const int lo = min(n, static_cast<int>(threadIdx.x) * seg), hi = min(n, lo + seg);
  int gt = 0, eq = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(__ldg(s + j)) & mask;
    gt += key > prefix;
    eq += key == prefix;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, sm.warp_tot, tot);
  const int eq_take = max(0, min(eq, remaining - eq_before));
  const int out_before = block_exclusive_scan(gt + eq_take, sm.warp_tot, tot);
  int pos = out_before, eq_seen = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = order_key(__ldg(s + j)) & mask;
    bool keep = key > prefix;
    if (key == prefix) {
      keep = eq_seen < eq_take;
      ++eq_seen;
    }
    if (keep) emit<kPlain>(sm, o, s, pos++, j);
  }
}

// Positions visible to query token t (0..p).
__device__ __forceinline__ int visible(const int32_t* seq_lens, const int32_t* qsl, int batch, int t) {
  const int b = seq_of_token(qsl, batch, t);
  const int q0 = __ldg(qsl + b), n_q = __ldg(qsl + b + 1) - q0;
  return __ldg(seq_lens + b) - n_q + (t - q0) + 1;
}

// The exact top-k among the per-warp candidate lists (list w: `list_off` entries into cand for the
// calling warp, wcnt[w] long; kPacked: the lists sit at woff[w]), written in position order.
template <bool kPlain, bool kPacked>
__device__ __forceinline__ void select_from_lists(TopkSmem& sm, const float* __restrict__ s, int k, int32_t* o,
                                                  int list_off, int count) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long* list = sm.cand + list_off;
  // ---- exact k-th largest key T among the candidates ----
  int need_eq;
  uint32_t tmask;
  const uint32_t T = radix_select_lists<kPacked>(sm, k, need_eq, tmask);
  // ---- every warp counts its keys above T and equal to T ----
  {
    int gt = 0, eq = 0;
    for (int j = lane; j < count; j += 32) {
      const uint32_t key = static_cast<uint32_t>(list[j] >> 32) & tmask;
      gt += key > T;
      eq += key == T;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      gt += __shfl_xor_sync(0xffffffffu, gt, o2);
      eq += __shfl_xor_sync(0xffffffffu, eq, o2);
    }
    if (lane == 0) {
      sm.wgt[warp] = gt;
      sm.weq[warp] = eq;
    }
  }
  __syncthreads();
  // ---- lists are in position order and warps cover increasing segments: each warp writes its
  // kept positions straight to their output slots (ties keep the lowest positions) ----
  int eq_before = 0, out_off = 0;
  for (int w = 0; w < warp; ++w) {
    const int take = max(0, min(sm.weq[w], need_eq - eq_before));
    eq_before += sm.weq[w];
    out_off += sm.wgt[w] + take;
  }
  const int take_eq = max(0, min(sm.weq[warp], need_eq - eq_before));
  int written = 0, ties_seen = 0;
  for (int j0 = 0; j0 < count; j0 += 32) {
    const int j = j0 + lane;
    uint32_t key = 0;
    int pos = 0;
    if (j < count) {
      key = static_cast<uint32_t>(list[j] >> 32) & tmask;
      pos = static_cast<int>(~static_cast<uint32_t>(list[j] & 0xFFFFFFFFull));
    }
    const bool is_eq = j < count && key == T;
    const uint32_t eq_mask = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t below = (1u << lane) - 1u;
    const bool keep = j < count && (key > T || (is_eq && ties_seen + __popc(eq_mask & below) < take_eq));
    const uint32_t keep_mask = __ballot_sync(0xffffffffu, keep);
    if (keep) emit<kPlain>(sm, o, s, out_off + written + __popc(keep_mask & below), pos);
    written += __popc(keep_mask);
    ties_seen += __popc(eq_mask);
  }
}

// Rows whose hits overflow some warp's list but fit the buffer together: the hits cluster in a few
// warps' segments (as the highest scores of a real row cluster on recent positions).  Each warp
// collects its hits again (same row, same threshold) after those of the warps before it, so the
// lists stay in position order, and the selection runs over the packed lists.
template <bool kPlain>
__device__ void select_packed(TopkSmem& sm, const float* __restrict__ s, int k, int32_t* o, int p_lo,
                                           int p_hi, uint32_t thr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int before = 0;
  for (int w = 0; w < warp; ++w) before += sm.wcnt[w];
  __syncthreads();  // every warp has read the counts before any list is overwritten
  unsigned long long* list = sm.cand + before;
  const int cap = kCap - before;
  int count = 0;
  for (int base = p_lo; base < p_hi; base += kSpan) {
    const int p0 = base + 16 * lane;
    uint32_t hit = 0;
    uint32_t keys[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      const int j = p0 + 4 * u;
      if (j + 3 < p_hi) {
        v = __ldg(reinterpret_cast<const float4*>(s + j));
      } else {
        if (j < p_hi) v.x = __ldg(s + j);
        if (j + 1 < p_hi) v.y = __ldg(s + j + 1);
        if (j + 2 < p_hi) v.z = __ldg(s + j + 2);
      }
      keys[4 * u] = order_key(v.x);
      keys[4 * u + 1] = order_key(v.y);
      keys[4 * u + 2] = order_key(v.z);
      keys[4 * u + 3] = order_key(v.w);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (p0 + e < p_hi && keys[e] >= thr) hit |= 1u << e;
    const int cnt = __popc(hit);
    int incl = cnt;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o2);
      if (lane >= o2) incl += y;
    }
    int pos = count + incl - cnt;
    while (hit) {
      const int e = __ffs(hit) - 1;
      hit &= hit - 1;
      if (pos < cap)
        list[pos] = (static_cast<unsigned long long>(keys[e]) << 32) | static_cast<uint32_t>(~(p0 + e));
      ++pos;
    }
    count += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) sm.woff[warp] = before;
  __syncthreads();
  select_from_lists<kPlain, true>(sm, s, k, o, before, sm.wcnt[warp]);
}

// The top-k of the n scores s[0..n) (every thread of the CTA; each branch below is CTA-uniform).
template <bool kPlain>
__device__ void topk_core(TopkSmem& sm, const float* __restrict__ s, int n, int k, int32_t* o) {
  if (n <= k) {
    for (int i = threadIdx.x; i < k; i += kThreads) {
      if (i < n) emit<kPlain>(sm, o, s, i, i);
      else emit_pad<kPlain>(sm, o, i);
    }
    return;
  }
  if (k > kMaxK) {
    topk_slow<kPlain>(sm, s, n, k, o);
    return;
  }
  // Segment of warp w in the collection pass below.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (n + kWarps * kSpan - 1) / (kWarps * kSpan) * kSpan;
  const int p_lo = min(n, warp * seg), p_hi = min(n, p_lo + seg);
  const bool aligned = (reinterpret_cast<uintptr_t>(s) & 15) == 0;
  const auto prefetch = [&](int from, int to) {  // whole 16-byte granules of positions [from, to)
    const int bytes = ((to - from) * 4) & ~15;
    if (bytes > 0) prefetch_l2_bulk(s + from, static_cast<uint32_t>(bytes));
  };
  // ---- threshold from a sample (skipped when every position fits) ----
  uint32_t thr = 0;  // keep keys >= thr
  if (n > kCap) {
    // sample: kSample / 32 runs of 32 consecutive positions (a 128-byte line each when the row is
    // aligned), evenly spread over the row; thread f reads 4 positions of run f / 8
    uint32_t* samp = reinterpret_cast<uint32_t*>(sm.cand);
    constexpr int runs = kSample / 32;
#pragma unroll 4
    for (int f = threadIdx.x; f < kSample / 4; f += kThreads) {
      const int j = static_cast<int>((static_cast<int64_t>(f >> 3) * (n - 32)) / (runs - 1));
      if (aligned) {  // runs start on a 128-byte boundary of the row: whole-line vector loads
        const float4 v = __ldg(reinterpret_cast<const float4*>(s + (j & ~31) + 4 * (f & 7)));
        *reinterpret_cast<uint4*>(samp + 4 * f) = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
      } else {
#pragma unroll
        for (int x = 0; x < 4; ++x) samp[4 * f + x] = order_key(__ldg(s + j + 4 * (f & 7) + x));
      }
    }
    // rank of the threshold in the sample: expected rank of the k-th largest plus a margin
    const int r = static_cast<int>((static_cast<int64_t>(k) * kSample + n - 1) / n);
    const int want = min(kSample, r + 4 * static_cast<int>(sqrtf(static_cast<float>(r))) + 16);
    __syncthreads();
    int rem;
    thr = radix_select(sm, samp, kSample, want, rem, 2);  // 24 bits: the threshold's bin is kept whole
  }
  if (!aligned) {  // rows that are not 16-byte aligned
    topk_slow<kPlain>(sm, s, n, k, o);
    return;
  }
  // ---- one pass: warp w scans its own contiguous segment and appends every key >= thr, in
  // position order, to its own list (16 keys per lane per iteration, the next 16 in flight,
  // and the L2 request kPrefetchAhead positions ahead) ----
  unsigned long long* list = sm.cand + warp * kWarpCap;
  const auto load = [&](int p0, float4 (&v)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = p0 + 4 * u;
      if (j + 3 < p_hi) {
        v[u] = __ldg(reinterpret_cast<const float4*>(s + j));
      } else {
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < p_hi) v[u].x = __ldg(s + j);
        if (j + 1 < p_hi) v[u].y = __ldg(s + j + 1);
        if (j + 2 < p_hi) v[u].z = __ldg(s + j + 2);
      }
    }
  };
  int count = 0;  // warp-uniform length of this warp's list
  {
    float4 cur[4], nxt[4];
    if (p_lo < p_hi) load(p_lo + 16 * lane, cur);
    for (int base = p_lo; base < p_hi; base += kSpan) {
      const int p0 = base + 16 * lane;
      if (lane == 0 && base + kPrefetchAhead < p_hi)
        prefetch(base + kPrefetchAhead, min(p_hi, base + kPrefetchAhead + kSpan));
      if (base + kSpan < p_hi) load(p0 + kSpan, nxt);
      uint32_t keys[16];
      uint32_t hit = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        keys[4 * u] = order_key(cur[u].x);
        keys[4 * u + 1] = order_key(cur[u].y);
        keys[4 * u + 2] = order_key(cur[u].z);
        keys[4 * u + 3] = order_key(cur[u].w);
      }
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (p0 + e < p_hi && keys[e] >= thr) hit |= 1u << e;
      const int cnt = __popc(hit);
      int incl = cnt;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o2);
        if (lane >= o2) incl += y;
      }
      int pos = count + incl - cnt;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (hit & (1u << e)) {
          if (pos < kWarpCap)
            list[pos] = (static_cast<unsigned long long>(keys[e]) << 32) | static_cast<uint32_t>(~(p0 + e));
          ++pos;
        }
      }
      count += __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
      for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
    }
  }
  if (lane == 0) sm.wcnt[warp] = count;
  __syncthreads();
  int n_cand = 0;
  bool over = false;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    n_cand += sm.wcnt[w];
    over |= sm.wcnt[w] > kWarpCap;
  }
  if (over && n_cand >= k && n_cand <= kCap) {  // clustered hits: collect them again, packed
    select_packed<kPlain>(sm, s, k, o, p_lo, p_hi, thr);
    return;
  }
  if (n_cand < k || over) {  // the sample's guess missed: exact radix select over the row
    topk_slow<kPlain>(sm, s, n, k, o);
    return;
  }
  select_from_lists<kPlain, false>(sm, s, k, o, warp * kWarpCap, count);
}

// One CTA per row while the rows fit one wave of resident CTAs.  Beyond that the grid is
// one wave and CTA c takes the rows c, 2G-1-c, 2G+c, 4G-1-c, ... (G = gridDim.x): every
// pass over G rows runs in the opposite direction to the one before, so a CTA pairs a
// front row with a back row.  In causal prefill, where a row's length grows with its
// position, this evens the CTAs' work in the manner of front/back context pairing.
//
// Rows longer than the batch can fill the GPU with are split (stage 1 and 2): stage 1 takes the
// n_seg contiguous segments of every row as rows of their own and writes each segment's top-k
// (positions and scores) as candidates; stage 2 selects the top-k of each row's n_seg * k
// candidates.  A position of the row's top-k is in its segment's top-k (at most k - 1 positions
// of the segment rank above it), so the candidates hold the answer; they are laid out in segment
// order with ascending positions inside, so candidate order is position order and stage 2's ties
// (lower index) and ascending output are the row's.
template <bool kPlain>
__global__ void __launch_bounds__(kThreads, 2) topk_kernel(int k, const float* __restrict__ scores, int64_t stride,
                                                        const int32_t* __restrict__ seq_lens,
                                                        const int32_t* __restrict__ qsl, int batch, int tok_begin,
                                                        int n_rows, int32_t* __restrict__ out, int stage, int n_seg,
                                                        int32_t* __restrict__ cand_pos,
                                                        float* __restrict__ cand_score) {
  extern __shared__ uint8_t smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  const int G = static_cast<int>(gridDim.x);
  for (int base = 0, pass = 0; base < n_rows; base += G, ++pass) {
    const int row = base + ((pass & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
    if constexpr (kPlain) {  // one row per CTA pass, positions written as they are
      if (row < n_rows)
        topk_core<true>(sm, scores + static_cast<int64_t>(row) * stride,
                        visible(seq_lens, qsl, batch, tok_begin + row), k, out + static_cast<int64_t>(row) * k);
    } else if (row < n_rows) {
      const float* s;
      int n;
      int32_t* o = out + static_cast<int64_t>(row) * k;
      int pos_base = 0;
      const int32_t* map = nullptr;
      float* score_out = nullptr;
      if (stage == 2) {
        const int64_t c0 = static_cast<int64_t>(row) * n_seg * k;
        s = cand_score + c0;
        n = n_seg * k;
        map = cand_pos + c0;
      } else {
        const int tr = stage == 1 ? row / n_seg : row;
        n = visible(seq_lens, qsl, batch, tok_begin + tr);
        s = scores + static_cast<int64_t>(tr) * stride;
        if (stage == 1) {
          const int len = ((n + n_seg - 1) / n_seg + 3) & ~3;  // 16-byte aligned segment starts
          const int lo = min(n, (row % n_seg) * len), hi = min(n, lo + len);
          const int64_t c0 = static_cast<int64_t>(row) * k;
          s += lo;
          n = hi - lo;
          o = cand_pos + c0;
          pos_base = lo;
          score_out = cand_score + c0;
        }
      }
      if (threadIdx.x == 0) {
        sm.pos_base = pos_base;
        sm.map = map;
        sm.score_out = score_out;
      }
      __syncthreads();
      topk_core<false>(sm, s, n, k, o);
    }
    __syncthreads();  // shared memory is reused by the next row
  }
}


}  // namespace

int topk_wave() {
  static std::atomic<int> wave[kMaxDeviceSlots] = {};
  const int dev = current_device_index();
  if (dev < 0) return 0;
  int w = wave[dev].load(std::memory_order_acquire);
  if (w == 0) {
    const size_t smem = sizeof(TopkSmem);
    if (cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
      return 0;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel<true>, kThreads, smem) != cudaSuccess ||
        per_sm <= 0)
      return 0;
    w = per_sm * device_sm_count();
    wave[dev].store(w, std::memory_order_release);
  }
  return w;
}

smla_status_t launch_topk(int top_k, const float* scores, int64_t scores_stride, const int32_t* seq_lens,
                          const int32_t* query_start_loc, int batch, int tok_begin, int tok_end, int32_t* topk_idx,
                          cudaStream_t stream, unsigned* err, void* split_ws, size_t split_ws_bytes) {
  (void)err;
  const int rows = tok_end - tok_begin;
  if (rows <= 0) return SMLA_OK;
  const int wave = topk_wave();
  if (wave <= 0) return SMLA_ERR_CUDA;
  // Fewer rows than a wave of CTAs, and rows long against k: split each row into n_seg segments
  // (stage 1, rows x n_seg CTAs) and merge their candidates (stage 2).  A pass costs a fixed
  // ~23 us (sample, selections) plus its positions, so two passes over n / n_seg and n_seg * k
  // positions beat one over n only for rows of more than ~64k positions; n_seg ~ sqrt(n / k)
  // balances the two passes.
  int n_seg = 1;
  if (split_ws != nullptr && rows < wave && top_k <= kMaxK && scores_stride >= 64 * static_cast<int64_t>(top_k)) {
    int by_len = 1;
    while (static_cast<int64_t>(by_len + 1) * (by_len + 1) * top_k <= scores_stride) ++by_len;
    n_seg = min(min(wave / rows, by_len), kMaxTopkSplitRows / rows);
    while (n_seg > 1 && topk_split_bytes(rows * n_seg, top_k) > split_ws_bytes) --n_seg;
  }
  if (n_seg >= 2) {
    const int seg_rows = rows * n_seg;
    int32_t* cand_pos = static_cast<int32_t*>(split_ws);
    float* cand_score = reinterpret_cast<float*>(static_cast<uint8_t*>(split_ws) + topk_split_bytes(seg_rows, top_k) / 2);
    topk_kernel<false><<<min(seg_rows, wave), kThreads, sizeof(TopkSmem), stream>>>(
        top_k, scores, scores_stride, seq_lens, query_start_loc, batch, tok_begin, seg_rows, topk_idx, 1, n_seg,
        cand_pos, cand_score);
    if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
    topk_kernel<false><<<rows, kThreads, sizeof(TopkSmem), stream>>>(top_k, scores, scores_stride, seq_lens,
                                                              query_start_loc, batch, tok_begin, rows, topk_idx, 2,
                                                              n_seg, cand_pos, cand_score);
    return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
  }
  const int grid = rows < wave ? rows : wave;
  topk_kernel<true><<<grid, kThreads, sizeof(TopkSmem), stream>>>(top_k, scores, scores_stride, seq_lens, query_start_loc,
                                                             batch, tok_begin, rows, topk_idx, 0, 1, nullptr, nullptr);
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
