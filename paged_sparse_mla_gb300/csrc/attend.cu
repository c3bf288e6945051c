// smla_attend: latent MQA attention of each query token over its top-k positions.
//
// [AgentX "Kimi K3"], [GLM-5.3 "What is new"]: MLA keeps one latent KV shared
// by all 64 query heads, so attention is MQA over the latent; V is the latent.
// [AgentX "DeepSeek V4"]: sparse MLA attends only over the top-k entries, and
// gathering them dominates.  [AgentX "Kimi K3"] (DCP): the output carries
// log-sum-exp statistics so partial results can be merged.
//
// Design (sm_103a, one persistent CTA per SM, one query token at a time):
//   * 64 selected positions form a tile, and the tile buffer is double-buffered
//     so that gathering tile t+1 overlaps the MMAs and the softmax of tile t.
//     Eleven producer warps translate the logical positions through the block
//     table two tiles ahead, read the 656-byte records (one warp per record,
//     two coalesced loads), dequantise the E4M3 latent with its per-128 fp32
//     scales to bf16, and write the tile as 9 chunks of [64 keys x 64 dims] with
//     the 128-byte swizzle (8 latent chunks + 1 rope chunk); the query is staged
//     the same way (64 heads).
//   * MMA1 (warp 8): S^T[key, head] = Khat[key, :] . q[head, :] over 576 dims,
//     M = 64 keys, N = 64 heads, fp32 in tensor memory, two buffers.  Key i of
//     the tile sits in TMEM lane (i % 16) + 32 (i / 16).
//   * Softmax (warps 0-7; warp w holds keys 16 (w % 4) .. + 15 and heads
//     32 (w / 4) .. + 31): the 16x32bx2 tensor-memory load gives lane l of the
//     warp key l % 16 and 16 of the 32 heads (half l / 16), so every lane has
//     scores (the other 16 lanes of each TMEM sub-partition hold none);
//     per-head tile maxima by shuffles within each half-warp, online softmax
//     with lazy rescaling (the running max only moves when a head's tile max
//     exceeds it by 2^8), P^T[key, head] written as bf16 into the rope chunk
//     (free after MMA1), per-thread partial row sums reduced within the
//     half-warps at the end of the token.
//   * MMA2: O^T[dim, head] += V^T[dim, key] . P^T[key, head] with both operands
//     MN-major: the same swizzled latent chunks serve as V^T without a
//     transpose; M = 128 dims x 4 tiles, N = 64 heads, K = 64 keys.  The MMA
//     warp polls both: MMA2 of a tile as soon as its probabilities are written
//     (it releases that buffer to the producers), MMA1 of the next tile as soon
//     as it is gathered (the next scores are computed while the softmax works).
//   * Epilogue: O^T / l -> bf16 out[t, h, d] (thread = dim, coalesced) and
//     lse = ln(sum) from the running max and the reduced row sums.
#include <cstring>

#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kTile = 64;      // keys per tile (MMA1 M)
constexpr int kHeads = 64;     // MMA N: query heads (zero padded)
// Warp roles: warpgroups 0-1 = softmax (warps 0-7); warp 8 = MMA issuer; warps 9-19 =
// producers.  setmaxnreg moves registers to the softmax warpgroups.
constexpr int kSoftmaxThreads = 256;
constexpr int kMmaWarp = 8;
constexpr int kFirstProducerWarp = 9;
constexpr int kProducerThreads = 32 * 11;
constexpr int kThreads = 32 * 20;
constexpr int kLaunchRegs = 96;        // per thread at launch (65536 / 640, rounded down to 8)
constexpr int kSoftmaxRegs = 120;
constexpr int kOtherRegs = 80;         // 256*120 + 384*80 <= 640*96
static_assert(kSoftmaxThreads * kSoftmaxRegs + (kThreads - kSoftmaxThreads) * kOtherRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int NCH>
struct __align__(1024) AttnSmem {
  uint8_t kv[2][NCH][kTile * 128];  // buffer, chunk c: [64 keys][64 dims] bf16, swizzled; chunk NCH-1: rope, then P^T
  uint8_t q[NCH][kHeads * 128];     // chunk c: [64 heads][64 dims] bf16, swizzled
  const uint8_t* rec[3][kTile];     // record address per key of tiles t, t+1, t+2 (nullptr = masked)
  float red[4][kHeads];
  float m_tile[kHeads];
  float m_run[kHeads];
  float alpha[kHeads];
  float l_fin[kHeads];              // 1 / row sum per head
  int ntiles[2];                    // tiles of the unit in each tok slot
  int tbeg[2];                      // its first tile within the row
  uint64_t tok_full[2], tok_empty[2];
  uint64_t q_full, q_empty;
  uint64_t kv_full[2], kv_empty[2], s_full[2], s_empty[2], p_full[2];
  uint64_t o_done, final_bar;
  uint32_t tmem_slot;
  int abort;
};

struct AttnArgs {
  KernelLayout L;
  int n_heads, top_k, layer;
  float scale_log2;  // softmax_scale * log2(e)
  const uint8_t* pool;
  const __nv_bfloat16* q;
  const __nv_bfloat16* q_pe;
  const int32_t* topk;  // rows relative to tok_begin
  const int32_t* block_table;
  int bt_stride;
  int64_t max_pos;  // bt_stride * block_size: positions at or past it have no block-table entry
  const int32_t* qsl;
  int batch, tok_begin, n_rows;
  __nv_bfloat16* out;
  float* lse;
  unsigned* err;
  // host tier: records of block b live at host_records + (host_block_map[b] * n_layers + layer) *
  // block_size * rec_stride when host_block_map[b] >= 0 (nullptr map = every record in the pool)
  const uint8_t* host_records;
  const int32_t* host_block_map;
  int64_t n_host_blocks;
  // 1: the query tile is loaded by the tensor-memory-access unit (nine 2-D tensor-map copies of
  // 64 heads x 64 dims, 128-byte swizzled as the MMA reads them); 0: by the producer threads
  int q_tma;
  // Split of each row's tiles into n_splits contiguous ranges (work units u = row * n_splits +
  // split).  With n_splits > 1 a unit writes its normalised partial output (fp32) and its lse to
  // part_out [n_splits][n_rows][n_heads][d_latent] and part_lse [n_splits][n_rows][n_heads].
  int n_splits;
  float* part_out;
  float* part_lse;
  // Balanced units (mode 2): CTA c takes the nominal tiles [c * T / G, (c + 1) * T / G) of the
  // n_rows * row_tiles_nom tiles, G = gridDim.x.  A row is then split over at most two CTAs: the
  // first CTA's part goes to partial slot 2c + 1, the second's to slot 2 (c + 1); whole rows are
  // written directly.
  int row_tiles_nom;
  int mode;  // 0 plain, 1 split, 2 balanced
};

// Work units of a CTA: kMode 0, rows c, c + G, ...; kMode 1, (row, split) pairs u = c, c + G, ...
// with u = row * n_splits + split (the split's tile range follows from the row's valid tiles);
// kMode 2, the rows its balanced range of nominal tiles meets, with tiles [ta, tb) of each.
// slot: the partial-output slot of the unit, or -1 when it writes the row's output itself.
template <int kMode>
__device__ __forceinline__ bool unit_at(const AttnArgs& A, int i, int& tr, int& split, int& ta, int& tb, int& slot) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  if constexpr (kMode == 2) {
    const int64_t T = A.row_tiles_nom, tot = static_cast<int64_t>(A.n_rows) * T;
    const int64_t g0 = c * tot / G, g1 = (c + 1) * tot / G;
    const int64_t r = g0 / T + i;
    if (r * T >= g1) return false;
    tr = static_cast<int>(r);
    split = 0;
    ta = static_cast<int>(max(g0, r * T) - r * T);
    tb = static_cast<int>(min(g1, (r + 1) * T) - r * T);
    slot = (ta == 0 && tb == T) ? -1 : (ta > 0 ? 2 * c : 2 * c + 1);
    return true;
  } else {
    const int n_splits = kMode == 1 ? A.n_splits : 1;
    const int u = c + i * G;
    if (u >= A.n_rows * n_splits) return false;
    tr = u / n_splits;
    split = u % n_splits;
    ta = 0;
    tb = 0x7fffffff;
    slot = kMode == 1 ? split * A.n_rows + tr : -1;
    return true;
  }
}

// Within each half-warp: lane 16 u + l holds, in v[0], the sum over the half's 16 lanes of value l.
__device__ __forceinline__ void half_transpose_sum16(float (&v)[16], int lane) {
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int off = 8 >> st;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}

// tcgen05.ld 16x32bx2: 16 TMEM lanes read twice, the second time `kSplit` columns further on;
// thread t holds lane t % 16, columns (t / 16) * kSplit + 0 .. 15.
template <int kSplit>
__device__ __forceinline__ void tmem_ld16x32bx2_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr), "n"(kSplit));
}

// Non-blocking test of the phase of `bar` with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// 2^x with the hardware approximation (MUFU; relative error ~2^-22, -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Eight bf16 values from 2-byte aligned memory; entries at or beyond `avail` read as zero.
__device__ __forceinline__ uint4 load_bf16x8_padded(const uint16_t* src, int avail) {
  uint32_t w[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const uint32_t lo = (2 * x < avail) ? src[2 * x] : 0u;
    const uint32_t hi = (2 * x + 1 < avail) ? src[2 * x + 1] : 0u;
    w[x] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Producer unit -> (key, piece).  A warp's 32 consecutive units cover 8
// consecutive keys x 4 consecutive pieces, with lane & 7 selecting the key: the
// eight lanes of each quarter-warp then store the same piece of 8 consecutive
// rows, which the 128-byte swizzle spreads over all 32 banks, and each key's 4
// pieces (64 contiguous record bytes) are read by one warp instruction.
__device__ __forceinline__ void latent_unit(int u, int parts, int& key, int& part) {
  const int lane = u & 31, w = u >> 5;
  const int pgroups = parts / 4;
  key = 8 * (w / pgroups) + (lane & 7);
  part = 4 * (w % pgroups) + (lane >> 3);
}
__device__ __forceinline__ void rope_unit(int ur, int& key, int& v) {
  const int lane = ur & 31, w = ur >> 5;
  key = 8 * (w >> 1) + (lane & 7);
  v = 4 * (w & 1) + (lane >> 3);
}

// Loads for one batch of the producer unit stream (see the key-tile loop):
// latent units fetch 16 E4M3 codes and their fp32 scale, rope units fetch 8
// bf16 (zero padded past d_rope).  Masked keys (nullptr record) read as zero.
constexpr int kBatch = 4;
__device__ __forceinline__ void load_units(const uint8_t* const* rec, int u0, int n_lat, int n_units, int parts,
                                           int DL, int DR, int qtile, int n_scales, bool rope16,
                                           uint4 (&val)[kBatch], float (&sc)[kBatch]) {
#pragma unroll
  for (int b = 0; b < kBatch; ++b) {
    const int u = u0 + b * kProducerThreads;
    val[b] = make_uint4(0, 0, 0, 0);
    sc[b] = 0.f;
    if (u < n_lat) {
      int key, part;
      latent_unit(u, parts, key, part);
      const uint8_t* r = rec[key];
      if (r != nullptr) {
        val[b] = __ldg(reinterpret_cast<const uint4*>(r) + part);
        sc[b] = __ldg(reinterpret_cast<const float*>(r + DL) + (part * 16) / qtile);
      }
    } else if (u < n_units) {
      int key, v;
      rope_unit(u - n_lat, key, v);
      const uint8_t* r = rec[key];
      if (r != nullptr && v * 8 < DR) {
        const uint8_t* src = r + DL + 4 * n_scales + v * 16;
        if (rope16 && v * 8 + 8 <= DR)
          val[b] = __ldg(reinterpret_cast<const uint4*>(src));
        else
          val[b] = load_bf16x8_padded(reinterpret_cast<const uint16_t*>(src), DR - v * 8);
      }
    }
  }
}

// (a.x * s, a.y * s) with one packed fp32 multiply (each product rounded as by a scalar multiply).
__device__ __forceinline__ float2 mul2(float2 a, float s) {
  uint64_t r;
  asm("{\n\t.reg .b64 x, y;\n\t"
      "mov.b64 x, {%1, %2};\n\t"
      "mov.b64 y, {%3, %3};\n\t"
      "mul.rn.f32x2 %0, x, y;\n\t}"
      : "=l"(r)
      : "f"(a.x), "f"(a.y), "f"(s));
  return make_float2(__uint_as_float(static_cast<uint32_t>(r)), __uint_as_float(static_cast<uint32_t>(r >> 32)));
}

// 16 E4M3 codes (little-endian in `codes`) times `sc` -> 16 bf16 in two 16-byte words.
__device__ __forceinline__ void dequant16(const uint4& codes, float sc, uint4& o0, uint4& o1) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t ow[8];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(cw[x] & 0xFFFFu), __NV_E4M3);
    const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(cw[x] >> 16), __NV_E4M3);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    const float2 p01 = mul2(f01, sc), p23 = mul2(f23, sc);
    ow[2 * x] = pack_bf16x2(p01.x, p01.y);
    ow[2 * x + 1] = pack_bf16x2(p23.x, p23.y);
  }
  o0 = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  o1 = make_uint4(ow[4], ow[5], ow[6], ow[7]);
}

// Number of 128-key tiles a row needs: one past the last valid entry.  A row
// whose final entry is valid needs every tile (one load); otherwise the warp
// scans the row with all of its loads in flight at once.
__device__ __forceinline__ int row_tiles(const int32_t* row, int k, int lane) {
  if (__ldg(row + k - 1) >= 0) return (k + kTile - 1) / kTile;
  int last = -1;
  constexpr int kUnroll = 8;
  for (int base = 0; base < k; base += 32 * kUnroll) {
    int v[kUnroll];
#pragma unroll
    for (int x = 0; x < kUnroll; ++x) {
      const int i = base + x * 32 + lane;
      v[x] = i < k ? __ldg(row + i) : -1;
    }
#pragma unroll
    for (int x = 0; x < kUnroll; ++x)
      if (v[x] >= 0) last = max(last, base + x * 32 + lane);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  return (last + kTile) / kTile;
}

template <int NCH, bool WR, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attend_kernel(const AttnArgs A, const __grid_constant__ CUtensorMap q_map,
                  const __grid_constant__ CUtensorMap qpe_map) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base, formed by pointer arithmetic on the shared array so that accesses stay shared-space
  AttnSmem<NCH>& sm = *reinterpret_cast<AttnSmem<NCH>*>(
      smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u));
  constexpr int kLatChunks = NCH - 1;
  constexpr int kChunkBytes = kTile * 128;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const KernelLayout& L = A.L;
  constexpr int DL = (NCH - 1) * 64;  // latent dims (8 chunks of 64 for 512)
  constexpr int kDTiles = (DL + 127) / 128;
  const int DR = L.d_rope;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tok_full[i], 1);
      mbar_init(&sm.tok_empty[i], 1 + kSoftmaxThreads / 32);
      mbar_init(&sm.kv_full[i], kProducerThreads / 32);  // one arrive per producer warp
      mbar_init(&sm.kv_empty[i], 1);                     // MMA2 of the tile done
      mbar_init(&sm.s_full[i], 1);                       // MMA1 of the tile done
      mbar_init(&sm.s_empty[i], kSoftmaxThreads / 32);   // scores read by every softmax warp
      mbar_init(&sm.p_full[i], kSoftmaxThreads / 32);    // P^T written by every softmax warp
    }
    mbar_init(&sm.q_full, A.q_tma ? 1 : kProducerThreads / 32);  // the copy's arrive, or one per warp
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&sm.tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t tmem_o = tmem;         // O^T: 4 d-tiles x 64 columns
  const uint32_t tmem_s = tmem + 256;   // S^T: two buffers of 64 columns
  volatile int* abort = &sm.abort;

  if (warp >= kFirstProducerWarp) {
    // ------------------------------ producers ------------------------------
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    const int ptid = threadIdx.x - 32 * kFirstProducerWarp;  // 0..351
    uint32_t n = 0, nw = 0, kk = 0;
    uint32_t q_issued = 0;  // query-tile copies issued by this thread (ptid 0 on the copy path)
    constexpr int parts = DL / 16;       // 16-code parts per record
    const bool rope16 = ((DL + 4 * L.n_scales) % 16) == 0;
    // WR: 512 latent codes, four per-128 scales and 64 rope values = 41 aligned 16-byte pieces
    constexpr bool whole_records = WR;
    // A failed wait never makes one warp leave alone: the thread carries on to the next
    // group barrier (what it writes meanwhile is discarded), where the failure is ORed in
    // (bar.red), so that every producer warp leaves the loop together and none is left
    // waiting at a named barrier.
    const int n_splits = MODE == 1 ? A.n_splits : 1;  // compile-time 1 without the split
    int tr, split, ta, tb_nom, slot;
    for (int ui = 0; unit_at<MODE>(A, ui, tr, split, ta, tb_nom, slot); ++ui, ++n) {
      const int t = A.tok_begin + tr;
      const int32_t* idx = A.topk + static_cast<int64_t>(tr) * A.top_k;
      const int row_nt = row_tiles(idx, A.top_k, lane);
      // this unit's tiles: [tb, tb + ntiles) of the row's valid ones
      const int tb = MODE == 1 ? split * row_nt / n_splits : ta;
      const int ntiles = MODE == 1 ? (split + 1) * row_nt / n_splits - tb : max(0, min(tb_nom, row_nt) - ta);
      bool fail = *abort != 0;
      if (warp == kFirstProducerWarp && lane == 0 && !fail) {
        if (mbar_wait(&sm.tok_empty[n & 1], ((n >> 1) & 1) ^ 1, A.err, abort)) {
          sm.ntiles[n & 1] = ntiles;
          if (MODE != 0) sm.tbeg[n & 1] = tb;
          mbar_arrive(&sm.tok_full[n & 1]);
        } else {
          fail = true;
        }
      }
      if (bar_red_or(2, kProducerThreads, fail)) break;
      if (ntiles == 0) continue;
      const int b = seq_of_token(A.qsl, A.batch, t);
      const int32_t* bt = A.block_table + static_cast<int64_t>(b) * A.bt_stride;
      // ---- query -> swizzled bf16 chunks (heads and rope dims zero padded) ----
      const bool q_ok = mbar_wait(&sm.q_empty, (nw & 1) ^ 1, A.err, abort);
      if (A.q_tma) {
        // one thread issues the nine tile copies; their bytes complete q_full
        if (ptid == 0 && q_ok) {
          mbar_arrive_expect_tx(&sm.q_full, NCH * kChunkBytes);
          const int y = t * A.n_heads;
#pragma unroll
          for (int c = 0; c < kLatChunks; ++c) tma_load_2d(smem_u32(sm.q[c]), &q_map, c * 64, y, &sm.q_full);
          tma_load_2d(smem_u32(sm.q[kLatChunks]), &qpe_map, 0, y, &sm.q_full);
          ++q_issued;
        }
      } else {
#pragma unroll 4
      for (int u = ptid; u < kHeads * NCH * 8; u += kProducerThreads) {
        const int h = u / (NCH * 8), rem = u % (NCH * 8), c = rem / 8, v = rem % 8;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (h < A.n_heads) {
          if (c < kLatChunks) {
            val = __ldg(reinterpret_cast<const uint4*>(A.q + (static_cast<int64_t>(t) * A.n_heads + h) * DL + c * 64) + v);
          } else if (v * 8 < DR) {
            const uint16_t* src =
                reinterpret_cast<const uint16_t*>(A.q_pe + (static_cast<int64_t>(t) * A.n_heads + h) * DR) + v * 8;
            val = load_bf16x8_padded(src, DR - v * 8);
          }
        }
        *reinterpret_cast<uint4*>(&sm.q[c][sw128_off(h, v)]) = val;
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.q_full);
      }
      // ---- key tiles ----
      // Unit stream of one tile: units [0, 64*parts) are 16-code latent pieces,
      // units [64*parts, 64*(parts+8)) are 16-byte rope pieces (see latent_unit).
      constexpr int n_lat = kTile * parts;
      constexpr int n_units = n_lat + kTile * 8;
      // Record addresses run two tiles ahead of the gather: during tile t, thread p < 64 reads
      // the top-k entry of key p of tile t+2 (before the gather), its block-table entry (after
      // the first batch), and publishes the record address (at the end).
      const auto rec_of = [&](int j, int blk) -> const uint8_t* {
        if (j < 0) return nullptr;
        if (blk < 0 || blk >= L.num_blocks) {
          latch_error(A.err, SMLA_ERR_BAD_INDEX);
          return nullptr;
        }
        if (A.host_block_map != nullptr) {
          const int hb = __ldg(A.host_block_map + blk);
          if (hb >= 0) {  // the record lives in the host tier (read over the CPU-GPU link)
            if (hb >= A.n_host_blocks) {
              latch_error(A.err, SMLA_ERR_BAD_INDEX);
              return nullptr;
            }
            return A.host_records +
                   ((static_cast<int64_t>(hb) * L.n_layers + A.layer) * L.block_size + j % L.block_size) * L.rec_stride;
          }
        }
        return A.pool + static_cast<int64_t>(blk) * L.block_stride + static_cast<int64_t>(A.layer) * L.layer_stride +
               L.rec_off + static_cast<int64_t>(j % L.block_size) * L.rec_stride;
      };
      const auto entry = [&](int tile) -> int {
        const int e = (tb + tile) * kTile + ptid;
        return (ptid < kTile && tile < ntiles && e < A.top_k) ? __ldg(idx + e) : -1;
      };
      // a position past the sequence's block-table row reads no entry; rec_of latches it as a bad index
      const auto block_of = [&](int j) -> int { return j >= 0 && j < A.max_pos ? __ldg(bt + j / L.block_size) : -1; };
      if (ptid < kTile) {
        const int j0 = entry(0), j1 = entry(1);
        const int b0 = block_of(j0), b1 = block_of(j1);
        sm.rec[0][ptid] = rec_of(j0, b0);
        sm.rec[1][ptid] = rec_of(j1, b1);
      }
      if (bar_red_or(2, kProducerThreads, !q_ok)) break;
      bool failed = false;
      for (int tile = 0; tile < ntiles; ++tile, ++kk) {
        const int kb = kk & 1;
        const uint8_t* const* rec = sm.rec[tile % 3];
        const int j_ahead = entry(tile + 2);
        int blk_ahead = -1;
        bool ok;
        if constexpr (whole_records) {
          // Whole-record gather: producer warp pw takes keys pw, pw + 11, ...; for each key,
          // lane l loads latent piece l (16 codes) and, for l < 9, the piece after the latent
          // codes (lane 0: the four scales; lanes 1-8: the rope), so every record is read by
          // two coalesced warp loads.  Two keys per batch, three batches per tile, two batches in
          // registers: both are requested before the wait for the tile buffer (their latency
          // overlaps the previous tiles' MMAs and softmax instead of following the buffer's
          // release), and a batch register set is refilled with the third batch as soon as it has
          // been stored.
          const int pw = warp - kFirstProducerWarp;
          constexpr int kPW = kProducerThreads / 32;
          constexpr int kR = 2;
          uint4 lat[2][kR], ext[2][kR];
          const auto load_batch = [&](int i0, uint4 (&la)[kR], uint4 (&ex)[kR]) {
#pragma unroll
            for (int i = 0; i < kR; ++i) {
              const int key = pw + kPW * (i0 + i);
              const uint8_t* r = key < kTile ? rec[key] : nullptr;
              la[i] = make_uint4(0, 0, 0, 0);
              ex[i] = make_uint4(0, 0, 0, 0);
              if (r != nullptr) {
                la[i] = __ldg(reinterpret_cast<const uint4*>(r) + lane);
                if (lane < 9) ex[i] = __ldg(reinterpret_cast<const uint4*>(r + DL) + lane);
              }
            }
          };
          const auto store_batch = [&](int i0, const uint4 (&la)[kR], const uint4 (&ex)[kR]) {
#pragma unroll
            for (int i = 0; i < kR; ++i) {
              const int key = pw + kPW * (i0 + i);
              if (key >= kTile) break;
              const float s0 = __shfl_sync(0xffffffffu, __uint_as_float(ex[i].x), 0);
              const float s1 = __shfl_sync(0xffffffffu, __uint_as_float(ex[i].y), 0);
              const float s2 = __shfl_sync(0xffffffffu, __uint_as_float(ex[i].z), 0);
              const float s3 = __shfl_sync(0xffffffffu, __uint_as_float(ex[i].w), 0);
              const int qb = lane >> 3;  // 128-dim scale block of this lane's codes
              const float sc = qb == 0 ? s0 : qb == 1 ? s1 : qb == 2 ? s2 : s3;
              uint4 o0, o1;
              dequant16(la[i], sc, o0, o1);
              // chunk c = lane / 4, 16-byte slots 2 (lane % 4) and + 1; odd chunks store the
              // second slot first so that a quarter-warp's stores hit eight different banks
              const int c = lane >> 2, v0 = 2 * (lane & 3), odd = c & 1;
              *reinterpret_cast<uint4*>(&sm.kv[kb][c][sw128_off(key, v0 + odd)]) = odd ? o1 : o0;
              *reinterpret_cast<uint4*>(&sm.kv[kb][c][sw128_off(key, v0 + 1 - odd)]) = odd ? o0 : o1;
              if (lane >= 1 && lane <= 8)
                *reinterpret_cast<uint4*>(&sm.kv[kb][kLatChunks][sw128_off(key, lane - 1)]) = ex[i];
            }
          };
          constexpr int kNB = ((kTile + kPW - 1) / kPW + kR - 1) / kR;  // batches per tile
          load_batch(0, lat[0], ext[0]);
          if (kNB > 1) load_batch(kR, lat[1], ext[1]);
          ok = mbar_wait(&sm.kv_empty[kb], ((kk >> 1) & 1) ^ 1, A.err, abort);
#pragma unroll
          for (int bi = 0; bi < kNB; ++bi) {
            if (bi == 0) blk_ahead = block_of(j_ahead);
            store_batch(bi * kR, lat[bi & 1], ext[bi & 1]);
            if (bi + 2 < kNB) load_batch((bi + 2) * kR, lat[bi & 1], ext[bi & 1]);
          }
        } else {
        // first batch of loads is issued before waiting for the tile buffer
        uint4 cur[kBatch];
        float csc[kBatch];
        load_units(rec, ptid, n_lat, n_units, parts, DL, DR, L.quant_tile, L.n_scales, rope16, cur, csc);
        ok = mbar_wait(&sm.kv_empty[kb], ((kk >> 1) & 1) ^ 1, A.err, abort);
        for (int base = 0; base < n_units; base += kBatch * kProducerThreads) {
          uint4 nxt[kBatch];
          float nsc[kBatch];
          const int nbase = base + kBatch * kProducerThreads;
          if (nbase < n_units)
            load_units(rec, nbase + ptid, n_lat, n_units, parts, DL, DR, L.quant_tile, L.n_scales, rope16, nxt, nsc);
          if (base == 0) blk_ahead = block_of(j_ahead);
#pragma unroll
          for (int bb = 0; bb < kBatch; ++bb) {
            const int u = base + ptid + bb * kProducerThreads;
            if (u >= n_units) break;
            if (u < n_lat) {
              int r, part;
              latent_unit(u, parts, r, part);
              uint4 o0, o1;
              dequant16(cur[bb], csc[bb], o0, o1);
              const int d0 = part * 16;
              const int c = d0 / 64, v0 = (d0 % 64) / 8;
              *reinterpret_cast<uint4*>(&sm.kv[kb][c][sw128_off(r, v0)]) = o0;
              *reinterpret_cast<uint4*>(&sm.kv[kb][c][sw128_off(r, v0 + 1)]) = o1;
            } else {
              int r, v;
              rope_unit(u - n_lat, r, v);
              *reinterpret_cast<uint4*>(&sm.kv[kb][kLatChunks][sw128_off(r, v)]) = cur[bb];
            }
          }
#pragma unroll
          for (int bb = 0; bb < kBatch; ++bb) {
            cur[bb] = nxt[bb];
            csc[bb] = nsc[bb];
          }
        }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.kv_full[kb]);
        // tile t+2's addresses after the hand-off: the block-table load must not delay the MMA
        if (ptid < kTile) sm.rec[(tile + 2) % 3][ptid] = rec_of(j_ahead, blk_ahead);
        // tile t+2's addresses complete; this tile's reads done; any failed wait ends the row
        if (bar_red_or(2, kProducerThreads, !ok)) {
          failed = true;
          break;
        }
      }
      if (failed) break;
      ++nw;
    }
    // Leave only after the last query-tile copy has landed (it has, unless a wait gave up).
    if (q_issued > 0) mbar_drain(&sm.q_full, (q_issued - 1) & 1);
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ------------------------------
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (lane == 0) {
      uint32_t n = 0, nw = 0, kk = 0;
      bool issued = false;
      const uint32_t idesc1 = make_idesc(kTile, kHeads, 1, 1, 0, 0);  // bf16, both K-major, M = 64 keys
      const uint32_t idesc2 = make_idesc(128, kHeads, 1, 1, 1, 1);    // bf16, both MN-major, M = 128 dims
      // Shared-memory descriptors are built once: an operand address that moves by `off`
      // bytes moves the descriptor's start-address field (bits 0-13, address / 16) by off / 16,
      // which stays inside the field for every shared-memory address.
      const uint64_t dq = sw128_desc(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t dk10 = sw128_desc(smem_u32(sm.kv[0][0]), 16, 1024);
      const uint64_t dk11 = sw128_desc(smem_u32(sm.kv[1][0]), 16, 1024);
      const uint64_t dv20 = sw128_desc(smem_u32(sm.kv[0][0]), kChunkBytes, 1024);
      const uint64_t dv21 = sw128_desc(smem_u32(sm.kv[1][0]), kChunkBytes, 1024);
      const uint64_t dp20 = sw128_desc(smem_u32(sm.kv[0][kLatChunks]), kChunkBytes, 1024);
      const uint64_t dp21 = sw128_desc(smem_u32(sm.kv[1][kLatChunks]), kChunkBytes, 1024);
      // MMA2 of global tile k2: O^T += V^T . P^T over the tile's 64 keys.
      const auto mma2 = [&](uint32_t k2, bool first) {
        const int b2 = k2 & 1;
        const uint64_t va = b2 ? dv21 : dv20, pb = b2 ? dp21 : dp20;
#pragma unroll
        for (int d2 = 0; d2 < kDTiles; ++d2) {
#pragma unroll
          for (int k16 = 0; k16 < kTile / 16; ++k16) {
            mma_f16(tmem_o + d2 * kHeads, va + ((2 * d2 * kChunkBytes + k16 * 2048) >> 4), pb + ((k16 * 2048) >> 4),
                    idesc2, !(first && k16 == 0));
          }
        }
        mma_commit(&sm.kv_empty[b2]);
      };
      // MMA1 of global tile k1: S^T = Khat . q^T over 576 dims into S buffer k1 % 2.  Every three
      // 64-dim chunks it calls between(): the previous tile's MMA2 is issued there as soon as its
      // probabilities are written, instead of after all 36 MMA1 instructions, so that tile's
      // buffer goes back to the producers sooner.  (The tensor pipe runs the instructions in
      // issue order; each commit covers everything issued before it.)
      const auto mma1 = [&](uint32_t k1, auto&& between) {
        const int b1 = k1 & 1;
        const uint64_t ka = b1 ? dk11 : dk10;
        const uint32_t ts = tmem_s + b1 * kHeads;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            mma_f16(ts, ka + ((c * kChunkBytes + k4 * 32) >> 4), dq + ((c * kHeads * 128 + k4 * 32) >> 4), idesc1,
                    (c | k4) != 0);
          }
          if (c % 3 == 2 && c + 1 < NCH) between();
        }
        mma_commit(&sm.s_full[b1]);
      };
      int tr, split, ta, tb_nom, slot;
      for (int ui = 0; !*abort && unit_at<MODE>(A, ui, tr, split, ta, tb_nom, slot); ++ui, ++n) {
        if (!mbar_wait(&sm.tok_full[n & 1], (n >> 1) & 1, A.err, abort)) break;
        const int ntiles = sm.ntiles[n & 1];
        mbar_arrive(&sm.tok_empty[n & 1]);
        if (ntiles == 0) continue;
        if (!mbar_wait(&sm.q_full, nw & 1, A.err, abort)) break;
        // Issue whichever is ready: MMA2 of the oldest tile whose probabilities are written
        // (it releases that tile buffer to the producers), else MMA1 of the next gathered tile
        // (so the next scores are computed while the softmax works).
        const uint32_t kbeg = kk, kend = kk + ntiles;
        uint32_t k1 = kbeg, k2 = kbeg;
        uint64_t t_last = globaltimer_ns();
        bool ok = true;
        // during MMA1 of tile k1 the only MMA2 that can be pending is tile k1 - 1's
        const auto mma2_if_ready = [&]() {
          if (k2 < k1 && mbar_test(&sm.p_full[k2 & 1], (k2 >> 1) & 1)) {
            tc_fence_after();
            mma2(k2, k2 == kbeg);
            ++k2;
          }
        };
        while (k2 < kend) {
          bool progress = false;
          if (k2 < k1 && mbar_test(&sm.p_full[k2 & 1], (k2 >> 1) & 1)) {
            tc_fence_after();
            mma2(k2, k2 == kbeg);
            ++k2;
            progress = true;
          } else if (k1 < kend && mbar_test(&sm.kv_full[k1 & 1], (k1 >> 1) & 1) &&
                     mbar_test(&sm.s_empty[k1 & 1], ((k1 >> 1) & 1) ^ 1)) {
            tc_fence_after();
            mma1(k1, mma2_if_ready);
            issued = true;
            if (k1 == kend - 1) mma_commit(&sm.q_empty);
            ++k1;
            progress = true;
          }
          if (progress) {
            t_last = globaltimer_ns();
          } else {
            if (*abort) {
              ok = false;
              break;
            }
            if (globaltimer_ns() - t_last > kWaitLimitNs) {
              latch_error(A.err, SMLA_ERR_TIMEOUT);
              *abort = 1;
              ok = false;
              break;
            }
            __nanosleep(20);
          }
        }
        kk = kend;
        if (!ok) break;
        mma_commit(&sm.o_done);
        ++nw;
      }
      if (issued) {
        mma_commit(&sm.final_bar);
        mbar_drain(&sm.final_bar, 0);
      }
    }
  } else {
    // ------------------------------ softmax + epilogue (warps 0-7) ------------------------------
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    const int tid = threadIdx.x;            // 0..255
    const int sp = warp & 3;                // TMEM sub-partition
    const int hh = warp >> 2;               // head half: heads 32 hh .. 32 hh + 31
    const int key = 16 * sp + (lane & 15);  // key of the tile (S^T rows sit in TMEM lanes 0-15 of a sub-partition)
    const int hs = lane >> 4;               // this thread's heads: 32 hh + 16 hs .. + 15
    const uint32_t lane_base = static_cast<uint32_t>(sp * 32) << 16;
    uint32_t n = 0, nw = 0, kk = 0;
    // As in the producers, a failed wait skips nothing: the thread finishes the tile (what it
    // computes is discarded) and the failure is ORed into the next group barrier, so that the
    // eight warps leave together.
    int tr, split, ta, tb_nom, slot;
    for (int ui = 0; unit_at<MODE>(A, ui, tr, split, ta, tb_nom, slot); ++ui, ++n) {
      const int t = A.tok_begin + tr;
      const bool partial = MODE != 0 && slot >= 0;  // unit-uniform
      const bool go = *abort == 0 && mbar_wait(&sm.tok_full[n & 1], (n >> 1) & 1, A.err, abort);
      if (bar_red_or(1, kSoftmaxThreads, !go)) break;
      const int ntiles = sm.ntiles[n & 1];
      const int tb = MODE != 0 ? sm.tbeg[n & 1] : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tok_empty[n & 1]);
      // destination of this unit: the row's output, or its partial slot
      const int64_t prow = slot;
      __nv_bfloat16* out_row = A.out + static_cast<int64_t>(t) * A.n_heads * DL;
      float* part_row = partial ? A.part_out + prow * A.n_heads * DL : nullptr;
      float* lse_row = partial ? A.part_lse + prow * A.n_heads : A.lse + static_cast<int64_t>(t) * A.n_heads;
      if (ntiles == 0) {
        for (int i = tid; i < A.n_heads * DL; i += kSoftmaxThreads) {
          if (partial) part_row[i] = 0.f;
          else out_row[i] = __float2bfloat16(0.f);
        }
        if (tid < A.n_heads) lse_row[tid] = -INFINITY;
        continue;
      }
      const int32_t* idx = A.topk + static_cast<int64_t>(tr) * A.top_k;
      float l_part[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) l_part[h] = 0.f;
      bool ok = true, failed = false;
      for (int tile = 0; tile < ntiles; ++tile, ++kk) {
        const int kb = kk & 1;
        const int e = (tb + tile) * kTile + key;
        const bool valid = e < A.top_k && __ldg(idx + e) >= 0;
        ok = ok && mbar_wait(&sm.s_full[kb], (kk >> 1) & 1, A.err, abort);
        tc_fence_after();
        float sc[16];
        {
          uint32_t r[16];
          tmem_ld16x32bx2_x16<16>(tmem_s + lane_base + kb * kHeads + 32 * hh, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int h = 0; h < 16; ++h) sc[h] = valid ? __uint_as_float(r[h]) * A.scale_log2 : -INFINITY;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_empty[kb]);  // the scores are in registers
        // Does any running max have to move?  A head's max moves only when a score of this tile
        // exceeds it by the threshold, so each thread first tests its own scores against the
        // running maxima; the per-head tile maxima (a reduction across lanes and warps) are only
        // formed when some thread found one, which after the first tile is rare.  A failed wait in
        // any warp (here or in the previous tile's rescale) also takes that branch and ends the
        // token for all warps at its barrier.
        int exceed = tile == 0 || !ok;
        if (!exceed) {
#pragma unroll
          for (int h = 0; h < 16; ++h) exceed |= sc[h] > sm.m_run[32 * hh + 16 * hs + h] + kRescaleThreshold;
        }
        bool moved = false;
        if (bar_red_or(1, kSoftmaxThreads, exceed)) {
          // per-head maximum of this tile over the warp's 16 keys; lane 16 hs + h keeps head 32 hh + 16 hs + h
          {
            float mine = -INFINITY;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
              float m = sc[h];
#pragma unroll
              for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
              mine = (lane & 15) == h ? m : mine;
            }
            sm.red[sp][32 * hh + lane] = mine;
          }
          // this tile's maxima are complete
          if (bar_red_or(1, kSoftmaxThreads, !ok)) {
            failed = true;
            break;
          }
          int need_h = 0;
          if (tid < kHeads) {
            const float mt = fmaxf(fmaxf(sm.red[0][tid], sm.red[1][tid]), fmaxf(sm.red[2][tid], sm.red[3][tid]));
            sm.m_tile[tid] = mt;
            need_h = tile == 0 || mt > sm.m_run[tid] + kRescaleThreshold;
          }
          // one barrier that also ORs the per-head "running max must move" flags
          moved = bar_red_or(1, kSoftmaxThreads, need_h) != 0;
        }
        if (moved) {
          if (tid < kHeads) {
            const float old = tile == 0 ? -INFINITY : sm.m_run[tid];
            const float mn = fmaxf(old, sm.m_tile[tid]);
            sm.alpha[tid] = (tile == 0 || mn == -INFINITY) ? 1.f : exp2f(old - mn);
            sm.m_run[tid] = mn;
          }
          named_bar_sync(1, kSoftmaxThreads);
          if (tile > 0) {
#pragma unroll
            for (int h = 0; h < 16; ++h) l_part[h] *= sm.alpha[32 * hh + 16 * hs + h];
          }
        }
        // probabilities -> bf16 P^T row (this key, this warp's 32 heads) in the rope chunk
        {
          uint32_t pw[8];
#pragma unroll
          for (int hx = 0; hx < 16; hx += 2) {
            const int h = 32 * hh + 16 * hs + hx;
            const float m0 = sm.m_run[h], m1 = sm.m_run[h + 1];
            const float p0 = fast_exp2(sc[hx] - (m0 == -INFINITY ? 0.f : m0));
            const float p1 = fast_exp2(sc[hx + 1] - (m1 == -INFINITY ? 0.f : m1));
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            const float2 pf = __bfloat1622float2(pb);
            l_part[hx] += pf.x;
            l_part[hx + 1] += pf.y;
            pw[hx / 2] = (static_cast<uint32_t>(__bfloat16_as_ushort(pb.y)) << 16) | __bfloat16_as_ushort(pb.x);
          }
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            *reinterpret_cast<uint4*>(&sm.kv[kb][kLatChunks][sw128_off(key, 4 * hh + 2 * hs + v)]) =
                make_uint4(pw[4 * v], pw[4 * v + 1], pw[4 * v + 2], pw[4 * v + 3]);
          }
        }
        // rescale O^T when a running max moved; it holds MMA2 of the previous tile once that
        // tile's buffer was released, and MMA2 of this tile waits for p_full below
        if (moved && tile > 0) {
          const uint32_t kp = kk - 1;
          ok = mbar_wait(&sm.kv_empty[kp & 1], (kp >> 1) & 1, A.err, abort) && ok;
          tc_fence_after();
#pragma unroll 1
          for (int d2 = 0; d2 < kDTiles; ++d2) {
            uint32_t o[32];
            tmem_ld32(tmem_o + lane_base + d2 * kHeads + 32 * hh, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * sm.alpha[32 * hh + x]);
            tmem_st32(tmem_o + lane_base + d2 * kHeads + 32 * hh, o);
          }
          tmem_st_wait();
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[kb]);
      }
      if (failed) break;
      // ---- end of token: row sums, normalisation, lse ----
      ok = ok && mbar_wait(&sm.o_done, nw & 1, A.err, abort);
      tc_fence_after();
      half_transpose_sum16(l_part, lane);
      sm.red[sp][32 * hh + lane] = l_part[0];
      if (bar_red_or(1, kSoftmaxThreads, !ok)) break;
      if (tid < kHeads) {
        const float l = (sm.red[0][tid] + sm.red[1][tid]) + (sm.red[2][tid] + sm.red[3][tid]);
        sm.l_fin[tid] = 1.f / l;  // normalisation as one reciprocal per head
        if (tid < A.n_heads) lse_row[tid] = (sm.m_run[tid] + log2f(l)) * kLn2;
      }
      named_bar_sync(1, kSoftmaxThreads);
#pragma unroll 1
      for (int d2 = 0; d2 < kDTiles; ++d2) {
        const int d = d2 * 128 + sp * 32 + lane;
        uint32_t o[32];
        tmem_ld32(tmem_o + lane_base + d2 * kHeads + 32 * hh, o);
        tmem_ld_wait(o);
        if (d < DL && !partial) {
          // Lane l holds dim d for 32 heads.  Four heads at a time, a 4x4 transpose within each
          // group of four lanes gives lane 4g + i head i's four consecutive dims of the group, which
          // go out as one 8-byte store (instead of four 2-byte ones).  d < DL is warp-uniform.
          const int i4 = lane & 3;
          const int dg = d - i4;  // first dim of this lane's group
#pragma unroll
          for (int x0 = 0; x0 < 32; x0 += 4) {
            float a[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) a[jj] = __uint_as_float(o[x0 + jj]) * sm.l_fin[32 * hh + x0 + jj];
#pragma unroll
            for (int st = 2; st >= 1; st >>= 1) {
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                if ((jj & st) == 0) {
                  const bool hi = (i4 & st) != 0;
                  const float recv = __shfl_xor_sync(0xffffffffu, hi ? a[jj] : a[jj | st], st);
                  if (hi) a[jj] = recv;
                  else a[jj | st] = recv;
                }
              }
            }
            // a[jj] = head (x0 + i4) at dim dg + jj
            const int h = 32 * hh + x0 + i4;
            if (h < A.n_heads)
              *reinterpret_cast<uint2*>(out_row + h * DL + dg) = make_uint2(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]));
          }
        } else if (d < DL) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int h = 32 * hh + x;
            if (h < A.n_heads) part_row[h * DL + d] = __uint_as_float(o[x]) * sm.l_fin[h];
          }
        }
      }
      tc_fence_before();
      named_bar_sync(1, kSoftmaxThreads);  // l_fin / m_run reused by the next token
      ++nw;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of a split row's partials: lse = ln sum_s exp(lse_s), out = sum_s exp(lse_s - lse) out_s
// (fp32, then bf16).  One warp per (token, head); 4 dims per lane per step.
__global__ void split_merge_kernel(const float* __restrict__ parts, const float* __restrict__ parts_lse,
                                   int n_splits, int64_t rows, int d, __nv_bfloat16* __restrict__ out,
                                   float* __restrict__ lse) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, __ldg(parts_lse + s * rows + row));
  float z = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const float l = __ldg(parts_lse + s * rows + row);
    z += (mx == -INFINITY || l == -INFINITY) ? 0.f : expf(l - mx);
  }
  const float inv_z = z > 0.f ? 1.f / z : 0.f;
  for (int d0 = 4 * lane; d0 < d; d0 += 4 * 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_splits; ++s) {
      const float l = __ldg(parts_lse + s * rows + row);
      if (mx == -INFINITY || l == -INFINITY) continue;
      const float w = expf(l - mx) * inv_z;
      const float4 v = __ldg(reinterpret_cast<const float4*>(parts + (s * rows + row) * d + d0));
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    *reinterpret_cast<uint2*>(out + row * d + d0) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
  if (lane == 0) lse[row] = z > 0.f ? mx + logf(z) : -INFINITY;
}

// Merge of the rows that balanced units split between neighbouring CTAs: the range of CTA cb
// (cb = 1 .. G - 1) starts at nominal tile g; if g falls inside row r, that row's first part is
// slot 2 cb - 1 (CTA cb - 1's last unit) and its second part slot 2 cb (CTA cb's first unit).
// lse = ln(e^lse_a + e^lse_b), out = e^(lse_a - lse) out_a + e^(lse_b - lse) out_b, in fp32.
// One block per (boundary, 8 heads), one warp per head; every load of a warp is issued before
// the first is used (the merge is latency-bound otherwise).
template <int D>
__global__ void __launch_bounds__(256) balanced_merge_kernel(const float* __restrict__ parts,
                                                              const float* __restrict__ parts_lse, int G, int n_rows,
                                                              int T, int n_heads, __nv_bfloat16* __restrict__ out,
                                                              float* __restrict__ lse) {
  const int cb = static_cast<int>(blockIdx.x) + 1;
  const int64_t tot = static_cast<int64_t>(n_rows) * T;
  const int64_t g = cb * tot / G;
  if (g % T == 0) return;  // the boundary falls between rows: nothing to merge
  const int64_t r = g / T;
  const int lane = threadIdx.x & 31;
  const int h = static_cast<int>(blockIdx.y) * 8 + (threadIdx.x >> 5);
  if (h >= n_heads) return;
  const int64_t sa = 2 * cb - 1, sb = 2 * cb;
  constexpr int kIt = (D + 127) / 128;  // float4 steps per lane
  const float* pa = parts + (sa * n_heads + h) * D;
  const float* pb = parts + (sb * n_heads + h) * D;
  float4 a[kIt], b[kIt];
#pragma unroll
  for (int i = 0; i < kIt; ++i) {
    const int d0 = 4 * lane + 128 * i;
    a[i] = d0 < D ? __ldg(reinterpret_cast<const float4*>(pa + d0)) : make_float4(0.f, 0.f, 0.f, 0.f);
    b[i] = d0 < D ? __ldg(reinterpret_cast<const float4*>(pb + d0)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float la = __ldg(parts_lse + sa * n_heads + h), lb = __ldg(parts_lse + sb * n_heads + h);
  const float mx = fmaxf(la, lb);
  const float wa = (mx == -INFINITY || la == -INFINITY) ? 0.f : expf(la - mx);
  const float wb = (mx == -INFINITY || lb == -INFINITY) ? 0.f : expf(lb - mx);
  const float z = wa + wb;
  const float inv_z = z > 0.f ? 1.f / z : 0.f;
  const float ca = wa * inv_z, cbw = wb * inv_z;
  __nv_bfloat16* o = out + (r * n_heads + h) * D;
#pragma unroll
  for (int i = 0; i < kIt; ++i) {
    const int d0 = 4 * lane + 128 * i;
    if (d0 < D)
      *reinterpret_cast<uint2*>(o + d0) =
          make_uint2(pack_bf16x2(ca * a[i].x + cbw * b[i].x, ca * a[i].y + cbw * b[i].y),
                     pack_bf16x2(ca * a[i].z + cbw * b[i].z, ca * a[i].w + cbw * b[i].w));
  }
  if (lane == 0) lse[r * n_heads + h] = z > 0.f ? mx + logf(z) : -INFINITY;
}

template <int NCH, bool WR>
smla_status_t launch_nch(AttnArgs A, cudaStream_t stream) {
  const size_t smem = sizeof(AttnSmem<NCH>) + 1024;
  static std::atomic<bool> attr_set[kMaxDeviceSlots] = {};
  const int dev = current_device_index();
  if (dev < 0) return SMLA_ERR_CUDA;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(attend_kernel<NCH, WR, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(attend_kernel<NCH, WR, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(attend_kernel<NCH, WR, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return SMLA_ERR_CUDA;
    // setmaxnreg.inc can only draw on the registers the CTA was launched with;
    // refuse to launch if the compiled allocation does not cover the split.
    cudaFuncAttributes fa, fs, fb;
    if (cudaFuncGetAttributes(&fa, attend_kernel<NCH, WR, 0>) != cudaSuccess ||
        cudaFuncGetAttributes(&fs, attend_kernel<NCH, WR, 1>) != cudaSuccess ||
        cudaFuncGetAttributes(&fb, attend_kernel<NCH, WR, 2>) != cudaSuccess)
      return SMLA_ERR_CUDA;
    if (fa.numRegs < kLaunchRegs || fs.numRegs < kLaunchRegs || fb.numRegs < kLaunchRegs) return SMLA_ERR_UNSUPPORTED;
    attr_set[dev].store(true, std::memory_order_release);
  }
  // Query tiles by tensor-map copies when they match the shared-memory tile exactly: 64 heads,
  // 64-dim chunks (the latent in NCH - 1 of them, the rope in one), 16-byte aligned rows.
  CUtensorMap q_map, qpe_map;
  std::memset(&q_map, 0, sizeof(q_map));
  std::memset(&qpe_map, 0, sizeof(qpe_map));
  A.q_tma = 0;
  constexpr int DL = (NCH - 1) * 64;
  if (A.n_heads == kHeads && A.L.d_rope == 64 && (reinterpret_cast<uintptr_t>(A.q) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(A.q_pe) & 15) == 0) {
    EncodeTiledFn enc = encode_tiled();
    const cuuint64_t rows = static_cast<cuuint64_t>(A.tok_begin + A.n_rows) * A.n_heads;
    const cuuint64_t q_dims[2] = {static_cast<cuuint64_t>(DL), rows};
    const cuuint64_t q_strides[1] = {static_cast<cuuint64_t>(DL) * 2};
    const cuuint64_t pe_dims[2] = {64, rows};
    const cuuint64_t pe_strides[1] = {128};
    const cuuint32_t box[2] = {64, kHeads};
    const cuuint32_t estr[2] = {1, 1};
    if (enc != nullptr &&
        enc(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(A.q), q_dims, q_strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
        enc(&qpe_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(A.q_pe), pe_dims, pe_strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      A.q_tma = 1;
  }
  const int sms = device_sm_count();
  const int grid = A.mode == 2 ? sms : min(A.n_rows * A.n_splits, sms);
  if (A.mode == 1)
    attend_kernel<NCH, WR, 1><<<grid, kThreads, smem, stream>>>(A, q_map, qpe_map);
  else if (A.mode == 2)
    attend_kernel<NCH, WR, 2><<<grid, kThreads, smem, stream>>>(A, q_map, qpe_map);
  else
    attend_kernel<NCH, WR, 0><<<grid, kThreads, smem, stream>>>(A, q_map, qpe_map);
  if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
  if (A.mode == 2) {
    balanced_merge_kernel<(NCH - 1) * 64><<<dim3(grid - 1, (A.n_heads + 7) / 8), 256, 0, stream>>>(
        A.part_out, A.part_lse, grid, A.n_rows, A.row_tiles_nom, A.n_heads,
        A.out + static_cast<int64_t>(A.tok_begin) * A.n_heads * (NCH - 1) * 64,
        A.lse + static_cast<int64_t>(A.tok_begin) * A.n_heads);
    if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
  }
  if (A.mode == 1) {
    const int64_t rows = static_cast<int64_t>(A.n_rows) * A.n_heads;
    constexpr int kMergeWarps = 8;
    split_merge_kernel<<<static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps), 32 * kMergeWarps, 0, stream>>>(
        A.part_out, A.part_lse, A.n_splits, rows, (NCH - 1) * 64,
        A.out + static_cast<int64_t>(A.tok_begin) * A.n_heads * (NCH - 1) * 64,
        A.lse + static_cast<int64_t>(A.tok_begin) * A.n_heads);
    if (cudaGetLastError() != cudaSuccess) return SMLA_ERR_CUDA;
  }
  return SMLA_OK;
}

}  // namespace

// Up to 64 heads, rope of at most 64 dims, a latent of 64 or 512 dims.
bool attend_shape_supported(const KernelLayout& L, int n_heads) {
  return n_heads > 0 && n_heads <= kHeads && L.d_rope <= 64 && (L.d_latent == 64 || L.d_latent == 512);
}

smla_status_t launch_attend(const KernelLayout& L, int n_heads, int top_k, float softmax_scale, const void* pool,
                            int layer, const void* q, const void* q_pe, const int32_t* topk_idx,
                            const int32_t* block_table, int bt_stride, const int32_t* query_start_loc, int batch,
                            int tok_begin, int tok_end, void* out, float* lse, cudaStream_t stream, unsigned* err,
                            const void* host_records, const int32_t* host_block_map, int64_t n_host_blocks,
                            void* split_ws, size_t split_ws_bytes) {
  if (tok_end <= tok_begin) return SMLA_OK;
  if (!attend_shape_supported(L, n_heads)) return SMLA_ERR_UNSUPPORTED;
  // Fewer rows than SMs: each row's tiles are split over up to sms / rows CTAs (one wave of
  // units), as far as the caller's scratch holds the partials.
  const int n_rows = tok_end - tok_begin;
  const int sms = device_sm_count();
  const int row_tiles_max = (top_k + kTile - 1) / kTile;
  int n_splits = 1;
  if (split_ws != nullptr && n_rows < sms && row_tiles_max > 1) {
    n_splits = min(sms / n_rows, row_tiles_max);
    while (n_splits > 1 && attend_split_bytes(n_heads, L.d_latent, n_rows * n_splits) > split_ws_bytes) --n_splits;
  }
  // More rows than SMs, with a last round of rows that would leave most SMs idle (at most half of
  // them busy): every CTA takes the same number of tiles instead (balanced units), and rows that
  // straddle two CTAs are merged by their lse.  With a fuller last round the one-row-per-CTA
  // schedule is kept: the gathers of all SMs together are bound by the memory system, so a CTA's
  // tiles run faster while fewer SMs are busy (measured: 256 rows on 152 SMs, 0.243 ms plain
  // against 0.262 ms balanced).
  const int rem = n_rows % sms;
  const bool balanced = split_ws != nullptr && n_rows > sms && n_rows < 8 * sms && rem != 0 && rem <= sms / 2 &&
                        row_tiles_max > 1 && attend_split_bytes(n_heads, L.d_latent, 2 * sms) <= split_ws_bytes;
  const int parts = n_splits > 1 ? n_rows * n_splits : (balanced ? 2 * sms : 0);
  AttnArgs A;
  A.L = L;
  A.n_heads = n_heads;
  A.top_k = top_k;
  A.layer = layer;
  A.scale_log2 = softmax_scale * kLog2e;
  A.pool = static_cast<const uint8_t*>(pool);
  A.q = static_cast<const __nv_bfloat16*>(q);
  A.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
  A.topk = topk_idx;
  A.block_table = block_table;
  A.bt_stride = bt_stride;
  A.max_pos = static_cast<int64_t>(bt_stride) * L.block_size;
  A.qsl = query_start_loc;
  A.batch = batch;
  A.tok_begin = tok_begin;
  A.n_rows = tok_end - tok_begin;
  A.out = static_cast<__nv_bfloat16*>(out);
  A.lse = lse;
  A.err = err;
  A.host_records = static_cast<const uint8_t*>(host_records);
  A.host_block_map = host_block_map;
  A.n_host_blocks = n_host_blocks;
  A.n_splits = n_splits;
  A.mode = n_splits > 1 ? 1 : (balanced ? 2 : 0);
  A.row_tiles_nom = row_tiles_max;
  A.part_out = parts > 0 ? static_cast<float*>(split_ws) : nullptr;
  A.part_lse = parts > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(split_ws) +
                                                    split_out_bytes(n_heads, L.d_latent, parts))
                         : nullptr;
  switch (L.d_latent / 64) {
    case 1: return launch_nch<2, false>(A, stream);
    case 8: {
      // records of 512 codes, four per-128 scales and 64 rope values take the whole-record gather
      const bool wr = L.n_scales == 4 && L.quant_tile == 128 && L.d_rope == 64 && (512 + 4 * L.n_scales) % 16 == 0;
      return wr ? launch_nch<9, true>(A, stream) : launch_nch<9, false>(A, stream);
    }
    default: return SMLA_ERR_UNSUPPORTED;
  }
}

}  // namespace smla
