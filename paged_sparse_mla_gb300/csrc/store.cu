// kvpack_store: new tokens -> packed FP8 records of the shared block pool.
//
// [GLM-5.3 "How to try", "Config and numbers"]: the KV cache is FP8.
// [AgentX "Hybrid KV cache management"]: one packed allocation per block
// holds every cache group (latent records, indexer keys, indexer scales).
//
// One warp per token.  Lane l owns latent elements [l*E, l*E+E) (E = d_latent/32);
// a quantisation tile spans quant_tile/E consecutive lanes, whose amax is
// combined with xor-shuffles.  scale = amax / 448 is an IEEE fp32 division
// (the library is built without fast-math), x / scale likewise, and the E4M3
// code is the hardware's round-to-nearest-even saturating conversion.
#include "smla_internal.h"

namespace smla {

template <int E>
__global__ void __launch_bounds__(256) kvpack_store_kernel(KernelLayout L, uint8_t* __restrict__ pool, int layer,
                                                           const __nv_bfloat16* __restrict__ latent,
                                                           const __nv_bfloat16* __restrict__ rope,
                                                           const uint8_t* __restrict__ idx_k,
                                                           const float* __restrict__ idx_scale,
                                                           const int64_t* __restrict__ slot_mapping, int n_tokens,
                                                           bool vec, unsigned* err) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n_tokens) return;
  // The token's inputs do not depend on its slot: their loads are issued together with the slot's.
  // `vec` (set by the launcher) says every source and destination of the 32-bit and 16-byte
  // accesses below is aligned for them.
  const int64_t slot = __ldg(slot_mapping + warp);
  float x[E];
  const __nv_bfloat16* src = latent + static_cast<int64_t>(warp) * L.d_latent + lane * E;
  if constexpr (E % 8 == 0) {
    if (vec) {
#pragma unroll
      for (int v = 0; v < E / 8; ++v) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + v);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          x[8 * v + 2 * q] = __uint_as_float(ws[q] << 16);
          x[8 * v + 2 * q + 1] = __uint_as_float(ws[q] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] = __bfloat162float(src[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = __bfloat162float(src[i]);
  }
  // rope and indexer key as 32-bit words (at most two per lane on the vector path)
  const int rope_words = L.d_rope / 2, key_words = L.key_bytes / 4;
  const bool words = vec && rope_words <= 64 && key_words <= 64;
  uint32_t rw[2] = {0, 0}, kw[2] = {0, 0};
  if (words) {
    const uint32_t* rs = reinterpret_cast<const uint32_t*>(rope) + static_cast<int64_t>(warp) * rope_words;
    const uint32_t* ks = reinterpret_cast<const uint32_t*>(idx_k) + static_cast<int64_t>(warp) * key_words;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (lane + 32 * q < rope_words) rw[q] = __ldg(rs + lane + 32 * q);
      if (lane + 32 * q < key_words) kw[q] = __ldg(ks + lane + 32 * q);
    }
  }
  const float kscale = lane == 0 ? __ldg(idx_scale + warp) : 0.f;
  if (slot < 0) return;
  if (slot >= L.num_blocks * L.block_size) {
    if (lane == 0) latch_error(err, SMLA_ERR_BAD_INDEX);
    return;
  }
  const int64_t blk = slot / L.block_size;
  const int off = static_cast<int>(slot - blk * L.block_size);
  uint8_t* layer_base = pool + blk * L.block_stride + static_cast<int64_t>(layer) * L.layer_stride;
  uint8_t* rec = layer_base + L.rec_off + static_cast<int64_t>(off) * L.rec_stride;

  // ---- latent: per-tile amax, scale, E4M3 codes ----
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const int lanes_per_tile = L.quant_tile / E;  // power of two, <= 32
  for (int m = 1; m < lanes_per_tile; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  float scale = amax / 448.0f;
  if (scale == 0.0f) scale = 1.0f;
  uint8_t codes[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    codes[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(x[i] / scale, __NV_SATFINITE, __NV_E4M3));
  }
  if constexpr (E % 16 == 0) {
    if (vec) {
#pragma unroll
      for (int v = 0; v < E / 16; ++v) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = codes[16 * v + 4 * q] | (codes[16 * v + 4 * q + 1] << 8) | (codes[16 * v + 4 * q + 2] << 16) |
                 (static_cast<uint32_t>(codes[16 * v + 4 * q + 3]) << 24);
        reinterpret_cast<uint4*>(rec + lane * E)[v] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) rec[lane * E + i] = codes[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) rec[lane * E + i] = codes[i];
  }
  if ((lane * E) % L.quant_tile == 0) {
    reinterpret_cast<float*>(rec + L.d_latent)[(lane * E) / L.quant_tile] = scale;
  }
  uint8_t* kdst = layer_base + L.idx_key_off + static_cast<int64_t>(off) * L.key_bytes;
  uint8_t* rdst8 = rec + L.d_latent + 4 * L.n_scales;
  if (words) {
    // ---- rope (bf16) and indexer key (e4m3 or packed e2m1 bytes) verbatim, 32-bit words ----
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (lane + 32 * q < rope_words) reinterpret_cast<uint32_t*>(rdst8)[lane + 32 * q] = rw[q];
      if (lane + 32 * q < key_words) reinterpret_cast<uint32_t*>(kdst)[lane + 32 * q] = kw[q];
    }
  } else {
    // ---- the same in 2-byte and 1-byte units ----
    const uint16_t* rsrc = reinterpret_cast<const uint16_t*>(rope) + static_cast<int64_t>(warp) * L.d_rope;
    uint16_t* rdst = reinterpret_cast<uint16_t*>(rdst8);
    for (int i = lane; i < L.d_rope; i += 32) rdst[i] = rsrc[i];
    const uint8_t* ksrc = idx_k + static_cast<int64_t>(warp) * L.key_bytes;
    for (int i = lane; i < L.key_bytes; i += 32) kdst[i] = ksrc[i];
  }
  if (lane == 0) reinterpret_cast<float*>(layer_base + L.idx_scale_off)[off] = kscale;
}

bool store_shape_supported(const KernelLayout& L) {
  const int e = L.d_latent / 32;  // latent elements per lane
  return L.d_latent % 32 == 0 && (e == 2 || e == 4 || e == 8 || e == 16);
}

smla_status_t launch_kvpack_store(const KernelLayout& L, void* pool, int layer, const void* latent,
                                  const void* rope, const uint8_t* idx_k, const float* idx_scale,
                                  const int64_t* slot_mapping, int n_tokens, cudaStream_t stream, unsigned* err) {
  if (n_tokens == 0) return SMLA_OK;
  if (!store_shape_supported(L)) return SMLA_ERR_UNSUPPORTED;
  const int threads = 256;
  const int blocks = (n_tokens * 32 + threads - 1) / threads;
  auto* pl = static_cast<uint8_t*>(pool);
  auto* lat = static_cast<const __nv_bfloat16*>(latent);
  auto* rp = static_cast<const __nv_bfloat16*>(rope);
  // Vector accesses: 16-byte latent loads and code stores, 32-bit rope and key words.  Every
  // address they touch is a multiple of its width when these bases and strides are.
  const auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  const bool vec = al(pool, 16) && al(latent, 16) && al(rope, 4) && al(idx_k, 4) && L.d_latent % 8 == 0 &&
                   L.block_stride % 16 == 0 && L.layer_stride % 16 == 0 && L.rec_off % 16 == 0 &&
                   L.rec_stride % 16 == 0 && (L.d_latent + 4 * L.n_scales) % 4 == 0 && L.d_rope % 2 == 0 &&
                   L.idx_key_off % 4 == 0 && L.key_bytes % 4 == 0;
  switch (L.d_latent / 32) {
    case 2:
      kvpack_store_kernel<2><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                             n_tokens, vec, err);
      break;
    case 4:
      kvpack_store_kernel<4><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                             n_tokens, vec, err);
      break;
    case 8:
      kvpack_store_kernel<8><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                             n_tokens, vec, err);
      break;
    case 16:
      kvpack_store_kernel<16><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                              n_tokens, vec, err);
      break;
    default:
      return SMLA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
