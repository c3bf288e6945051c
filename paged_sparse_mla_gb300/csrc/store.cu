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
                                                           unsigned* err) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n_tokens) return;
  const int64_t slot = slot_mapping[warp];
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
  float x[E];
  const __nv_bfloat16* src = latent + static_cast<int64_t>(warp) * L.d_latent + lane * E;
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] = __bfloat162float(src[i]);
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
#pragma unroll
  for (int i = 0; i < E; ++i) rec[lane * E + i] = codes[i];
  if ((lane * E) % L.quant_tile == 0) {
    reinterpret_cast<float*>(rec + L.d_latent)[(lane * E) / L.quant_tile] = scale;
  }
  // ---- rope (bf16) verbatim, 2-byte units ----
  const uint16_t* rsrc = reinterpret_cast<const uint16_t*>(rope) + static_cast<int64_t>(warp) * L.d_rope;
  uint16_t* rdst = reinterpret_cast<uint16_t*>(rec + L.d_latent + 4 * L.n_scales);
  for (int i = lane; i < L.d_rope; i += 32) rdst[i] = rsrc[i];
  // ---- indexer key (e4m3 bytes) and its fp32 scale verbatim ----
  const uint8_t* ksrc = idx_k + static_cast<int64_t>(warp) * L.key_bytes;
  uint8_t* kdst = layer_base + L.idx_key_off + static_cast<int64_t>(off) * L.key_bytes;
  for (int i = lane; i < L.key_bytes; i += 32) kdst[i] = ksrc[i];
  if (lane == 0) {
    reinterpret_cast<float*>(layer_base + L.idx_scale_off)[off] = idx_scale[warp];
  }
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
  switch (L.d_latent / 32) {
    case 2:
      kvpack_store_kernel<2><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                             n_tokens, err);
      break;
    case 4:
      kvpack_store_kernel<4><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                             n_tokens, err);
      break;
    case 8:
      kvpack_store_kernel<8><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                             n_tokens, err);
      break;
    case 16:
      kvpack_store_kernel<16><<<blocks, threads, 0, stream>>>(L, pl, layer, lat, rp, idx_k, idx_scale, slot_mapping,
                                                              n_tokens, err);
      break;
    default:
      return SMLA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace smla
