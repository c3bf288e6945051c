// smla_decode_static: the fused step for callers that cannot allocate device memory.
//
// smla_decode needs a caller-provided workspace for the fp32 indexer scores and
// the top-k indices.  Some callers have no way to provide one: their device
// memory is owned by a serving engine's allocator (for example one that reserves
// all free HBM for the KV block pool at start-up and hands out no other
// buffers), or they are written against a host runtime that exposes no device
// allocation hook at all.  This entry point serves them with a fixed scratch
// array that lives in the library's own module memory.
//
// The scratch is a file-scope static __device__ array of kStaticScratchBytes
// (64 MiB).  Every GPU that loads the library holds it until the process exits.
// Host code must not pass the array's name to a kernel (on the host it is only
// a stand-in symbol); its device address is taken once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device.  Make that first call before any stream capture begins.
//
// Every call shares the one array and leaves its contents behind.  Nothing in it
// has to start at zero: each query group's score rows are written by the indexer
// for every position the top-k reads, and every top-k row is written in full.
// Calls whose kernels overlap on the GPU (different streams without ordering
// between them) race on the array; order them on one stream.
#include <atomic>

#include "smla_internal.h"

namespace smla {
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr int kMaxDevicesStatic = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of the array per device (nullptr until the first call there).  Racing
// first calls from several host threads all look up the same address; the atomic store
// publishes it to the others.
std::atomic<uint8_t*> g_static_scratch_addr[kMaxDevicesStatic] = {};

inline int64_t round_up_static(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Device address of the static scratch on the current device (set up once).
smla_status_t static_scratch(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesStatic) return SMLA_ERR_CUDA;
  uint8_t* addr = g_static_scratch_addr[dev].load(std::memory_order_acquire);
  if (addr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return SMLA_ERR_CUDA;
    addr = static_cast<uint8_t*>(p);
    g_static_scratch_addr[dev].store(addr, std::memory_order_release);
  }
  *out = addr;
  return SMLA_OK;
}

}  // namespace
}  // namespace smla

using namespace smla;

extern "C" smla_status_t smla_decode_static(const smla_layout_t* layout, const smla_params_t* params, void* pool,
                                            int layer, const void* new_latent, const void* new_rope,
                                            const uint8_t* new_idx_k, const float* new_idx_scale,
                                            const int64_t* slot_mapping, const void* q, const void* q_pe,
                                            const uint8_t* q_idx, const float* w, const int32_t* block_table,
                                            int bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                                            int batch, int n_tokens, int max_q, int max_ctx, void* out, float* lse,
                                            int32_t* topk_idx_out, void* stream) {
  // the same argument checks, in the same order, as smla_decode
  const StepArgs args{layout,   params,     pool,    layer,   new_latent, new_rope,  new_idx_k,       new_idx_scale,
                      slot_mapping, q,      q_pe,    q_idx,   w,          block_table, bt_stride,     seq_lens,
                      query_start_loc, batch, n_tokens, max_q, max_ctx,   out,       lse};
  smla_status_t st = check_step(args);
  if (st != SMLA_OK || n_tokens == 0) return st;
  // Query tokens go in groups whose scores and indices fit the static scratch.
  const int64_t stride = round_up_static(max_ctx, 4);
  const int64_t per_token = stride * 4 + static_cast<int64_t>(params->top_k) * 4;
  int64_t g = static_cast<int64_t>(kStaticScratchBytes - 512) / per_token;
  if (g < 1) return SMLA_ERR_SCRATCH_LIMIT;  // one token's score row and indices exceed the scratch
  unsigned* err = nullptr;
  st = checked_device(&err);  // sm_103 device (as smla_decode), and its error word
  if (st != SMLA_OK) return st;
  g = wave_aligned_group(g, n_tokens);
  uint8_t* scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != SMLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const KernelLayout L = kernel_layout(*layout);
  if (slot_mapping != nullptr) {
    st = launch_kvpack_store(L, pool, layer, new_latent, new_rope, new_idx_k, new_idx_scale, slot_mapping, n_tokens, s,
                             err);
    if (st != SMLA_OK) return st;
  }
  float* scores = reinterpret_cast<float*>(scratch);
  int32_t* topk_ws = reinterpret_cast<int32_t*>(scratch + round_up_static(g * stride * 4, 256));
  // what the group leaves of the scratch holds the split-attention partials
  const int64_t used = round_up_static(g * stride * 4, 256) + round_up_static(g * params->top_k * 4, 256);
  const size_t split_bytes = static_cast<size_t>(kStaticScratchBytes) > static_cast<size_t>(used)
                                 ? static_cast<size_t>(kStaticScratchBytes) - static_cast<size_t>(used)
                                 : 0;
  void* split_ws = split_bytes > 0 ? scratch + used : nullptr;
  for (int t0 = 0; t0 < n_tokens; t0 += static_cast<int>(g)) {
    const int t1 = t0 + static_cast<int>(g) < n_tokens ? t0 + static_cast<int>(g) : n_tokens;
    int32_t* topk = topk_idx_out ? topk_idx_out + static_cast<int64_t>(t0) * params->top_k : topk_ws;
    st = launch_index_scores(L, params->n_idx_heads, pool, layer, q_idx, w, block_table, bt_stride, seq_lens,
                             query_start_loc, batch, t0, t1, max_q, max_ctx, scores, stride, s, err);
    if (st != SMLA_OK) return st;
    st = launch_topk(params->top_k, scores, stride, seq_lens, query_start_loc, batch, t0, t1, topk, s, err, split_ws,
                     split_bytes);
    if (st != SMLA_OK) return st;
    st = launch_attend(L, params->n_heads, params->top_k, params->softmax_scale, pool, layer, q, q_pe, topk,
                       block_table, bt_stride, query_start_loc, batch, t0, t1, out, lse, s, err, nullptr, nullptr, 0,
                       split_ws, split_bytes);
    if (st != SMLA_OK) return st;
  }
  return SMLA_OK;
}
