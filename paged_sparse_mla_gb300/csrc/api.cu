// C ABI of libsmla: argument checks, workspace sizing, the fused step, and the
// latched device error word.  Every entry point is declared in include/smla.h.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "smla_internal.h"

namespace smla {
namespace {

__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
constexpr size_t kScoreBudget = size_t(512) << 20;  // bytes of fp32 scores per query group

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// The exit protocol of the warp-specialised kernels on a barrier that never
// completes: warp 0 waits on bar[0], which no thread arrives at; warps 1-3 wait
// on bar[1], whose first phase thread 32 completes.  The failed wait is made
// warp-uniform and ORed into the group barrier, so that the four warps leave
// together.
__global__ void wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 32) mbar_arrive(&bar[1]);
  const int warp = threadIdx.x >> 5;
  volatile int* abort = &abort_flag;
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar[warp == 0 ? 0 : 1], 0, err, abort, limit_ns));
  bar_red_or(1, 128, !ok);
}

struct DeviceInfo {
  std::atomic<bool> init{false};  // set (release) once the fields below are filled in
  int sms = 0;
  bool supported = false;
  unsigned* err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;  // serialises the one-time set-up of a device's entry

// The calling thread's current device, its attributes and the device address of
// the error word; filled in once per device, safely when host threads race to it.
DeviceInfo* current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& d = g_dev[dev];
  if (d.init.load(std::memory_order_acquire)) return &d;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!d.init.load(std::memory_order_relaxed)) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    d.supported = (major == 10 && minor == 3);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    d.err = static_cast<unsigned*>(p);
    d.init.store(true, std::memory_order_release);
  }
  return &d;
}

smla_status_t check_device(DeviceInfo** out) {
  DeviceInfo* d = current_device();
  if (d == nullptr) return SMLA_ERR_CUDA;
  if (!d->supported) return SMLA_ERR_UNSUPPORTED;
  *out = d;
  return SMLA_OK;
}

// Query tokens per group so the fp32 score scratch stays within kScoreBudget.
int query_group(int n_tokens, int64_t stride) {
  int64_t g = static_cast<int64_t>(kScoreBudget / (static_cast<size_t>(stride) * 4));
  if (g < 1) g = 1;
  if (g > n_tokens) g = n_tokens;
  return static_cast<int>(g);
}

}  // namespace

int current_device_index() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDeviceSlots) return -1;
  return dev;
}

unsigned* device_error_word() {
  DeviceInfo* d = current_device();
  return d ? d->err : nullptr;
}

int device_sm_count() {
  DeviceInfo* d = current_device();
  return d && d->sms > 0 ? d->sms : 1;
}

smla_status_t checked_device(unsigned** err) {
  DeviceInfo* d = nullptr;
  const smla_status_t st = check_device(&d);
  if (st == SMLA_OK) *err = d->err;
  return st;
}

bool layout_ok(const smla_layout_t* l) {
  if (l == nullptr) return false;
  smla_layout_t ref;
  if (smla_layout_init_keys(&ref, l->block_size, l->n_layers, l->d_latent, l->d_rope, l->quant_tile, l->d_index,
                            l->idx_key_format, l->num_blocks) != SMLA_OK)
    return false;
  return l->idx_key_format == ref.idx_key_format && l->n_scales == ref.n_scales && l->rec_bytes == ref.rec_bytes && l->rec_stride == ref.rec_stride &&
         l->rec_off == ref.rec_off && l->idx_key_off == ref.idx_key_off && l->idx_scale_off == ref.idx_scale_off &&
         l->layer_stride == ref.layer_stride && l->block_stride == ref.block_stride;
}

smla_status_t check_step(const StepArgs& a) {
  const smla_layout_t* layout = a.layout;
  const smla_params_t* params = a.params;
  if (!layout_ok(layout) || !params || a.layer < 0 || a.layer >= layout->n_layers || a.batch <= 0 ||
      a.n_tokens < 0 || a.max_q <= 0 || a.max_ctx <= 0 || params->top_k <= 0 || params->n_heads <= 0 ||
      params->n_idx_heads <= 0)
    return SMLA_ERR_INVALID_ARG;
  if (a.n_tokens == 0) return SMLA_OK;
  if (!a.pool || !a.q || (layout->d_rope > 0 && !a.q_pe) || !a.q_idx || !a.w || !a.block_table || !a.seq_lens ||
      !a.query_start_loc || !a.out || !a.lse || a.bt_stride <= 0 ||
      static_cast<int64_t>(a.bt_stride) * layout->block_size < a.max_ctx)
    return SMLA_ERR_INVALID_ARG;
  if (a.slot_mapping != nullptr &&
      (!a.new_latent || !a.new_idx_k || !a.new_idx_scale || (layout->d_rope > 0 && !a.new_rope)))
    return SMLA_ERR_INVALID_ARG;
  const KernelLayout L = kernel_layout(*layout);
  if ((a.slot_mapping != nullptr && !store_shape_supported(L)) || !index_shape_supported(L, params->n_idx_heads) ||
      !attend_shape_supported(L, params->n_heads))
    return SMLA_ERR_UNSUPPORTED;
  return SMLA_OK;
}

}  // namespace smla

using namespace smla;

extern "C" {

int smla_version(void) { return 100; }

const char* smla_status_string(smla_status_t s) {
  switch (s) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_INVALID_ARG: return "SMLA_ERR_INVALID_ARG";
    case SMLA_ERR_UNSUPPORTED: return "SMLA_ERR_UNSUPPORTED";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA";
    case SMLA_ERR_BAD_INDEX: return "SMLA_ERR_BAD_INDEX";
    case SMLA_ERR_TIMEOUT: return "SMLA_ERR_TIMEOUT";
    case SMLA_ERR_SCRATCH_LIMIT: return "SMLA_ERR_SCRATCH_LIMIT";
  }
  return "SMLA_ERR_UNKNOWN";
}

smla_status_t smla_layout_init(smla_layout_t* l, int block_size, int n_layers, int d_latent, int d_rope,
                               int quant_tile, int d_index, int64_t num_blocks) {
  return smla_layout_init_keys(l, block_size, n_layers, d_latent, d_rope, quant_tile, d_index, SMLA_KEY_E4M3,
                               num_blocks);
}

smla_status_t smla_layout_init_keys(smla_layout_t* l, int block_size, int n_layers, int d_latent, int d_rope,
                                    int quant_tile, int d_index, int key_format, int64_t num_blocks) {
  if (l == nullptr || block_size <= 0 || n_layers <= 0 || d_latent <= 0 || d_rope < 0 || quant_tile <= 0 ||
      d_index <= 0 || num_blocks <= 0)
    return SMLA_ERR_INVALID_ARG;
  if (d_latent % quant_tile != 0 || d_latent % 32 != 0 || d_rope % 2 != 0 || d_index % 16 != 0)
    return SMLA_ERR_INVALID_ARG;
  if (key_format != SMLA_KEY_E4M3 && (key_format != SMLA_KEY_E2M1 || d_index % 32 != 0))
    return SMLA_ERR_INVALID_ARG;
  const int e = d_latent / 32;  // latent elements per lane in the store
  if (quant_tile % e != 0 || (quant_tile / e) > 32 || ((quant_tile / e) & (quant_tile / e - 1)) != 0)
    return SMLA_ERR_INVALID_ARG;
  std::memset(l, 0, sizeof(*l));
  l->block_size = block_size;
  l->n_layers = n_layers;
  l->d_latent = d_latent;
  l->d_rope = d_rope;
  l->quant_tile = quant_tile;
  l->d_index = d_index;
  l->idx_key_format = key_format;
  l->num_blocks = num_blocks;
  l->n_scales = d_latent / quant_tile;
  l->rec_bytes = d_latent + 4 * l->n_scales + 2 * d_rope;
  l->rec_stride = static_cast<int32_t>(round_up(l->rec_bytes, 16));
  l->rec_off = 0;
  l->idx_key_off = round_up(static_cast<int64_t>(block_size) * l->rec_stride, 256);
  l->idx_scale_off = round_up(l->idx_key_off + static_cast<int64_t>(block_size) * key_bytes_of(d_index, key_format), 256);
  l->layer_stride = round_up(l->idx_scale_off + 4ll * block_size, 256);
  l->block_stride = l->layer_stride * n_layers;
  return SMLA_OK;
}

size_t smla_workspace_size(const smla_layout_t* layout, const smla_params_t* params, int n_tokens, int max_ctx) {
  if (!layout_ok(layout) || params == nullptr || n_tokens <= 0 || max_ctx <= 0 || params->top_k <= 0) return 0;
  const int64_t stride = round_up(max_ctx, 4);
  const int g = query_group(n_tokens, stride);
  // the split top-k's candidates and the split attention's partials share one region (the stream
  // runs them one after the other)
  const size_t split = std::max(smla_attend_workspace_size(layout, params, g), smla_topk_workspace_size(params, g));
  return static_cast<size_t>(round_up(static_cast<int64_t>(g) * stride * 4, 256) +
                             round_up(static_cast<int64_t>(g) * params->top_k * 4, 256)) +
         split;
}

size_t smla_attend_workspace_size(const smla_layout_t* layout, const smla_params_t* params, int n_tokens) {
  if (!layout_ok(layout) || params == nullptr || n_tokens <= 0 || params->n_heads <= 0) return 0;
  // rows fewer than the SMs are split (rows x splits stay within kMaxSplitUnits, >= any SM count);
  // up to eight rows per SM are balanced over the SMs (two partial slots per SM)
  return n_tokens < 8 * kMaxSplitUnits ? attend_split_bytes(params->n_heads, layout->d_latent, 2 * kMaxSplitUnits)
                                       : 0;
}

smla_status_t kvpack_store(const smla_layout_t* layout, void* pool, int layer, const void* latent, const void* rope,
                           const uint8_t* idx_k, const float* idx_scale, const int64_t* slot_mapping, int n_tokens,
                           void* stream) {
  if (!layout_ok(layout) || n_tokens < 0 || layer < 0 || layer >= layout->n_layers) return SMLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return SMLA_OK;
  if (!pool || !latent || !idx_k || !idx_scale || !slot_mapping || (layout->d_rope > 0 && !rope))
    return SMLA_ERR_INVALID_ARG;
  DeviceInfo* d;
  smla_status_t st = check_device(&d);
  if (st != SMLA_OK) return st;
  return launch_kvpack_store(kernel_layout(*layout), pool, layer, latent, rope, idx_k, idx_scale, slot_mapping,
                             n_tokens, static_cast<cudaStream_t>(stream), d->err);
}

smla_status_t smla_index_scores(const smla_layout_t* layout, const smla_params_t* params, const void* pool, int layer,
                                const uint8_t* q_idx, const float* w, const int32_t* block_table, int bt_stride,
                                const int32_t* seq_lens, const int32_t* query_start_loc, int batch, int n_tokens,
                                int max_q, int max_ctx, float* scores, int64_t scores_stride, void* stream) {
  if (!layout_ok(layout) || !params || layer < 0 || layer >= layout->n_layers || batch <= 0 || n_tokens < 0 ||
      max_q < 0 || max_ctx < 0)
    return SMLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return SMLA_OK;
  if (!pool || !q_idx || !w || !block_table || !seq_lens || !query_start_loc || !scores || scores_stride < max_ctx ||
      static_cast<int64_t>(bt_stride) * layout->block_size < max_ctx || max_q <= 0)
    return SMLA_ERR_INVALID_ARG;
  DeviceInfo* d;
  smla_status_t st = check_device(&d);
  if (st != SMLA_OK) return st;
  return launch_index_scores(kernel_layout(*layout), params->n_idx_heads, pool, layer, q_idx, w, block_table,
                             bt_stride, seq_lens, query_start_loc, batch, 0, n_tokens, max_q, max_ctx, scores,
                             scores_stride, static_cast<cudaStream_t>(stream), d->err);
}

smla_status_t smla_topk(const smla_params_t* params, const float* scores, int64_t scores_stride,
                        const int32_t* seq_lens, const int32_t* query_start_loc, int batch, int n_tokens,
                        int32_t* topk_idx, void* workspace, size_t workspace_bytes, void* stream) {
  if (!params || params->top_k <= 0 || batch <= 0 || n_tokens < 0 || scores_stride <= 0 ||
      (workspace == nullptr && workspace_bytes != 0))
    return SMLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return SMLA_OK;
  if (!scores || !seq_lens || !query_start_loc || !topk_idx) return SMLA_ERR_INVALID_ARG;
  DeviceInfo* d;
  smla_status_t st = check_device(&d);
  if (st != SMLA_OK) return st;
  return launch_topk(params->top_k, scores, scores_stride, seq_lens, query_start_loc, batch, 0, n_tokens, topk_idx,
                     static_cast<cudaStream_t>(stream), d->err, workspace, workspace_bytes);
}

size_t smla_topk_workspace_size(const smla_params_t* params, int n_tokens) {
  if (params == nullptr || params->top_k <= 0 || n_tokens <= 0) return 0;
  // rows fewer than a wave of top-k CTAs are split; rows x segments stay within kMaxTopkSplitRows
  return n_tokens < kMaxTopkSplitRows ? topk_split_bytes(kMaxTopkSplitRows, params->top_k) : 0;
}

smla_status_t smla_attend(const smla_layout_t* layout, const smla_params_t* params, const void* pool, int layer,
                          const void* q, const void* q_pe, const int32_t* topk_idx, const int32_t* block_table,
                          int bt_stride, const int32_t* query_start_loc, int batch, int n_tokens, void* out,
                          float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!layout_ok(layout) || !params || layer < 0 || layer >= layout->n_layers || batch <= 0 || n_tokens < 0 ||
      params->top_k <= 0 || params->n_heads <= 0 || (workspace == nullptr && workspace_bytes != 0))
    return SMLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return SMLA_OK;
  if (!pool || !q || (layout->d_rope > 0 && !q_pe) || !topk_idx || !block_table || !query_start_loc || !out || !lse ||
      bt_stride <= 0)
    return SMLA_ERR_INVALID_ARG;
  DeviceInfo* d;
  smla_status_t st = check_device(&d);
  if (st != SMLA_OK) return st;
  return launch_attend(kernel_layout(*layout), params->n_heads, params->top_k, params->softmax_scale, pool, layer, q,
                       q_pe, topk_idx, block_table, bt_stride, query_start_loc, batch, 0, n_tokens, out, lse,
                       static_cast<cudaStream_t>(stream), d->err, nullptr, nullptr, 0, workspace, workspace_bytes);
}

smla_status_t smla_attend_hisparse(const smla_layout_t* layout, const smla_params_t* params, const void* pool,
                                   int layer, const void* host_records, const int32_t* host_block_map,
                                   int64_t n_host_blocks, const void* q, const void* q_pe, const int32_t* topk_idx,
                                   const int32_t* block_table, int bt_stride, const int32_t* query_start_loc,
                                   int batch, int n_tokens, void* out, float* lse, void* stream) {
  if (!layout_ok(layout) || !params || layer < 0 || layer >= layout->n_layers || batch <= 0 || n_tokens < 0 ||
      params->top_k <= 0 || params->n_heads <= 0 || n_host_blocks < 0)
    return SMLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return SMLA_OK;
  if (!pool || !q || (layout->d_rope > 0 && !q_pe) || !topk_idx || !block_table || !query_start_loc || !out || !lse ||
      bt_stride <= 0 || !host_block_map || (n_host_blocks > 0 && !host_records) ||
      (reinterpret_cast<uintptr_t>(host_records) & 15) != 0)
    return SMLA_ERR_INVALID_ARG;
  DeviceInfo* d;
  smla_status_t st = check_device(&d);
  if (st != SMLA_OK) return st;
  return launch_attend(kernel_layout(*layout), params->n_heads, params->top_k, params->softmax_scale, pool, layer, q,
                       q_pe, topk_idx, block_table, bt_stride, query_start_loc, batch, 0, n_tokens, out, lse,
                       static_cast<cudaStream_t>(stream), d->err, host_records, host_block_map, n_host_blocks);
}

smla_status_t smla_decode(const smla_layout_t* layout, const smla_params_t* params, void* pool, int layer,
                          const void* new_latent, const void* new_rope, const uint8_t* new_idx_k,
                          const float* new_idx_scale, const int64_t* slot_mapping, const void* q, const void* q_pe,
                          const uint8_t* q_idx, const float* w, const int32_t* block_table, int bt_stride,
                          const int32_t* seq_lens, const int32_t* query_start_loc, int batch, int n_tokens,
                          int max_q, int max_ctx, void* out, float* lse, int32_t* topk_idx_out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  const StepArgs args{layout,   params,     pool,    layer,   new_latent, new_rope,  new_idx_k,       new_idx_scale,
                      slot_mapping, q,      q_pe,    q_idx,   w,          block_table, bt_stride,     seq_lens,
                      query_start_loc, batch, n_tokens, max_q, max_ctx,   out,       lse};
  smla_status_t st = check_step(args);
  if (st != SMLA_OK || n_tokens == 0) return st;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
      workspace_bytes < smla_workspace_size(layout, params, n_tokens, max_ctx))
    return SMLA_ERR_INVALID_ARG;
  DeviceInfo* d;
  st = check_device(&d);
  if (st != SMLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const KernelLayout L = kernel_layout(*layout);
  if (slot_mapping != nullptr) {
    st = launch_kvpack_store(L, pool, layer, new_latent, new_rope, new_idx_k, new_idx_scale, slot_mapping, n_tokens,
                             s, d->err);
    if (st != SMLA_OK) return st;
  }
  const int64_t stride = round_up(max_ctx, 4);
  const int g = static_cast<int>(wave_aligned_group(query_group(n_tokens, stride), n_tokens));
  float* scores = static_cast<float*>(workspace);
  int32_t* topk_ws =
      reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + round_up(static_cast<int64_t>(g) * stride * 4, 256));
  // the rest of the workspace holds the split-attention partials
  const size_t used = static_cast<size_t>(round_up(static_cast<int64_t>(g) * stride * 4, 256) +
                                          round_up(static_cast<int64_t>(g) * params->top_k * 4, 256));
  void* split_ws = workspace_bytes > used ? static_cast<uint8_t*>(workspace) + used : nullptr;
  const size_t split_bytes = workspace_bytes > used ? workspace_bytes - used : 0;
  for (int t0 = 0; t0 < n_tokens; t0 += g) {
    const int t1 = t0 + g < n_tokens ? t0 + g : n_tokens;
    int32_t* topk = topk_idx_out ? topk_idx_out + static_cast<int64_t>(t0) * params->top_k : topk_ws;
    st = launch_index_scores(L, params->n_idx_heads, pool, layer, q_idx, w, block_table, bt_stride, seq_lens,
                             query_start_loc, batch, t0, t1, max_q, max_ctx, scores, stride, s, d->err);
    if (st != SMLA_OK) return st;
    st = launch_topk(params->top_k, scores, stride, seq_lens, query_start_loc, batch, t0, t1, topk, s, d->err,
                     split_ws, split_bytes);
    if (st != SMLA_OK) return st;
    st = launch_attend(L, params->n_heads, params->top_k, params->softmax_scale, pool, layer, q, q_pe, topk,
                       block_table, bt_stride, query_start_loc, batch, t0, t1, out, lse, s, d->err, nullptr, nullptr,
                       0, split_ws, split_bytes);
    if (st != SMLA_OK) return st;
  }
  return SMLA_OK;
}

smla_status_t smla_prefill_chunk(const smla_layout_t* layout, const smla_params_t* params, void* pool, int layer,
                                 const void* chunk_latent, const void* chunk_rope, const uint8_t* chunk_idx_k,
                                 const float* chunk_idx_scale, const int64_t* slot_mapping, const void* q,
                                 const void* q_pe, const uint8_t* q_idx, const float* w, const int32_t* block_table,
                                 int bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc, int batch,
                                 int n_tokens, int chunk_len, int max_ctx, void* out, float* lse,
                                 int32_t* topk_idx_out, void* workspace, size_t workspace_bytes, void* stream) {
  // The chunk's own keys must be in the pool before any of its tokens is scored.
  if (n_tokens > 0 && (slot_mapping == nullptr || chunk_latent == nullptr || chunk_idx_k == nullptr ||
                       chunk_idx_scale == nullptr || (layout != nullptr && layout->d_rope > 0 && chunk_rope == nullptr)))
    return SMLA_ERR_INVALID_ARG;
  return smla_decode(layout, params, pool, layer, chunk_latent, chunk_rope, chunk_idx_k, chunk_idx_scale, slot_mapping,
                     q, q_pe, q_idx, w, block_table, bt_stride, seq_lens, query_start_loc, batch, n_tokens, chunk_len,
                     max_ctx, out, lse, topk_idx_out, workspace, workspace_bytes, stream);
}

smla_status_t smla_selftest_wait(int64_t limit_ns, void* stream) {
  if (limit_ns < 1000000 || limit_ns > 10000000000ll) return SMLA_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  if (smla_status_t st = check_device(&d); st != SMLA_OK) return st;
  wait_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(d->err, static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

smla_status_t smla_get_last_error(void* stream) {
  DeviceInfo* d = current_device();
  if (d == nullptr) return SMLA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SMLA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return SMLA_ERR_CUDA;
  const unsigned zero = 0;
  if (v != 0 && cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return SMLA_ERR_CUDA;
  return static_cast<smla_status_t>(v);
}

}  // extern "C"
