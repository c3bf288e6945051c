// Internal declarations shared by the libsmla translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "smla.h"
#include "smla_device.cuh"

namespace smla {

// Kernel-side copy of smla_layout_t (passed by value).
struct KernelLayout {
  int32_t block_size, n_layers, d_latent, d_rope, quant_tile, d_index, n_scales, rec_stride;
  int32_t key_format, key_bytes;  // smla_key_format_t; bytes of one cached indexer key
  int64_t num_blocks, rec_off, idx_key_off, idx_scale_off, layer_stride, block_stride;
};

// Bytes of one cached indexer key of d_index elements in the given format.
inline int32_t key_bytes_of(int32_t d_index, int32_t key_format) {
  return key_format == SMLA_KEY_E2M1 ? d_index / 2 : d_index;
}

inline KernelLayout kernel_layout(const smla_layout_t& l) {
  KernelLayout k;
  k.block_size = l.block_size;
  k.n_layers = l.n_layers;
  k.d_latent = l.d_latent;
  k.d_rope = l.d_rope;
  k.quant_tile = l.quant_tile;
  k.d_index = l.d_index;
  k.n_scales = l.n_scales;
  k.rec_stride = l.rec_stride;
  k.key_format = l.idx_key_format;
  k.key_bytes = key_bytes_of(l.d_index, l.idx_key_format);
  k.num_blocks = l.num_blocks;
  k.rec_off = l.rec_off;
  k.idx_key_off = l.idx_key_off;
  k.idx_scale_off = l.idx_scale_off;
  k.layer_stride = l.layer_stride;
  k.block_stride = l.block_stride;
  return k;
}

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry point (nullptr if absent).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// Device error word (defined in api.cu); launchers receive its address.
unsigned* device_error_word();
int device_sm_count();
// The current device's error word, after checking that the device is sm_103 (SMLA_ERR_UNSUPPORTED
// otherwise; SMLA_ERR_CUDA if the device or the word's address cannot be read).
smla_status_t checked_device(unsigned** err);

// A layout is accepted only as smla_layout_init produced it: its shape fields pass that call's
// checks and every derived field (record size, region offsets, strides) equals what it computes.
bool layout_ok(const smla_layout_t* l);

// Shapes compiled into the kernels; the entry points refuse others with SMLA_ERR_UNSUPPORTED
// before anything is enqueued.
bool store_shape_supported(const KernelLayout& L);
bool index_shape_supported(const KernelLayout& L, int n_idx_heads);
bool attend_shape_supported(const KernelLayout& L, int n_heads);

// Arguments of one fused step (smla_decode and smla_decode_static take the same ones apart from
// the scratch), checked by check_step() in the same order for both.
struct StepArgs {
  const smla_layout_t* layout;
  const smla_params_t* params;
  void* pool;
  int layer;
  const void *new_latent, *new_rope;
  const uint8_t* new_idx_k;
  const float* new_idx_scale;
  const int64_t* slot_mapping;
  const void *q, *q_pe;
  const uint8_t* q_idx;
  const float* w;
  const int32_t* block_table;
  int bt_stride;
  const int32_t *seq_lens, *query_start_loc;
  int batch, n_tokens, max_q, max_ctx;
  void* out;
  float* lse;
};
// SMLA_ERR_INVALID_ARG for a bad pointer, size or layout, SMLA_ERR_UNSUPPORTED for a shape the
// kernels do not build, else SMLA_OK (also for n_tokens == 0, which enqueues nothing).
smla_status_t check_step(const StepArgs& a);
// Launch attributes (shared-memory opt-in, occupancy) belong to a device: launchers keep
// them per device, in tables of kMaxDeviceSlots entries indexed by current_device_index().
constexpr int kMaxDeviceSlots = 64;
// The calling thread's current device, or -1 if it cannot be read or is beyond the table.
int current_device_index();

smla_status_t launch_kvpack_store(const KernelLayout& L, void* pool, int layer, const void* latent,
                                  const void* rope, const uint8_t* idx_k, const float* idx_scale,
                                  const int64_t* slot_mapping, int n_tokens, cudaStream_t stream, unsigned* err);

smla_status_t launch_index_scores(const KernelLayout& L, int n_idx_heads, const void* pool, int layer,
                                  const uint8_t* q_idx, const float* w, const int32_t* block_table, int bt_stride,
                                  const int32_t* seq_lens, const int32_t* query_start_loc, int batch, int tok_begin,
                                  int tok_end, int max_q, int max_ctx, float* scores, int64_t scores_stride,
                                  cudaStream_t stream, unsigned* err);

// CTAs of the top-k kernel resident at once on the current device (0 if unknown).
int topk_wave();

// Query tokens per group, rounded down to whole waves of the top-k kernel (which
// also gives the persistent attention grid a whole number of rows per CTA) when
// the group is smaller than the batch.  `g` is the largest group the scratch holds.
inline int64_t wave_aligned_group(int64_t g, int n_tokens) {
  if (g >= n_tokens) return n_tokens;
  const int wave = topk_wave();
  return (wave > 0 && g >= wave) ? g - g % wave : g;
}

// Scratch of the split top-k: candidate positions, then candidate scores, for `seg_rows`
// (row, segment) pairs of k entries each (two 256-byte rounded halves).
inline size_t topk_split_bytes(int seg_rows, int k) {
  return 2 * ((static_cast<size_t>(seg_rows) * k * 4 + 255) / 256 * 256);
}
// (row, segment) pairs the split top-k may use (any wave of top-k CTAs fits).
constexpr int kMaxTopkSplitRows = 512;

// split_ws / split_ws_bytes: scratch for splitting rows into segments (nullptr: one CTA per row).
smla_status_t launch_topk(int top_k, const float* scores, int64_t scores_stride, const int32_t* seq_lens,
                          const int32_t* query_start_loc, int batch, int tok_begin, int tok_end, int32_t* topk_idx,
                          cudaStream_t stream, unsigned* err, void* split_ws = nullptr, size_t split_ws_bytes = 0);

// Scratch of split attention: fp32 partial outputs [units][n_heads][d_latent] (256-byte rounded),
// then fp32 partial lse [units][n_heads].
inline size_t split_out_bytes(int n_heads, int d_latent, int units) {
  return (static_cast<size_t>(units) * n_heads * d_latent * 4 + 255) / 256 * 256;
}
inline size_t attend_split_bytes(int n_heads, int d_latent, int units) {
  return split_out_bytes(n_heads, d_latent, units) + (static_cast<size_t>(units) * n_heads * 4 + 255) / 256 * 256;
}
// Units the fused entry points reserve scratch for (rows x splits never exceed the SM count).
constexpr int kMaxSplitUnits = 256;

// split_ws / split_ws_bytes: scratch for split attention (nullptr: each row on one CTA).
smla_status_t launch_attend(const KernelLayout& L, int n_heads, int top_k, float softmax_scale, const void* pool,
                            int layer, const void* q, const void* q_pe, const int32_t* topk_idx,
                            const int32_t* block_table, int bt_stride, const int32_t* query_start_loc, int batch,
                            int tok_begin, int tok_end, void* out, float* lse, cudaStream_t stream, unsigned* err,
                            const void* host_records = nullptr, const int32_t* host_block_map = nullptr,
                            int64_t n_host_blocks = 0, void* split_ws = nullptr, size_t split_ws_bytes = 0);

}  // namespace smla
