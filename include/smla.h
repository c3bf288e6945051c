/*
 * smla.h -- C ABI of the GB300 paged top-k sparse-MLA library (libsmla.so).
 *
 * The library computes the data-parallel hot path of top-k sparse MLA over a
 * paged FP8 KV cache held in one shared block pool:
 *
 *   kvpack_store       new tokens -> packed FP8 records in the pool
 *   smla_index_scores  per-query-token indexer scores over its visible context
 *   smla_topk          top-k cached positions per query token
 *   smla_attend        latent MQA attention over the selected positions
 *   smla_decode        the four steps above in one call (decode steps with
 *                      MTP draft tokens, and chunked prefill)
 *
 * Sources (cited by page title and section):
 *   [AgentX]  "vLLM、エージェント型ワークロード向け最適化技術「AgentX」を公開"
 *             (news.ainew.jp rendering of the vLLM AgentX post), sections
 *             "Hybrid KV cache management", "Kimi K3", "DeepSeek V4",
 *             "Closing the loop: kernels".
 *   [GLM-5.3] aisoku.org article on vLLM serving GLM-5.3 on 16xH200
 *             (PCP8xDCP8 prefill, Hybrid HiSparse decode), sections
 *             "What is new", "Config and numbers", "How to try".
 *
 * Conventions for every call
 *   - All array pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them after the call returns.  Host pointers are
 *     only the smla_layout_t / smla_params_t descriptors (read during the call).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = legacy default stream).  Nothing allocates device memory: scratch
 *     space is the caller's `workspace`.
 *   - Integer arrays are int32 unless stated; bf16 arrays are raw 16-bit
 *     bfloat16 patterns; "e4m3" arrays are uint8 OCP FP8 E4M3 codes.
 *   - Return value: SMLA_OK, or an error detected on the host before anything
 *     was enqueued (SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED) or at launch
 *     (SMLA_ERR_CUDA).  Errors found by the kernels themselves (an out-of-range
 *     block id or slot, a bounded wait that gave up) are latched in a device
 *     word and reported by smla_get_last_error(); the offending read is
 *     clamped or skipped, never performed out of bounds.
 *   - No C++ exceptions cross the ABI.  Calls on different streams may run
 *     concurrently; the latched error word is shared by all of them.  Calls
 *     may come from several host threads: the library's once-per-device
 *     set-up (device attributes, symbol addresses) is synchronised.
 *
 * Query geometry shared by the calls: sequence b has seq_lens[b] cached
 * tokens INCLUDING this step's tokens, and its query tokens are rows
 * query_start_loc[b] .. query_start_loc[b+1]-1.  Query i of the n_q tokens of
 * sequence b sits at position p = seq_lens[b] - n_q + i and sees positions
 * 0..p (itself included).  block_table[b * bt_stride + j / block_size] is the
 * physical block of logical position j.
 *
 * Values that are trusted, not checked: query_start_loc increases from 0 to
 * n_tokens, every sequence has at least as many cached tokens as query tokens,
 * and max_ctx (where a call takes it) is at least every seq_lens entry.  The
 * kernels size their loops from these values, so a call that breaks them
 * reads and writes outside the score rows and block-table rows it was given.
 * Block ids and slots, by contrast, are checked on the device (see above).
 */
#ifndef SMLA_H
#define SMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum smla_status {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size or stride          */
  SMLA_ERR_UNSUPPORTED = 2,  /* shape not built into this library / no sm_103a device */
  SMLA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed       */
  SMLA_ERR_BAD_INDEX = 4,    /* device saw a block id / slot outside the pool (read clamped) */
  SMLA_ERR_TIMEOUT = 5,      /* a bounded on-device wait gave up            */
  SMLA_ERR_SCRATCH_LIMIT = 6 /* smla_decode_static: one query token's scratch exceeds the static array */
} smla_status_t;

/*
 * Format of the cached indexer keys ([AgentX "Hybrid KV cache management"]:
 * with the FP4 indexer the packed layout needs a smaller allocation unit).
 *   SMLA_KEY_E4M3: d_index OCP FP8 E4M3 codes, one byte each.
 *   SMLA_KEY_E2M1: d_index OCP MX FP4 E2M1 codes, two per byte (element 2i in
 *                  the low nibble of byte i, element 2i+1 in the high nibble).
 * Either way the key's fp32 scale s_I multiplies its score after the head sum.
 */
typedef enum smla_key_format {
  SMLA_KEY_E4M3 = 0,
  SMLA_KEY_E2M1 = 1
} smla_key_format_t;

/*
 * Packed block-pool layout ([AgentX "Hybrid KV cache management"]: all cache
 * groups and layers of a block in one contiguous allocation; the block is the
 * single allocation unit).  Per block, per layer l:
 *
 *   [block_size latent records, rec_stride bytes each]
 *   [block_size indexer keys, d_index (E4M3) or d_index/2 (E2M1) bytes each]
 *   [block_size indexer key scales, fp32]
 *
 * every region on a 256-byte boundary; a record is
 *   [d_latent e4m3 codes][d_latent/quant_tile fp32 scales][d_rope bf16] (padded to 16 B).
 * Filled in by smla_layout_init(); read-only afterwards.  Every entry point
 * accepts a layout only as smla_layout_init filled it in: it recomputes the
 * derived fields from the shape fields and refuses any difference with
 * SMLA_ERR_INVALID_ARG.
 */
typedef struct smla_layout {
  int32_t block_size;     /* tokens per block                                  */
  int32_t n_layers;       /* layers packed in one block                        */
  int32_t d_latent;       /* latent (no-rope) dims, FP8 in the cache           */
  int32_t d_rope;         /* rope dims, bf16 in the cache                      */
  int32_t quant_tile;     /* latent elements per fp32 scale                    */
  int32_t d_index;        /* indexer key dims (e4m3)                           */
  int64_t num_blocks;     /* pool capacity in blocks                           */
  int32_t n_scales;       /* d_latent / quant_tile                             */
  int32_t rec_bytes;      /* d_latent + 4*n_scales + 2*d_rope                  */
  int32_t rec_stride;     /* rec_bytes rounded up to 16                        */
  int32_t idx_key_format; /* smla_key_format_t of the cached indexer keys      */
  int64_t rec_off;        /* byte offset of the record region in a layer slice */
  int64_t idx_key_off;    /* byte offset of the indexer-key region             */
  int64_t idx_scale_off;  /* byte offset of the indexer-scale region           */
  int64_t layer_stride;   /* bytes of one layer slice of a block               */
  int64_t block_stride;   /* bytes of one block (all layers)                   */
} smla_layout_t;

/* Attention / indexer hyper-parameters. */
typedef struct smla_params {
  int32_t n_heads;        /* query heads sharing the latent (<= 64)            */
  int32_t n_idx_heads;    /* indexer heads                                     */
  int32_t top_k;          /* positions kept per query token                    */
  float softmax_scale;    /* sigma in s = sigma * (q.K + q_pe.kpe)             */
} smla_params_t;

/* Fill `layout` from the shape, with E4M3 indexer keys; checks divisibility.
 * Host only, no device work. */
smla_status_t smla_layout_init(smla_layout_t* layout, int block_size, int n_layers, int d_latent,
                               int d_rope, int quant_tile, int d_index, int64_t num_blocks);

/* smla_layout_init with the indexer-key format (an smla_key_format_t).  E2M1
 * keys need d_index to be a multiple of 32; the key region then takes
 * block_size * d_index / 2 bytes (for the DeepSeek shape the block of one layer
 * shrinks from 50,432 to 46,336 bytes).  The indexer kernels are built for
 * E2M1 keys with 64 indexer heads of 128 dims. */
smla_status_t smla_layout_init_keys(smla_layout_t* layout, int block_size, int n_layers, int d_latent,
                                    int d_rope, int quant_tile, int d_index, int key_format,
                                    int64_t num_blocks);

/* Bytes of `workspace` that smla_decode needs for these sizes (scores + top-k
 * scratch, then the split-attention scratch of smla_attend_workspace_size,
 * 256-byte aligned pieces).  max_ctx = the largest seq_lens entry. */
size_t smla_workspace_size(const smla_layout_t* layout, const smla_params_t* params,
                           int n_tokens, int max_ctx);

/*
 * kvpack_store -- write n_tokens new tokens into layer `layer` of the pool.
 * [GLM-5.3 "How to try", "Config and numbers"]: the KV cache is FP8.
 *   latent      bf16 [n_tokens, d_latent]
 *   rope        bf16 [n_tokens, d_rope]
 *   idx_k       uint8 [n_tokens, key bytes] copied verbatim: d_index E4M3 codes,
 *               or d_index/2 bytes of packed E2M1 codes (layout.idx_key_format)
 *   idx_scale   fp32 [n_tokens]            copied verbatim
 *   slot_mapping int64 [n_tokens]          physical slot (block*block_size+off); -1 = skip
 * Per quant_tile of the latent: scale = amax/448 (IEEE fp32 division; 1.0 if
 * that is 0), code = E4M3 round-to-nearest-even, saturating, of x/scale.
 * Latent values must be finite.  Slots >= num_blocks*block_size are skipped
 * and latch SMLA_ERR_BAD_INDEX.
 */
smla_status_t kvpack_store(const smla_layout_t* layout, void* pool, int layer, const void* latent,
                           const void* rope, const uint8_t* idx_k, const float* idx_scale,
                           const int64_t* slot_mapping, int n_tokens, void* stream);

/*
 * smla_index_scores -- indexer scores of every query token over its context.
 * [AgentX "DeepSeek V4"]: 64 indexer heads produce one global selection per
 * token; [GLM-5.3 "What is new"]: the indexer cost is quadratic in context.
 *   I[t, j] = s_I[j] * sum_h w[t, h] * ReLU(sum_d q_idx[t, h, d] * k_I[j, d]),  j <= p(t)
 * computed with FP8 tensor-core MMAs (E2M1 keys times E4M3 queries when the
 * layout holds FP4 keys), fp32 accumulation and an fp32 head reduction in head
 * order.
 *   q_idx   e4m3 [n_tokens, n_idx_heads, d_index]
 *   w       fp32 [n_tokens, n_idx_heads]
 *   scores  fp32 [n_tokens, scores_stride]: entries j <= p(t) are written,
 *           the rest of each row is left untouched.  scores_stride >= max_ctx.
 *   max_q   largest number of query tokens of one sequence in this call
 *   max_ctx largest seq_lens entry
 */
smla_status_t smla_index_scores(const smla_layout_t* layout, const smla_params_t* params,
                                const void* pool, int layer, const uint8_t* q_idx, const float* w,
                                const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                                const int32_t* query_start_loc, int batch, int n_tokens, int max_q,
                                int max_ctx, float* scores, int64_t scores_stride, void* stream);

/*
 * smla_topk -- exact top-k of each row of `scores` over positions 0..p(t).
 * [GLM-5.3 "What is new"] (2,048 tokens), [AgentX "DeepSeek V4"].
 * Ties go to the lower position; scores compare as fp32 values (-0 == +0).
 *   topk_idx int32 [n_tokens, top_k]: kept logical positions in ascending
 *            order, -1 padded when p(t)+1 < top_k.
 */
smla_status_t smla_topk(const smla_params_t* params, const float* scores, int64_t scores_stride,
                        const int32_t* seq_lens, const int32_t* query_start_loc, int batch,
                        int n_tokens, int32_t* topk_idx, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Scratch bytes with which smla_topk splits long rows of a small batch into segments: each
 * segment's top-k (positions and scores) becomes a candidate list, then each row's top-k is
 * taken over its candidates (0 when n_tokens is too large to need it).  workspace may be
 * NULL (with workspace_bytes 0): every row then runs on one CTA. */
size_t smla_topk_workspace_size(const smla_params_t* params, int n_tokens);

/*
 * smla_attend -- latent MQA attention over the selected positions.
 * [AgentX "Kimi K3"], [GLM-5.3 "What is new"]: the latent KV is shared by
 * all query heads; [AgentX "DeepSeek V4"]: attention runs over the top-k only.
 *   s[h, j] = softmax_scale * (q[t, h] . K[j] + q_pe[t, h] . kpe[j]),
 *   out[t, h] = sum_j softmax_j(s)[h, j] * K[j],  lse[t, h] = ln sum_j exp(s[h, j])
 * with K[j] the dequantised latent and kpe[j] the cached rope.
 *   q        bf16 [n_tokens, n_heads, d_latent]
 *   q_pe     bf16 [n_tokens, n_heads, d_rope]
 *   topk_idx int32 [n_tokens, top_k]; entries < 0 are ignored.  An entry at or
 *            beyond bt_stride * block_size (past the sequence's block-table
 *            row) is not looked up: it latches SMLA_ERR_BAD_INDEX and its
 *            record reads as zeros, like an out-of-range block id.
 *   out      bf16 [n_tokens, n_heads, d_latent]
 *   lse      fp32 [n_tokens, n_heads]  (natural log; -inf and out = 0 when no entry is valid)
 *   workspace, workspace_bytes: optional device scratch (NULL and 0 allowed).  With fewer
 *     query tokens than SMs and at least smla_attend_workspace_size() bytes, each token's
 *     selected positions are split into contiguous ranges over several CTAs (one wave in
 *     all); every range yields a normalised fp32 partial output and its lse in the scratch,
 *     and a merge kernel combines them as lse = ln sum_r exp(lse_r),
 *     out = sum_r exp(lse_r - lse) out_r.  With more tokens than SMs but a last round that
 *     would keep at most half of the SMs busy (e.g. 160 tokens on 152 SMs), every CTA takes
 *     an equal share of all tokens' position tiles instead; a token whose tiles straddle two
 *     CTAs is merged the same way from two partials.  Without a scratch, each token runs on
 *     one CTA.  The result agrees with the one-CTA path within rounding.
 */
smla_status_t smla_attend(const smla_layout_t* layout, const smla_params_t* params, const void* pool,
                          int layer, const void* q, const void* q_pe, const int32_t* topk_idx,
                          const int32_t* block_table, int bt_stride, const int32_t* query_start_loc,
                          int batch, int n_tokens, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Scratch bytes with which smla_attend splits or balances the tokens' ranges over CTAs:
 * partial outputs for up to 512 ranges, about 64 MiB for 64 heads of 512 dims (0 when
 * n_tokens is too large to need it). */
size_t smla_attend_workspace_size(const smla_layout_t* layout, const smla_params_t* params, int n_tokens);

/*
 * smla_attend_hisparse -- smla_attend with a host tier for the selected
 * records ([GLM-5.3 "What is new"]: Hybrid HiSparse decode keeps part of the
 * KV in host memory and fetches the selected entries from there, so decode
 * concurrency is no longer bounded by HBM).  The indexer keys stay in the HBM
 * pool; the 656-byte records of evicted blocks live in a host buffer that the
 * GPU reads directly (pinned, mapped host memory: on GB300 the reads go over
 * NVLink-C2C).
 *   host_block_map: int32 [layout.num_blocks] device array; -1 = the block's
 *     records are in `pool`, h >= 0 = they are host block h of host_records
 *   host_records: host-tier records, [n_host_blocks][n_layers][block_size]
 *     records of layout.rec_stride bytes, 16-byte aligned, device-accessible
 *     (e.g. cudaHostAlloc'd)
 *   other arguments and results as smla_attend.  A map entry >= n_host_blocks
 *   is latched as SMLA_ERR_BAD_INDEX and the record reads as zeros.
 */
smla_status_t smla_attend_hisparse(const smla_layout_t* layout, const smla_params_t* params, const void* pool,
                                   int layer, const void* host_records, const int32_t* host_block_map,
                                   int64_t n_host_blocks, const void* q, const void* q_pe, const int32_t* topk_idx,
                                   const int32_t* block_table, int bt_stride, const int32_t* query_start_loc,
                                   int batch, int n_tokens, void* out, float* lse, void* stream);

/*
 * smla_decode -- one step of the whole path for one layer:
 * kvpack_store(new tokens) -> smla_index_scores -> smla_topk -> smla_attend.
 * Serves decode steps with MTP drafts ([GLM-5.3 "Config and numbers"]: MTP3)
 * and chunked prefill on a cached prefix (many query tokens per sequence).
 *   new_latent/new_rope/new_idx_k/new_idx_scale/slot_mapping: as kvpack_store,
 *     n_tokens rows (slot_mapping may be NULL to skip the store)
 *   topk_idx_out: optional int32 [n_tokens, top_k] copy of the selection (NULL = none)
 *   workspace: device scratch of at least smla_workspace_size(...) bytes,
 *     256-byte aligned
 * Query tokens are processed in groups so the score scratch stays bounded.
 * Refused before anything is enqueued: a layout not made by smla_layout_init,
 * n_heads, n_idx_heads or top_k <= 0, a NULL q_pe while d_rope > 0 (or a NULL
 * new-token input while slot_mapping is given), bt_stride * block_size below
 * max_ctx (SMLA_ERR_INVALID_ARG); head counts and dimensions the kernels are
 * not built for (SMLA_ERR_UNSUPPORTED).
 */
smla_status_t smla_decode(const smla_layout_t* layout, const smla_params_t* params, void* pool,
                          int layer, const void* new_latent, const void* new_rope,
                          const uint8_t* new_idx_k, const float* new_idx_scale,
                          const int64_t* slot_mapping, const void* q, const void* q_pe,
                          const uint8_t* q_idx, const float* w, const int32_t* block_table,
                          int bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                          int batch, int n_tokens, int max_q, int max_ctx, void* out, float* lse,
                          int32_t* topk_idx_out, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * smla_prefill_chunk -- chunked prefill on a cached prefix, one layer
 * ([AgentX "Head-of-line blocking"]: the chunked-prefill scheduler splits long
 * prefills into per-step token budgets; [GLM-5.3 "What is new"]: prefill of
 * long prompts split into chunks).  Each sequence b appends a chunk
 * of n_b = query_start_loc[b+1] - query_start_loc[b] tokens whose KV is stored
 * first (chunk_latent/chunk_rope/chunk_idx_k/chunk_idx_scale at slot_mapping,
 * required); seq_lens[b] includes the chunk, and chunk token i attends the
 * positions <= seq_lens[b] - n_b + i (causal within the chunk, the whole
 * prefix before it).
 *   chunk_len: the largest n_b of the call (the query-group bound of the
 *     indexer); other arguments and results as smla_decode.
 *   Returns SMLA_ERR_INVALID_ARG when slot_mapping or a chunk input is NULL.
 */
smla_status_t smla_prefill_chunk(const smla_layout_t* layout, const smla_params_t* params, void* pool,
                                 int layer, const void* chunk_latent, const void* chunk_rope,
                                 const uint8_t* chunk_idx_k, const float* chunk_idx_scale,
                                 const int64_t* slot_mapping, const void* q, const void* q_pe,
                                 const uint8_t* q_idx, const float* w, const int32_t* block_table,
                                 int bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                                 int batch, int n_tokens, int chunk_len, int max_ctx, void* out, float* lse,
                                 int32_t* topk_idx_out, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * smla_decode_static -- smla_decode for callers that cannot allocate device
 * memory, such as code whose device memory is entirely owned by a serving
 * engine's allocator (one that reserves all free HBM for the KV block pool and
 * hands out no other buffers) or a host runtime with no device-allocation hook.
 * The pages have no counterpart of this entry point; it only changes where the
 * scratch lives.
 *   Arguments and results are those of smla_decode without workspace /
 *   workspace_bytes, checked in the same order and refused with the same
 *   status (including SMLA_ERR_UNSUPPORTED on a device that is not sm_103):
 *   the fp32 scores and top-k indices live in a 64 MiB static
 *   __device__ array inside the library, which every GPU that loads the library
 *   holds until the process exits.  No cudaMalloc/cudaFree or other allocating
 *   call is made.
 *   Query tokens are processed in groups that fit the array; if a single query
 *   token needs more (4 * round_up(max_ctx, 4) + 4 * top_k bytes > 64 MiB - 512,
 *   i.e. max_ctx above about 16.7M positions), the call returns
 *   SMLA_ERR_SCRATCH_LIMIT before enqueuing anything.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make it before any stream
 *   capture.  All calls share the array and it keeps the last call's contents
 *   (nothing in it needs to start at zero); calls that overlap on the GPU race
 *   on it, so order them on one stream.
 */
smla_status_t smla_decode_static(const smla_layout_t* layout, const smla_params_t* params, void* pool,
                                 int layer, const void* new_latent, const void* new_rope,
                                 const uint8_t* new_idx_k, const float* new_idx_scale,
                                 const int64_t* slot_mapping, const void* q, const void* q_pe,
                                 const uint8_t* q_idx, const float* w, const int32_t* block_table,
                                 int bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                                 int batch, int n_tokens, int max_q, int max_ctx, void* out, float* lse,
                                 int32_t* topk_idx_out, void* stream);

/*
 * Split-context (DCP-style) decode, emulated with N token shards on one GPU
 * ([AgentX "Kimi K3"]: decode context parallelism with an LSE merge of partial
 * outputs; [GLM-5.3 "What is new"]: DCP8 decode).  Shard r holds the positions
 * j = N*i + r of every sequence at local position i; each shard runs
 * smla_index_scores and smla_topk over its own positions (a query at global
 * position p sees local positions 0 .. (p - r) / N), then:
 *
 * smla_dcp_topk_merge -- the candidate exchange.  For every query token t the
 * union of the shards' local top-k candidates (score, global position) is
 * reduced to the top_k highest by (score desc, global position asc), which is
 * the unsharded selection; shard r receives its selected local positions.
 *   shard_scores: fp32, shard r's score row of token t at
 *     shard_scores[r * shard_stride + t * row_stride + i] (i = local position)
 *   shard_topk: int32 [n_shards, n_tokens, top_k], each row ascending, -1 padded
 *     (smla_topk's output on each shard)
 *   shard_sel: int32 [n_shards, n_tokens, top_k] out, selected local positions
 *     ascending, -1 padded (the top-k input of smla_attend on shard r)
 *   merged: optional int32 [n_tokens, top_k] out, the selected global positions
 *     ascending, -1 padded (NULL = not written)
 *   n_shards * top_k <= 16384 and top_k <= 4096, else SMLA_ERR_UNSUPPORTED.
 */
smla_status_t smla_dcp_topk_merge(const float* shard_scores, int64_t shard_stride, int64_t row_stride,
                                  const int32_t* shard_topk, int n_shards, int n_tokens, int top_k,
                                  int32_t* shard_sel, int32_t* merged, void* stream);

/*
 * smla_lse_merge -- the output exchange: combine the shards' partial results
 * (smla_attend on each shard over its shard_sel) into
 *   lse = ln sum_r exp(lse_r),  out = sum_r exp(lse_r - lse) * out_r
 * in fp32 (a shard with lse_r = -inf contributes nothing; all -inf gives out = 0,
 * lse = -inf).
 *   parts_out: bf16 [n_shards, n_tokens, n_heads, d], 16-byte aligned, d % 8 == 0
 *   parts_lse: fp32 [n_shards, n_tokens, n_heads]
 *   out: bf16 [n_tokens, n_heads, d] (16-byte aligned), lse: fp32 [n_tokens, n_heads]
 */
smla_status_t smla_lse_merge(const void* parts_out, const float* parts_lse, int n_shards, int n_tokens,
                             int n_heads, int d, void* out, float* lse, void* stream);

/* Self-check of the on-device wait bound and of the pipelined kernels' exit
 * protocol.  One CTA of four warps: warp 0 waits on an mbarrier that no thread
 * ever arrives at, warps 1-3 on one that completes; the failed wait gives up
 * after `limit_ns` nanoseconds (1 ms .. 10 s of %globaltimer), latches
 * SMLA_ERR_TIMEOUT in the device error word and is ORed into the group barrier,
 * so that all four warps leave together and the kernel returns.  The caller reads
 * the status with smla_get_last_error(); the context stays usable.  Returns
 * SMLA_ERR_INVALID_ARG for a limit outside the range, else the launch status. */
smla_status_t smla_selftest_wait(int64_t limit_ns, void* stream);

/* Synchronise `stream`, return the latched device error (and clear it). */
smla_status_t smla_get_last_error(void* stream);

/* Human-readable name of a status code (static string). */
const char* smla_status_string(smla_status_t status);

/* Library version, major*10000 + minor*100 + patch. */
int smla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_H */
