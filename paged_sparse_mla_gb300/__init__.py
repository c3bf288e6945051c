"""Python binding of libsmla, the GB300 paged top-k sparse-MLA library.

Argument marshalling only: every function takes torch CUDA tensors on the
current device, checks their dtypes and that each holds at least the elements
the kernels read or write through it (a short buffer raises here instead of
being overrun on the GPU), and calls the same-named C entry point of
``include/smla.h`` through ctypes.  All computation happens in the library's
CUDA kernels; there is no CPU path.  If ``_build/libsmla.so`` is missing the
import of ``lib()`` raises -- build it with ``paged_sparse_mla_gb300.build_lib.build()``.
"""

import ctypes
import os

import torch

from . import build_lib

__all__ = [
    "SmlaError", "Layout", "Params", "lib", "layout_init", "workspace_size", "kvpack_store",
    "smla_index_scores", "smla_topk", "smla_attend", "smla_decode", "smla_get_last_error",
    "status_string", "version", "EXPORTED_SYMBOLS", "smla_decode_static", "smla_prefill_chunk",
    "smla_dcp_topk_merge", "smla_lse_merge", "smla_attend_hisparse", "smla_selftest_wait",
    "attend_workspace_size", "topk_workspace_size",
]

EXPORTED_SYMBOLS = (
    "smla_layout_init", "smla_workspace_size", "kvpack_store", "smla_index_scores", "smla_topk",
    "smla_attend", "smla_decode", "smla_get_last_error", "smla_status_string", "smla_version",
    "smla_decode_static", "smla_prefill_chunk", "smla_dcp_topk_merge", "smla_lse_merge", "smla_attend_hisparse",
    "smla_selftest_wait", "smla_attend_workspace_size", "smla_topk_workspace_size", "smla_layout_init_keys",
)

KEY_FORMATS = {"e4m3": 0, "e2m1": 1}  # smla_key_format_t

STATUS = {0: "SMLA_OK", 1: "SMLA_ERR_INVALID_ARG", 2: "SMLA_ERR_UNSUPPORTED", 3: "SMLA_ERR_CUDA",
          4: "SMLA_ERR_BAD_INDEX", 5: "SMLA_ERR_TIMEOUT", 6: "SMLA_ERR_SCRATCH_LIMIT"}


class SmlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class Layout(ctypes.Structure):
    """Mirror of smla_layout_t."""
    _fields_ = [
        ("block_size", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("d_latent", ctypes.c_int32),
        ("d_rope", ctypes.c_int32), ("quant_tile", ctypes.c_int32), ("d_index", ctypes.c_int32),
        ("num_blocks", ctypes.c_int64), ("n_scales", ctypes.c_int32), ("rec_bytes", ctypes.c_int32),
        ("rec_stride", ctypes.c_int32), ("idx_key_format", ctypes.c_int32), ("rec_off", ctypes.c_int64),
        ("idx_key_off", ctypes.c_int64), ("idx_scale_off", ctypes.c_int64), ("layer_stride", ctypes.c_int64),
        ("block_stride", ctypes.c_int64),
    ]

    @property
    def pool_bytes(self) -> int:
        return self.num_blocks * self.block_stride

    @property
    def key_bytes(self) -> int:
        """Bytes of one cached indexer key: d_index E4M3 codes, or d_index / 2 bytes of packed E2M1."""
        return self.d_index // 2 if self.idx_key_format == KEY_FORMATS["e2m1"] else self.d_index


class Params(ctypes.Structure):
    """Mirror of smla_params_t."""
    _fields_ = [("n_heads", ctypes.c_int32), ("n_idx_heads", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]


_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    """Load libsmla.so (built in-tree).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(build_lib.LIB):
            raise RuntimeError(f"libsmla.so not built ({build_lib.LIB}); run paged_sparse_mla_gb300.build_lib.build()")
        L = ctypes.CDLL(build_lib.LIB)
        LP, PP = ctypes.POINTER(Layout), ctypes.POINTER(Params)
        sig = {
            "smla_layout_init": (_I, [LP, _I, _I, _I, _I, _I, _I, _I64]),
            "smla_layout_init_keys": (_I, [LP, _I, _I, _I, _I, _I, _I, _I, _I64]),
            "smla_workspace_size": (ctypes.c_size_t, [LP, PP, _I, _I]),
            "kvpack_store": (_I, [LP, _P, _I, _P, _P, _P, _P, _P, _I, _P]),
            "smla_index_scores": (_I, [LP, PP, _P, _I, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _I64, _P]),
            "smla_topk": (_I, [PP, _P, _I64, _P, _P, _I, _I, _P, _P, ctypes.c_size_t, _P]),
            "smla_topk_workspace_size": (ctypes.c_size_t, [PP, _I]),
            "smla_attend": (_I, [LP, PP, _P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _P, _P, _P, ctypes.c_size_t, _P]),
            "smla_attend_workspace_size": (ctypes.c_size_t, [LP, PP, _I]),
            "smla_decode": (_I, [LP, PP, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I,
                                 _I, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "smla_decode_static": (_I, [LP, PP, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I,
                                        _I, _I, _I, _P, _P, _P, _P]),
            "smla_prefill_chunk": (_I, [LP, PP, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I,
                                        _I, _I, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
            "smla_dcp_topk_merge": (_I, [_P, _I64, _I64, _P, _I, _I, _I, _P, _P, _P]),
            "smla_attend_hisparse": (_I, [LP, PP, _P, _I, _P, _P, _I64, _P, _P, _P, _P, _I, _P, _I, _I, _P, _P, _P]),
            "smla_lse_merge": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P]),
            "smla_selftest_wait": (_I, [_I64, _P]),
            "smla_get_last_error": (_I, [_P]),
            "smla_status_string": (ctypes.c_char_p, [_I]),
            "smla_version": (_I, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _check(code: int, where: str) -> None:
    if code != 0:
        raise SmlaError(code, where)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libsmla takes CUDA tensors only")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError("libsmla takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _expect(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")


def _need(t, dtype, name, numel=0, dims=None):
    """A tensor argument's dtype, rank and minimum element count (the kernels read or write that many
    elements through its pointer).  None passes: the argument is optional or checked by the library."""
    if t is None:
        return
    _expect(t, dtype, name)
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name}: expected {dims} dimensions, got shape {tuple(t.shape)}")
    if t.numel() < numel:
        raise ValueError(f"{name}: needs at least {numel} elements, got shape {tuple(t.shape)}")


def _need_geometry(block_table, seq_lens, query_start_loc, batch):
    """block_table [>= batch, bt_stride], seq_lens [>= batch] and query_start_loc [>= batch + 1], int32."""
    _need(block_table, torch.int32, "block_table", dims=2)
    if block_table.shape[0] < batch:
        raise ValueError(f"block_table: needs a row per sequence ({batch}), got shape {tuple(block_table.shape)}")
    _need(seq_lens, torch.int32, "seq_lens", batch)
    _need(query_start_loc, torch.int32, "query_start_loc", batch + 1)


def _need_step(layout, params, pool, q, q_pe, q_idx, w, out, lse, topk_idx_out):
    """The per-query-token arrays of a fused step with T = q.shape[0] query tokens."""
    T, H, HI = q.shape[0], params.n_heads, params.n_idx_heads
    _need(pool, torch.uint8, "pool", layout.pool_bytes)
    _need(q, torch.bfloat16, "q", T * H * layout.d_latent)
    _need(q_pe, torch.bfloat16, "q_pe", T * H * layout.d_rope)
    _need(q_idx, torch.uint8, "q_idx", T * HI * layout.d_index)
    _need(w, torch.float32, "w", T * HI)
    _need(out, torch.bfloat16, "out", T * H * layout.d_latent)
    _need(lse, torch.float32, "lse", T * H)
    _need(topk_idx_out, torch.int32, "topk_idx_out", T * params.top_k)


def _need_new_tokens(layout, n, latent, rope, idx_k, idx_scale, slot_mapping, what="new"):
    """The n new tokens a step stores: latent, rope, indexer key and scale, slot per token."""
    _need(slot_mapping, torch.int64, "slot_mapping", n)
    _need(latent, torch.bfloat16, f"{what}_latent", n * layout.d_latent)
    _need(rope, torch.bfloat16, f"{what}_rope", n * layout.d_rope)
    _need(idx_k, torch.uint8, f"{what}_idx_k", n * layout.key_bytes)
    _need(idx_scale, torch.float32, f"{what}_idx_scale", n)


def version() -> int:
    return lib().smla_version()


def status_string(code: int) -> str:
    return lib().smla_status_string(code).decode()


def layout_init(block_size, n_layers, d_latent, d_rope, quant_tile, d_index, num_blocks, key_format="e4m3") -> Layout:
    """smla_layout_init (E4M3 indexer keys) or, with key_format="e2m1", smla_layout_init_keys (packed FP4 keys)."""
    lay = Layout()
    if key_format == "e4m3":
        _check(lib().smla_layout_init(ctypes.byref(lay), block_size, n_layers, d_latent, d_rope, quant_tile, d_index,
                                      num_blocks), "smla_layout_init")
    else:
        if key_format not in KEY_FORMATS:
            raise ValueError(f"unknown indexer key format {key_format!r}")
        _check(lib().smla_layout_init_keys(ctypes.byref(lay), block_size, n_layers, d_latent, d_rope, quant_tile,
                                           d_index, KEY_FORMATS[key_format], num_blocks), "smla_layout_init_keys")
    return lay


def make_params(n_heads, n_idx_heads, top_k, softmax_scale) -> Params:
    return Params(n_heads, n_idx_heads, top_k, softmax_scale)


def workspace_size(layout: Layout, params: Params, n_tokens: int, max_ctx: int) -> int:
    return int(lib().smla_workspace_size(ctypes.byref(layout), ctypes.byref(params), n_tokens, max_ctx))


def kvpack_store(layout, pool, layer, latent, rope, idx_k, idx_scale, slot_mapping, stream=None):
    _expect(slot_mapping, torch.int64, "slot_mapping")
    n = slot_mapping.numel()
    _need(pool, torch.uint8, "pool", layout.pool_bytes)
    _need(latent, torch.bfloat16, "latent", n * layout.d_latent)
    _need(rope, torch.bfloat16, "rope", n * layout.d_rope)
    _need(idx_k, torch.uint8, "idx_k", n * layout.key_bytes)
    _need(idx_scale, torch.float32, "idx_scale", n)
    _check(lib().kvpack_store(ctypes.byref(layout), _ptr(pool), layer, _ptr(latent), _ptr(rope), _ptr(idx_k),
                              _ptr(idx_scale), _ptr(slot_mapping), n, _stream(stream)), "kvpack_store")


def smla_index_scores(layout, params, pool, layer, q_idx, w, block_table, seq_lens, query_start_loc, max_q,
                      max_ctx, scores, stream=None):
    n_tokens = q_idx.shape[0]
    _need(pool, torch.uint8, "pool", layout.pool_bytes)
    _need(q_idx, torch.uint8, "q_idx", n_tokens * params.n_idx_heads * layout.d_index)
    _need(w, torch.float32, "w", n_tokens * params.n_idx_heads)
    _need_geometry(block_table, seq_lens, query_start_loc, seq_lens.numel())
    _need(scores, torch.float32, "scores", dims=2)
    if scores.shape[0] < n_tokens:
        raise ValueError(f"scores: needs a row per query token ({n_tokens}), got shape {tuple(scores.shape)}")
    _check(lib().smla_index_scores(ctypes.byref(layout), ctypes.byref(params), _ptr(pool), layer, _ptr(q_idx),
                                   _ptr(w), _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                   _ptr(query_start_loc), seq_lens.numel(), n_tokens, max_q, max_ctx, _ptr(scores),
                                   scores.stride(0), _stream(stream)), "smla_index_scores")


def topk_workspace_size(params, n_tokens) -> int:
    return int(lib().smla_topk_workspace_size(ctypes.byref(params), n_tokens))


def smla_topk(params, scores, seq_lens, query_start_loc, topk_idx, stream=None, workspace=None):
    """Exact top-k per row.  `workspace` (uint8 device tensor of at least topk_workspace_size(...)
    bytes, optional) lets a small batch of long rows split each row over CTAs."""
    _need(topk_idx, torch.int32, "topk_idx", dims=2)
    rows = topk_idx.shape[0]
    if topk_idx.shape[1] != params.top_k:
        raise ValueError(f"topk_idx: rows of top_k = {params.top_k} entries expected, got shape {tuple(topk_idx.shape)}")
    _need(scores, torch.float32, "scores", dims=2)
    if scores.shape[0] < rows:
        raise ValueError(f"scores: needs a row per top-k row ({rows}), got shape {tuple(scores.shape)}")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(query_start_loc, torch.int32, "query_start_loc", seq_lens.numel() + 1)
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().smla_topk(ctypes.byref(params), _ptr(scores), scores.stride(0), _ptr(seq_lens),
                           _ptr(query_start_loc), seq_lens.numel(), topk_idx.shape[0], _ptr(topk_idx),
                           _ptr(workspace), ws_bytes, _stream(stream)), "smla_topk")


def attend_workspace_size(layout, params, n_tokens) -> int:
    return int(lib().smla_attend_workspace_size(ctypes.byref(layout), ctypes.byref(params), n_tokens))


def _need_attend(layout, params, pool, q, q_pe, topk_idx, block_table, query_start_loc, out, lse):
    """Arrays of smla_attend with T = q.shape[0] query tokens and B = query_start_loc.numel() - 1 sequences."""
    T, H = q.shape[0], params.n_heads
    _need(pool, torch.uint8, "pool", layout.pool_bytes)
    _need(q, torch.bfloat16, "q", T * H * layout.d_latent)
    _need(q_pe, torch.bfloat16, "q_pe", T * H * layout.d_rope)
    _need(topk_idx, torch.int32, "topk_idx", T * params.top_k)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    batch = query_start_loc.numel() - 1
    _need(block_table, torch.int32, "block_table", dims=2)
    if block_table.shape[0] < batch:
        raise ValueError(f"block_table: needs a row per sequence ({batch}), got shape {tuple(block_table.shape)}")
    _need(out, torch.bfloat16, "out", T * H * layout.d_latent)
    _need(lse, torch.float32, "lse", T * H)


def smla_attend(layout, params, pool, layer, q, q_pe, topk_idx, block_table, query_start_loc, out, lse,
                stream=None, workspace=None):
    """Latent attention over the selected positions.  `workspace` (uint8 device tensor of at least
    attend_workspace_size(...) bytes, optional) lets a small batch split each token over CTAs."""
    _need_attend(layout, params, pool, q, q_pe, topk_idx, block_table, query_start_loc, out, lse)
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().smla_attend(ctypes.byref(layout), ctypes.byref(params), _ptr(pool), layer, _ptr(q), _ptr(q_pe),
                             _ptr(topk_idx), _ptr(block_table), block_table.shape[1], _ptr(query_start_loc),
                             query_start_loc.numel() - 1, q.shape[0], _ptr(out), _ptr(lse), _ptr(workspace),
                             ws_bytes, _stream(stream)),
           "smla_attend")


def smla_attend_hisparse(layout, params, pool, layer, host_records, host_block_map, q, q_pe, topk_idx, block_table,
                         query_start_loc, out, lse, stream=None):
    """smla_attend with the records of mapped blocks read from a pinned host buffer (host_records, uint8)."""
    _need_attend(layout, params, pool, q, q_pe, topk_idx, block_table, query_start_loc, out, lse)
    _need(host_block_map, torch.int32, "host_block_map", layout.num_blocks)
    _expect(host_records, torch.uint8, "host_records")
    if host_records.is_cuda or not host_records.is_pinned():
        raise ValueError("host_records must be pinned host memory")
    if not host_block_map.is_cuda:
        raise ValueError("host_block_map must be a CUDA tensor")
    rec_bytes = layout.n_layers * layout.block_size * layout.rec_stride
    n_host = host_records.numel() // rec_bytes
    _check(lib().smla_attend_hisparse(ctypes.byref(layout), ctypes.byref(params), _ptr(pool), layer,
                                      ctypes.c_void_p(host_records.data_ptr()), _ptr(host_block_map), n_host, _ptr(q),
                                      _ptr(q_pe), _ptr(topk_idx), _ptr(block_table), block_table.shape[1],
                                      _ptr(query_start_loc), query_start_loc.numel() - 1, q.shape[0], _ptr(out),
                                      _ptr(lse), _stream(stream)), "smla_attend_hisparse")


def smla_decode(layout, params, pool, layer, new_latent, new_rope, new_idx_k, new_idx_scale, slot_mapping, q, q_pe,
                q_idx, w, block_table, seq_lens, query_start_loc, max_q, max_ctx, out, lse, workspace,
                topk_idx_out=None, stream=None):
    T = q.shape[0]
    _need_step(layout, params, pool, q, q_pe, q_idx, w, out, lse, topk_idx_out)
    _need_geometry(block_table, seq_lens, query_start_loc, seq_lens.numel())
    if slot_mapping is not None:
        _need_new_tokens(layout, T, new_latent, new_rope, new_idx_k, new_idx_scale, slot_mapping)
    _need(workspace, torch.uint8, "workspace")
    _check(lib().smla_decode(ctypes.byref(layout), ctypes.byref(params), _ptr(pool), layer, _ptr(new_latent),
                             _ptr(new_rope), _ptr(new_idx_k), _ptr(new_idx_scale), _ptr(slot_mapping), _ptr(q),
                             _ptr(q_pe), _ptr(q_idx), _ptr(w), _ptr(block_table), block_table.shape[1],
                             _ptr(seq_lens), _ptr(query_start_loc), seq_lens.numel(), q.shape[0], max_q, max_ctx,
                             _ptr(out), _ptr(lse), _ptr(topk_idx_out), _ptr(workspace), workspace.numel(),
                             _stream(stream)), "smla_decode")


def smla_decode_static(layout, params, pool, layer, new_latent, new_rope, new_idx_k, new_idx_scale, slot_mapping,
                       q, q_pe, q_idx, w, block_table, seq_lens, query_start_loc, max_q, max_ctx, out, lse,
                       topk_idx_out=None, stream=None):
    """smla_decode without a workspace argument, for callers that cannot allocate device memory.

    The scores and top-k scratch live in the library's static 64 MiB device
    array; calls share it, so calls that overlap on the GPU race on it.
    """
    T = q.shape[0]
    _need_step(layout, params, pool, q, q_pe, q_idx, w, out, lse, topk_idx_out)
    _need_geometry(block_table, seq_lens, query_start_loc, seq_lens.numel())
    if slot_mapping is not None:
        _need_new_tokens(layout, T, new_latent, new_rope, new_idx_k, new_idx_scale, slot_mapping)
    _check(lib().smla_decode_static(ctypes.byref(layout), ctypes.byref(params), _ptr(pool), layer, _ptr(new_latent),
                                    _ptr(new_rope), _ptr(new_idx_k), _ptr(new_idx_scale), _ptr(slot_mapping), _ptr(q),
                                    _ptr(q_pe), _ptr(q_idx), _ptr(w), _ptr(block_table), block_table.shape[1],
                                    _ptr(seq_lens), _ptr(query_start_loc), seq_lens.numel(), q.shape[0], max_q,
                                    max_ctx, _ptr(out), _ptr(lse), _ptr(topk_idx_out), _stream(stream)),
           "smla_decode_static")


def smla_prefill_chunk(layout, params, pool, layer, chunk_latent, chunk_rope, chunk_idx_k, chunk_idx_scale,
                       slot_mapping, q, q_pe, q_idx, w, block_table, seq_lens, query_start_loc, chunk_len, max_ctx,
                       out, lse, workspace, topk_idx_out=None, stream=None):
    """A prefill chunk per sequence (its keys stored first), causal within the chunk."""
    T = q.shape[0]
    _need_step(layout, params, pool, q, q_pe, q_idx, w, out, lse, topk_idx_out)
    _need_geometry(block_table, seq_lens, query_start_loc, seq_lens.numel())
    _need_new_tokens(layout, T, chunk_latent, chunk_rope, chunk_idx_k, chunk_idx_scale, slot_mapping, "chunk")
    _need(workspace, torch.uint8, "workspace")
    _check(lib().smla_prefill_chunk(ctypes.byref(layout), ctypes.byref(params), _ptr(pool), layer, _ptr(chunk_latent),
                                    _ptr(chunk_rope), _ptr(chunk_idx_k), _ptr(chunk_idx_scale), _ptr(slot_mapping),
                                    _ptr(q), _ptr(q_pe), _ptr(q_idx), _ptr(w), _ptr(block_table), block_table.shape[1],
                                    _ptr(seq_lens), _ptr(query_start_loc), seq_lens.numel(), q.shape[0], chunk_len,
                                    max_ctx, _ptr(out), _ptr(lse), _ptr(topk_idx_out), _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "smla_prefill_chunk")


def smla_dcp_topk_merge(shard_scores, shard_topk, shard_sel, merged=None, stream=None):
    """Candidate merge over token shards.  shard_scores [N, T, stride] fp32, shard_topk / shard_sel [N, T, k] int32."""
    _need(shard_topk, torch.int32, "shard_topk", dims=3)
    n, t, k = shard_topk.shape
    _need(shard_scores, torch.float32, "shard_scores", dims=3)
    if shard_scores.shape[0] < n or shard_scores.shape[1] < t:
        raise ValueError(f"shard_scores: needs [{n}, {t}, >= visible] for shard_topk {tuple(shard_topk.shape)}, "
                         f"got {tuple(shard_scores.shape)}")
    _need(shard_sel, torch.int32, "shard_sel", n * t * k)
    _need(merged, torch.int32, "merged", t * k)
    _check(lib().smla_dcp_topk_merge(_ptr(shard_scores), shard_scores.stride(0), shard_scores.stride(1),
                                     _ptr(shard_topk), n, t, k, _ptr(shard_sel), _ptr(merged), _stream(stream)),
           "smla_dcp_topk_merge")


def smla_lse_merge(parts_out, parts_lse, out, lse, stream=None):
    """LSE merge of partial outputs.  parts_out [N, T, H, D] bf16, parts_lse [N, T, H] fp32."""
    _need(parts_out, torch.bfloat16, "parts_out", dims=4)
    n, t, h, d = parts_out.shape
    _need(parts_lse, torch.float32, "parts_lse", n * t * h)
    _need(out, torch.bfloat16, "out", t * h * d)
    _need(lse, torch.float32, "lse", t * h)
    _check(lib().smla_lse_merge(_ptr(parts_out), _ptr(parts_lse), n, t, h, d, _ptr(out), _ptr(lse), _stream(stream)),
           "smla_lse_merge")


def smla_selftest_wait(limit_ns, stream=None):
    """Launch the bounded-wait self-check (one wait never completes; it gives up after limit_ns)."""
    _check(lib().smla_selftest_wait(int(limit_ns), _stream(stream)), "smla_selftest_wait")


def smla_get_last_error(stream=None) -> int:
    return int(lib().smla_get_last_error(_stream(stream)))
