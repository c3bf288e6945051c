"""Helpers for the GPU parity tests: run the CUDA library on a generated workload."""
import numpy as np
import torch

import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300 import build_lib

# Attention tolerance (fp32 oracle vs bf16 output of the bf16 tensor-core path).
MAX_ERR = 2e-2
MEAN_ERR = 2e-3


def ensure_built():
    build_lib.build()
    return smla.lib()


def gpu_layout(wl):
    d = wl.dims
    return smla.layout_init(d.block_size, d.n_layers, d.d_latent, d.d_rope, d.quant_tile, d.d_index, wl.num_blocks,
                            d.key_format)


def gpu_params(wl, top_k=None):
    d = wl.dims
    return smla.make_params(d.n_heads, d.n_idx_heads, d.top_k if top_k is None else top_k, d.softmax_scale)


def gpu_pool(wl, layout, layer=0, chunk=1 << 20):
    """Pool holding the cached context, written by the CUDA store."""
    pool = torch.zeros(layout.pool_bytes, dtype=torch.uint8, device="cuda")
    s = wl.cached_slots.cuda()
    for c0 in range(0, s.numel(), chunk):
        sl = s[c0:c0 + chunk].contiguous()
        smla.kvpack_store(layout, pool, layer, wl.slot_latent[sl].contiguous(), wl.slot_rope[sl].contiguous(),
                          wl.slot_idx_k[sl].contiguous(), wl.slot_idx_s[sl].contiguous(), sl)
    return pool


def cuda_wl(wl):
    """Move every tensor of a workload to the GPU."""
    for name, val in list(vars(wl).items()):
        if isinstance(val, torch.Tensor):
            setattr(wl, name, val.cuda())
    return wl


def run_stages(wl, pool, layout, params, layer=0, store=True, split=True):
    """store -> index_scores -> topk -> attend as separate calls; returns host arrays.  With `split`
    the attention gets the scratch the fused step gives it (small batches split tokens over CTAs)."""
    d = wl.dims
    T = wl.n_tokens
    if store:
        smla.kvpack_store(layout, pool, layer, wl.new_latent, wl.new_rope, wl.new_idx_k, wl.new_idx_s,
                          wl.slot_mapping)
    stride = (wl.max_ctx + 3) // 4 * 4
    scores = torch.full((T, stride), float("nan"), dtype=torch.float32, device="cuda")
    smla.smla_index_scores(layout, params, pool, layer, wl.q_idx, wl.w, wl.block_table, wl.seq_lens,
                           wl.query_start_loc, wl.max_q, wl.max_ctx, scores)
    topk = torch.empty((T, params.top_k), dtype=torch.int32, device="cuda")
    tbytes = smla.topk_workspace_size(params, T) if split else 0
    tws = torch.empty(tbytes, dtype=torch.uint8, device="cuda") if tbytes else None
    smla.smla_topk(params, scores, wl.seq_lens, wl.query_start_loc, topk, workspace=tws)
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    nbytes = smla.attend_workspace_size(layout, params, T) if split else 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    smla.smla_attend(layout, params, pool, layer, wl.q, wl.q_pe, topk, wl.block_table, wl.query_start_loc, out, lse,
                     workspace=ws)
    err = smla.smla_get_last_error()
    return dict(scores=scores.cpu().numpy(), topk=topk.cpu().numpy(), out=out.float().cpu().numpy(),
                lse=lse.cpu().numpy(), err=err)


def run_decode(wl, pool, layout, params, layer=0, store=True):
    """The fused step through smla_decode."""
    d = wl.dims
    T = wl.n_tokens
    ws = torch.empty(smla.workspace_size(layout, params, T, wl.max_ctx), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    topk = torch.empty((T, params.top_k), dtype=torch.int32, device="cuda")
    smla.smla_decode(layout, params, pool, layer, wl.new_latent, wl.new_rope, wl.new_idx_k, wl.new_idx_s,
                     wl.slot_mapping if store else None, wl.q, wl.q_pe, wl.q_idx, wl.w, wl.block_table, wl.seq_lens,
                     wl.query_start_loc, wl.max_q, wl.max_ctx, out, lse, ws, topk_idx_out=topk)
    err = smla.smla_get_last_error()
    return dict(topk=topk.cpu().numpy(), out=out.float().cpu().numpy(), lse=lse.cpu().numpy(), err=err)


def canon(x):
    """fp32 bit patterns with -0 folded onto +0 (scores compare as values)."""
    return (np.asarray(x, dtype=np.float32) + np.float32(0)).view(np.uint32)


def assert_attention_close(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    e = np.abs(out_gpu.astype(np.float64) - out_ref)
    assert e.max() <= MAX_ERR and e.mean() <= MEAN_ERR, f"{what} out max {e.max():.3e} mean {e.mean():.3e}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse_gpu)), what
    el = np.abs(lse_gpu.astype(np.float64)[fin] - lse_ref[fin])
    if el.size:
        assert el.max() <= MAX_ERR and el.mean() <= MEAN_ERR, f"{what} lse max {el.max():.3e} mean {el.mean():.3e}"
