"""The Python binding's argument checks, on CPU.

Every entry point is called the way the GPU tests and the bench call it, with
CPU tensors of the right shapes: the checks must let those through, so that
the call stops only at "CUDA tensors only" (no kernel runs here).  A buffer
one element short, a wrong dtype or a missing row must be refused before
that, so that it can never reach a kernel that would overrun it.
"""
import pytest
import torch

import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300 import build_lib
from paged_sparse_mla_gb300.workloads import make_config

CUDA_ONLY = "CUDA tensors only"


@pytest.fixture(scope="module")
def env():
    build_lib.build()
    smla.lib()
    wl = make_config(1)
    d = wl.dims
    lay = smla.layout_init(d.block_size, d.n_layers, d.d_latent, d.d_rope, d.quant_tile, d.d_index, wl.num_blocks)
    prm = smla.make_params(d.n_heads, d.n_idx_heads, d.top_k, d.softmax_scale)
    T = wl.n_tokens
    bufs = dict(
        pool=torch.zeros(lay.pool_bytes, dtype=torch.uint8),
        out=torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16),
        lse=torch.empty((T, d.n_heads), dtype=torch.float32),
        topk=torch.empty((T, d.top_k), dtype=torch.int32),
        scores=torch.empty((T, (wl.max_ctx + 3) // 4 * 4), dtype=torch.float32),
        ws=torch.empty(smla.workspace_size(lay, prm, T, wl.max_ctx), dtype=torch.uint8),
    )
    return wl, lay, prm, bufs


def _short(t):
    """The same tensor one element short (flattened)."""
    return t.reshape(-1)[:-1]


def _decode(wl, lay, prm, b, **over):
    a = dict(new_latent=wl.new_latent, new_rope=wl.new_rope, new_idx_k=wl.new_idx_k, new_idx_scale=wl.new_idx_s,
             slot_mapping=wl.slot_mapping, q=wl.q, q_pe=wl.q_pe, q_idx=wl.q_idx, w=wl.w,
             block_table=wl.block_table, seq_lens=wl.seq_lens, query_start_loc=wl.query_start_loc,
             out=b["out"], lse=b["lse"], workspace=b["ws"], topk_idx_out=b["topk"], pool=b["pool"])
    a.update(over)
    smla.smla_decode(lay, prm, a["pool"], 0, a["new_latent"], a["new_rope"], a["new_idx_k"], a["new_idx_scale"],
                     a["slot_mapping"], a["q"], a["q_pe"], a["q_idx"], a["w"], a["block_table"], a["seq_lens"],
                     a["query_start_loc"], wl.max_q, wl.max_ctx, a["out"], a["lse"], a["workspace"],
                     topk_idx_out=a["topk_idx_out"])


def test_well_formed_calls_reach_the_device_check(env):
    wl, lay, prm, b = env
    s = wl.cached_slots
    calls = [
        lambda: smla.kvpack_store(lay, b["pool"], 0, wl.slot_latent[s].contiguous(), wl.slot_rope[s].contiguous(),
                                  wl.slot_idx_k[s].contiguous(), wl.slot_idx_s[s].contiguous(), s),
        lambda: smla.smla_index_scores(lay, prm, b["pool"], 0, wl.q_idx, wl.w, wl.block_table, wl.seq_lens,
                                       wl.query_start_loc, wl.max_q, wl.max_ctx, b["scores"]),
        lambda: smla.smla_topk(prm, b["scores"], wl.seq_lens, wl.query_start_loc, b["topk"]),
        lambda: smla.smla_attend(lay, prm, b["pool"], 0, wl.q, wl.q_pe, b["topk"], wl.block_table,
                                 wl.query_start_loc, b["out"], b["lse"]),
        lambda: _decode(wl, lay, prm, b),
        lambda: _decode(wl, lay, prm, b, slot_mapping=None),
        lambda: smla.smla_decode_static(lay, prm, b["pool"], 0, wl.new_latent, wl.new_rope, wl.new_idx_k,
                                        wl.new_idx_s, wl.slot_mapping, wl.q, wl.q_pe, wl.q_idx, wl.w,
                                        wl.block_table, wl.seq_lens, wl.query_start_loc, wl.max_q, wl.max_ctx,
                                        b["out"], b["lse"], topk_idx_out=b["topk"]),
        lambda: smla.smla_prefill_chunk(lay, prm, b["pool"], 0, wl.new_latent, wl.new_rope, wl.new_idx_k,
                                        wl.new_idx_s, wl.slot_mapping, wl.q, wl.q_pe, wl.q_idx, wl.w,
                                        wl.block_table, wl.seq_lens, wl.query_start_loc, wl.max_q, wl.max_ctx,
                                        b["out"], b["lse"], b["ws"], topk_idx_out=b["topk"]),
        lambda: smla.smla_dcp_topk_merge(torch.zeros((2, 3, 40)), torch.zeros((2, 3, 8), dtype=torch.int32),
                                         torch.zeros((2, 3, 8), dtype=torch.int32),
                                         torch.zeros((3, 8), dtype=torch.int32)),
        lambda: smla.smla_lse_merge(torch.zeros((2, 3, 4, 16), dtype=torch.bfloat16), torch.zeros((2, 3, 4)),
                                    torch.zeros((3, 4, 16), dtype=torch.bfloat16), torch.zeros((3, 4))),
    ]
    for i, call in enumerate(calls):
        with pytest.raises(ValueError, match=CUDA_ONLY):
            call()


@pytest.mark.parametrize("arg", ["out", "lse", "topk_idx_out", "q", "q_pe", "q_idx", "w", "new_latent", "new_rope",
                                 "new_idx_k", "new_idx_scale", "slot_mapping", "pool", "query_start_loc"])
def test_fused_step_refuses_a_short_buffer(env, arg):
    wl, lay, prm, b = env
    full = dict(out=b["out"], lse=b["lse"], topk_idx_out=b["topk"], pool=b["pool"], q=wl.q, q_pe=wl.q_pe,
                q_idx=wl.q_idx, w=wl.w, new_latent=wl.new_latent, new_rope=wl.new_rope, new_idx_k=wl.new_idx_k,
                new_idx_scale=wl.new_idx_s, slot_mapping=wl.slot_mapping, query_start_loc=wl.query_start_loc)
    with pytest.raises(ValueError, match="needs at least"):
        _decode(wl, lay, prm, b, **{arg: _short(full[arg])})


def test_stage_calls_refuse_short_or_mistyped_buffers(env):
    wl, lay, prm, b = env
    with pytest.raises(ValueError, match="needs a row per query token"):
        smla.smla_index_scores(lay, prm, b["pool"], 0, wl.q_idx, wl.w, wl.block_table, wl.seq_lens,
                               wl.query_start_loc, wl.max_q, wl.max_ctx, b["scores"][:1])
    with pytest.raises(ValueError, match="top_k"):
        smla.smla_topk(prm, b["scores"], wl.seq_lens, wl.query_start_loc, b["topk"][:, :-1].contiguous())
    with pytest.raises(TypeError):
        smla.smla_topk(prm, b["scores"], wl.seq_lens.long(), wl.query_start_loc, b["topk"])
    with pytest.raises(ValueError, match="needs a row per sequence"):
        smla.smla_attend(lay, prm, b["pool"], 0, wl.q, wl.q_pe, b["topk"], wl.block_table[:1], wl.query_start_loc,
                         b["out"], b["lse"])
    with pytest.raises(ValueError, match="needs at least"):
        smla.smla_attend(lay, prm, b["pool"], 0, wl.q, wl.q_pe, _short(b["topk"]), wl.block_table,
                         wl.query_start_loc, b["out"], b["lse"])
    with pytest.raises(ValueError, match="needs at least"):
        smla.kvpack_store(lay, b["pool"], 0, _short(wl.new_latent), wl.new_rope, wl.new_idx_k, wl.new_idx_s,
                          wl.slot_mapping)
    with pytest.raises(ValueError, match="needs at least"):
        smla.smla_lse_merge(torch.zeros((2, 3, 4, 16), dtype=torch.bfloat16), torch.zeros((2, 3, 4)),
                            torch.zeros((3, 4, 16), dtype=torch.bfloat16), torch.zeros((3, 3)))
    with pytest.raises(ValueError, match="shard_scores"):
        smla.smla_dcp_topk_merge(torch.zeros((2, 2, 40)), torch.zeros((2, 3, 8), dtype=torch.int32),
                                 torch.zeros((2, 3, 8), dtype=torch.int32))
