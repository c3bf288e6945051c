"""smla_decode_static -- the fused step for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace: their device memory
belongs to a serving engine's allocator that reserves all free HBM for the KV
block pool, or they run on a host runtime without a device-allocation hook.
smla_decode_static serves them from a 64 MiB static array inside the library.
These tests call it through the C ABI twice in a row (the array keeps the
previous call's contents) and compare with smla_decode, which uses a caller
workspace; they also check that a context too long for the array is refused
before anything runs.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from paged_sparse_mla_gb300.workloads import make_config, build_workload, FULL
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


def _run_static(wl, pool, lay, prm):
    d = wl.dims
    T = wl.n_tokens
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    topk = torch.empty((T, prm.top_k), dtype=torch.int32, device="cuda")
    G.smla.smla_decode_static(lay, prm, pool, 0, wl.new_latent, wl.new_rope, wl.new_idx_k, wl.new_idx_s,
                              wl.slot_mapping, wl.q, wl.q_pe, wl.q_idx, wl.w, wl.block_table, wl.seq_lens,
                              wl.query_start_loc, wl.max_q, wl.max_ctx, out, lse, topk_idx_out=topk)
    err = G.smla.smla_get_last_error()
    return dict(topk=topk.cpu().numpy(), out=out.float().cpu().numpy(), lse=lse.cpu().numpy(), err=err)


@pytest.mark.parametrize("make", [lambda: make_config(1), lambda: make_config(2, scale=0.1),
                                  lambda: make_config(3, scale=0.02)], ids=["tiny", "decode-b32", "agentic-mtp"])
def test_static_scratch_matches_workspace_entry_point_twice(make):
    wl = G.cuda_wl(make())
    lay, prm = G.gpu_layout(wl), G.gpu_params(wl)
    ref = G.run_decode(wl, G.gpu_pool(wl, lay), lay, prm)
    assert ref["err"] == 0
    pool = G.gpu_pool(wl, lay)
    for call in range(2):
        got = _run_static(wl, pool, lay, prm)
        assert got["err"] == 0, f"call {call}"
        assert np.array_equal(got["topk"], ref["topk"]), f"call {call}: top-k differs"
        G.assert_attention_close(got["out"], got["lse"], ref["out"].astype(np.float64),
                                 ref["lse"].astype(np.float64), f"call {call}")


def test_static_scratch_refuses_contexts_beyond_its_size():
    wl = G.cuda_wl(build_workload("one", FULL, [100], [1], seed=7))
    lay, prm = G.gpu_layout(wl), G.gpu_params(wl)
    pool = G.gpu_pool(wl, lay)
    d = wl.dims
    out = torch.empty((1, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, d.n_heads), dtype=torch.float32, device="cuda")
    huge = 20_000_000                                   # 80 MB of scores for one token > 64 MiB
    bt = torch.zeros((1, huge // d.block_size + 1), dtype=torch.int32, device="cuda")
    with pytest.raises(G.smla.SmlaError) as e:
        G.smla.smla_decode_static(lay, prm, pool, 0, wl.new_latent, wl.new_rope, wl.new_idx_k, wl.new_idx_s,
                                  wl.slot_mapping, wl.q, wl.q_pe, wl.q_idx, wl.w, bt, wl.seq_lens,
                                  wl.query_start_loc, 1, huge, out, lse)
    assert e.value.code == 6                            # SMLA_ERR_SCRATCH_LIMIT, nothing enqueued
    assert G.smla.smla_get_last_error() == 0
