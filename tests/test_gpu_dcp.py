"""GPU parity of the split-context (DCP-style) path: N token shards on one GPU.

Shard r holds the positions j = N*i + r of every sequence (round-robin), in its
own pool with its own block table.  Each shard runs smla_index_scores and
smla_topk over its positions; smla_dcp_topk_merge merges the candidates and
hands each shard its selected local positions; smla_attend runs per shard and
smla_lse_merge combines the partial outputs.  The global selection must equal
the oracle's unsharded top-k exactly, and out / lse the oracle's attention
within the attention tolerance.  The two merge kernels are also checked on
their own against oracle.dcp.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import dcp
import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300.workloads import FULL, TINY, build_workload, shard_pools
from tests.oracle_helpers import oracle_pool, oracle_step
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


def _make_shards(g, lay, pool, n_shards, seed):
    sh = shard_pools(g, lay, pool, n_shards, seed=seed)
    return [dict(lay=x["layout"], pool=x["pool"], bt=x["block_table"], seq_lens=x["seq_lens"], max_ctx=x["max_ctx"])
            for x in sh]


def _run_sharded(g, prm, shards):
    d = g.dims
    T, k, n = g.n_tokens, prm.top_k, len(shards)
    stride = max((s["max_ctx"] + 3) // 4 * 4 for s in shards)
    scores = torch.zeros((n, T, stride), dtype=torch.float32, device="cuda")
    topk = torch.empty((n, T, k), dtype=torch.int32, device="cuda")
    for r, s in enumerate(shards):
        smla.smla_index_scores(s["lay"], prm, s["pool"], 0, g.q_idx, g.w, s["bt"], s["seq_lens"], g.query_start_loc,
                               1, s["max_ctx"], scores[r])
        smla.smla_topk(prm, scores[r], s["seq_lens"], g.query_start_loc, topk[r])
    sel = torch.empty((n, T, k), dtype=torch.int32, device="cuda")
    merged = torch.empty((T, k), dtype=torch.int32, device="cuda")
    smla.smla_dcp_topk_merge(scores, topk, sel, merged)
    parts = torch.empty((n, T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    parts_lse = torch.empty((n, T, d.n_heads), dtype=torch.float32, device="cuda")
    for r, s in enumerate(shards):
        smla.smla_attend(s["lay"], prm, s["pool"], 0, g.q, g.q_pe, sel[r], s["bt"], g.query_start_loc, parts[r],
                         parts_lse[r])
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    smla.smla_lse_merge(parts, parts_lse, out, lse)
    err = smla.smla_get_last_error()
    return dict(merged=merged.cpu().numpy(), sel=sel.cpu().numpy(), out=out.float().cpu().numpy(),
                lse=lse.cpu().numpy(), err=err)


CASES = {
    "full-b5": lambda: build_workload("dcpf", FULL, [5000, 3001, 2049, 700, 1], [1, 1, 1, 1, 1], seed=71,
                                      slack_blocks=2),
    "tiny-b4": lambda: build_workload("dcpt", TINY, [200, 97, 64, 3], [1, 1, 1, 1], seed=72, slack_blocks=2),
}


@pytest.mark.parametrize("n_shards", [2, 4])
@pytest.mark.parametrize("name", list(CASES))
def test_sharded_decode_matches_oracle(name, n_shards):
    wl = CASES[name]()
    ref = oracle_step(wl, oracle_pool(wl))
    g = G.cuda_wl(CASES[name]())
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    whole = G.run_decode(g, pool, lay, prm)            # stores this step's tokens, unsharded result
    assert whole["err"] == 0
    res = _run_sharded(g, prm, _make_shards(g, lay, pool, n_shards, seed=5 + n_shards))
    assert res["err"] == 0
    for t in range(g.n_tokens):
        assert np.array_equal(res["merged"][t], ref[t]["topk"]), f"{name} N={n_shards}: global selection row {t}"
        sel = res["merged"][t]
        sel = sel[sel >= 0]
        for r in range(n_shards):
            loc = res["sel"][r, t]
            loc = loc[loc >= 0]
            assert np.array_equal(loc, np.sort(sel[sel % n_shards == r] // n_shards))
    out_ref = np.stack([ref[t]["out"] for t in range(g.n_tokens)])
    lse_ref = np.stack([ref[t]["lse"] for t in range(g.n_tokens)])
    G.assert_attention_close(res["out"], res["lse"], out_ref, lse_ref, f"{name} N={n_shards}")
    G.assert_attention_close(res["out"], res["lse"], whole["out"].astype(np.float64),
                             whole["lse"].astype(np.float64), f"{name} N={n_shards} vs unsharded")


@pytest.mark.parametrize("n_shards,k,n", [(2, 64, 300), (4, 128, 1000), (8, 2048, 20000), (3, 16, 5)])
def test_topk_merge_kernel_matches_oracle(n_shards, k, n):
    rng = np.random.default_rng(n_shards * 7 + k)
    T = 6
    full = rng.integers(-4, 5, size=(T, n)).astype(np.float32) * np.float32(0.25)   # heavy ties
    stride = (n + n_shards - 1) // n_shards + 3
    scores = np.zeros((n_shards, T, stride), dtype=np.float32)
    topk = np.full((n_shards, T, k), -1, dtype=np.int32)
    for r in range(n_shards):
        for t in range(T):
            row = full[t, r::n_shards]
            scores[r, t, :row.size] = row
            topk[r, t] = oracle.topk_select(row, k)
    sel = torch.empty((n_shards, T, k), dtype=torch.int32, device="cuda")
    merged = torch.empty((T, k), dtype=torch.int32, device="cuda")
    smla.smla_dcp_topk_merge(torch.as_tensor(scores, device="cuda"), torch.as_tensor(topk, device="cuda"), sel, merged)
    for t in range(T):
        glob, per = dcp.topk_merge([scores[r, t] for r in range(n_shards)], [topk[r, t] for r in range(n_shards)],
                                   n_shards, k)
        assert np.array_equal(merged[t].cpu().numpy(), glob)
        assert np.array_equal(glob, oracle.topk_select(full[t], k))
        assert np.array_equal(sel[:, t].cpu().numpy(), per)


@pytest.mark.parametrize("n_shards", [1, 2, 5])
def test_lse_merge_kernel_matches_oracle(n_shards):
    rng = np.random.default_rng(40 + n_shards)
    T, H, D = 7, 64, 512
    parts = torch.randn((n_shards, T, H, D), dtype=torch.float32).to(torch.bfloat16)
    lse = torch.as_tensor(rng.normal(scale=3.0, size=(n_shards, T, H)).astype(np.float32))
    lse[0, 0, :] = float("-inf")                  # an empty shard for one token
    if n_shards > 1:
        lse[:, 1, 3] = float("-inf")              # every shard empty for one head
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    lse_out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    smla.smla_lse_merge(parts.cuda(), lse.cuda(), out, lse_out)
    po = parts.float().numpy().astype(np.float64)
    pl = lse.numpy().astype(np.float64)
    for t in range(T):
        ro, rl = dcp.lse_merge(po[:, t], pl[:, t])
        go = out[t].float().cpu().numpy()
        gl = lse_out[t].cpu().numpy()
        assert np.array_equal(np.isfinite(gl), np.isfinite(rl))
        fin = np.isfinite(rl)
        assert np.abs(gl[fin] - rl[fin]).max(initial=0) <= 1e-5
        # bf16 output of an fp32 combination: within half a bf16 unit (plus fp32 rounding) of the value
        assert np.all(np.abs(go - ro) <= np.abs(ro) * 2.0 ** -8 + 1e-6)
