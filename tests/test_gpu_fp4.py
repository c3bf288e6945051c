"""GPU parity of the FP4 (E2M1) indexer-key path against the CPU oracle, through the C ABI.

The pool holds each indexer key as 128 packed E2M1 codes (64 bytes); the CUDA
indexer unpacks them in the copy into shared memory and multiplies them, as
E2M1, with the E4M3 queries on the tensor cores.  Key values are multiples of
0.5 up to 6 and queries integers up to 8, so every partial sum is exact in fp32:
scores compare bit for bit, top-k exactly, attention within the stated
tolerance.  Also: the same key values stored as E4M3 give bit-identical scores,
and the full-size shapes hold on sampled rows plus the exact-top-k property on
every row.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300.workloads import FULL, build_workload, make_config
from dataclasses import replace
from tests.oracle_helpers import bits, layout_of, npy, oracle_pool, oracle_step, sequence_slots
from tests import gpu_helpers as G
from tests.topk_properties import assert_topk_exact

pytestmark = pytest.mark.gpu

FP4 = replace(FULL, key_format="e2m1")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


CASES = {
    "decode-b32-scaled": lambda: make_config(2, scale=0.1, key_format="e2m1"),
    "agentic-mtp-scaled": lambda: make_config(3, scale=0.02, key_format="e2m1"),
    "longctx-scaled": lambda: make_config(4, scale=0.004, key_format="e2m1"),
    "prefill-scaled": lambda: make_config(5, scale=1 / 64, key_format="e2m1"),
    "short-contexts": lambda: build_workload("shortf4", FP4, [1, 5, 2048, 2049, 2177, 4100], [1, 1, 1, 4, 2, 3],
                                             seed=52, slack_blocks=5),
    "pow2-key-scales": lambda: build_workload("pow2f4", FP4, [3000, 700], [2, 1], seed=53,
                                              idx_scale=[0.5, 1.0, 2.0, 4.0]),
    "block16": lambda: build_workload("bs16f4", replace(FP4, block_size=16), [900, 4000], [1, 2], seed=54,
                                      slack_blocks=3),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fp4_stages_match_oracle(name):
    wl = CASES[name]()
    ref_pool = oracle_pool(wl)
    ref = oracle_step(wl, ref_pool)
    g = G.cuda_wl(CASES[name]())
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    assert lay.key_bytes == 64 and lay.block_stride == layout_of(wl).block_stride
    pool = G.gpu_pool(g, lay)
    res = G.run_stages(g, pool, lay, prm)
    assert res["err"] == 0
    assert np.array_equal(pool.cpu().numpy(), ref_pool), f"{name}: pool bytes differ after the store"
    for t in range(wl.n_tokens):
        n = ref[t]["pos"] + 1
        assert np.array_equal(G.canon(res["scores"][t, :n]), G.canon(ref[t]["scores"])), f"{name} scores row {t}"
        assert np.array_equal(res["topk"][t], ref[t]["topk"]), f"{name} topk row {t}"
    out_ref = np.stack([ref[t]["out"] for t in range(wl.n_tokens)])
    lse_ref = np.stack([ref[t]["lse"] for t in range(wl.n_tokens)])
    G.assert_attention_close(res["out"], res["lse"], out_ref, lse_ref, name)
    dec = G.run_decode(g, G.gpu_pool(g, lay), lay, prm)
    assert dec["err"] == 0 and np.array_equal(dec["topk"], res["topk"])


def _spec_table():
    t = np.zeros(16, np.float32)
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_spec_values.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            t[int(c, 16)] = float(v)
    return torch.from_numpy(t)


def test_fp4_scores_equal_e4m3_storage_of_the_same_values():
    """The same key values held as E4M3 codes (torch's fp8 cast of the spec table's values) in an
    E4M3 layout give bit-identical GPU scores and selections: only the key bytes read differ."""
    g4 = G.cuda_wl(make_config(2, scale=0.2, key_format="e2m1"))
    table = _spec_table().cuda()

    def as_e4m3(packed):
        v = torch.stack([table[(packed & 0xF).long()], table[(packed >> 4).long()]], dim=-1).reshape(packed.shape[0], -1)
        return v.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()

    lay4, prm = G.gpu_layout(g4), G.gpu_params(g4)
    a = G.run_stages(g4, G.gpu_pool(g4, lay4), lay4, prm)
    g8 = G.cuda_wl(make_config(2, scale=0.2, key_format="e2m1"))
    g8.dims = replace(g8.dims, key_format="e4m3")
    g8.slot_idx_k = as_e4m3(g8.slot_idx_k)
    g8.new_idx_k = as_e4m3(g8.new_idx_k)
    lay8 = G.gpu_layout(g8)
    assert lay8.block_stride > lay4.block_stride
    b = G.run_stages(g8, G.gpu_pool(g8, lay8), lay8, prm)
    assert a["err"] == 0 and b["err"] == 0
    for t in range(g4.n_tokens):
        n = int(g4.seq_lens[t])
        assert np.array_equal(G.canon(a["scores"][t, :n]), G.canon(b["scores"][t, :n])), f"row {t}"
    assert np.array_equal(a["topk"], b["topk"])
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [3, 4])
def test_fp4_full_size_sampled_rows(cfg):
    """Full-size FP4 shapes in the bench's launch configuration: every row's selection is the exact
    top-k of its GPU score row; sampled rows against the oracle (scores, top-k, attention)."""
    wl = make_config(cfg, device="cuda", key_format="e2m1")
    lay, prm = G.gpu_layout(wl), G.gpu_params(wl)
    pool = G.gpu_pool(wl, lay)
    res = G.run_decode(wl, pool, lay, prm, store=True)
    assert res["err"] == 0
    stride = (wl.max_ctx + 3) // 4 * 4
    scores = torch.empty((wl.n_tokens, stride), dtype=torch.float32, device="cuda")
    smla.smla_index_scores(lay, prm, pool, 0, wl.q_idx, wl.w, wl.block_table, wl.seq_lens, wl.query_start_loc,
                           wl.max_q, wl.max_ctx, scores)
    assert smla.smla_get_last_error() == 0
    seqs, pos = oracle.query_positions(npy(wl.seq_lens), npy(wl.query_start_loc))
    assert_topk_exact(scores, torch.from_numpy(res["topk"]).cuda(), torch.from_numpy(pos + 1), wl.dims.top_k,
                      f"fp4 config {cfg}")
    rows = [0] if cfg == 4 else [0, wl.n_tokens - 1]
    lo = layout_of(wl)
    for t in rows:
        b = int(seqs[t])
        ref_pool = oracle_pool(wl, slots=sequence_slots(wl, b))
        ref = oracle.decode_step(
            lo, ref_pool, 0, latent_new=bits(wl.new_latent), rope_new=bits(wl.new_rope), idxk_new=npy(wl.new_idx_k),
            idxs_new=npy(wl.new_idx_s), slot_mapping=npy(wl.slot_mapping), q=bits(wl.q), q_pe=bits(wl.q_pe),
            q_idx=npy(wl.q_idx), w=npy(wl.w), block_table=npy(wl.block_table), seq_lens=npy(wl.seq_lens),
            query_start_loc=npy(wl.query_start_loc), top_k=wl.dims.top_k, sigma=wl.dims.softmax_scale, rows=[t])
        n = int(pos[t]) + 1
        assert np.array_equal(G.canon(scores[t, :n].cpu().numpy()), G.canon(ref[t]["scores"])), f"scores row {t}"
        assert np.array_equal(res["topk"][t], ref[t]["topk"]), f"topk row {t}"
        G.assert_attention_close(res["out"][t], res["lse"][t], ref[t]["out"], ref[t]["lse"], f"fp4 cfg {cfg} row {t}")
