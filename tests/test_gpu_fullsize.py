"""Full-size parity on sampled query tokens, in the launch configuration bench.py times.

The whole step runs on the GPU through smla_decode for every query token of
the named workloads; the oracle recomputes chosen rows one by one (its pool
holds the sampled sequence's cached context, written by the oracle's store).
Indexer scores of those rows are compared bit for bit, top-k exactly,
attention within the stated tolerance.  Every other row's selection is checked
against its own GPU score row with the exact top-k characterisation of
tests/topk_properties.py (count, order, range, threshold, ties), which holds
at any size.  Once every selection is shown exact that way, every row's
attention output and lse are compared with oracle.sparse_attend over that
selection, on an oracle pool that holds the selected records (written by the
oracle's own store from the workload's inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_mla_gb300.workloads import make_config
from tests.oracle_helpers import bits, layout_of, npy, oracle_pool, sequence_slots
from tests import gpu_helpers as G
from tests.topk_properties import assert_topk_exact

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


def _sample_rows(wl, cfg):
    T = wl.n_tokens
    qsl = npy(wl.query_start_loc)
    if cfg == 3:
        parent = 0
        child = next(b for b, p in enumerate(wl.parents) if p == 0)
        return [int(qsl[parent]), int(qsl[child + 1] - 1)]
    if cfg == 4:
        return [0]
    if cfg == 5:
        return [0, T // 2 - 1, T - 1]
    return [0, T // 2, T - 1]


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_sampled_rows(cfg):
    wl = make_config(cfg, device="cuda")
    lay, prm = G.gpu_layout(wl), G.gpu_params(wl)
    pool = G.gpu_pool(wl, lay)
    res = G.run_decode(wl, pool, lay, prm, store=True)
    assert res["err"] == 0
    stride = (wl.max_ctx + 3) // 4 * 4
    scores = torch.empty((wl.n_tokens, stride), dtype=torch.float32, device="cuda")
    G.smla.smla_index_scores(lay, prm, pool, 0, wl.q_idx, wl.w, wl.block_table, wl.seq_lens, wl.query_start_loc,
                             wl.max_q, wl.max_ctx, scores)
    assert G.smla.smla_get_last_error() == 0
    rows = _sample_rows(wl, cfg)
    seqs, pos = oracle.query_positions(npy(wl.seq_lens), npy(wl.query_start_loc))
    # every row: the fused step's selection is the top-k of its score row
    assert_topk_exact(scores, torch.from_numpy(res["topk"]).cuda(), torch.from_numpy(pos + 1), wl.dims.top_k,
                      f"config {cfg}")
    lo = layout_of(wl)
    by_seq = {}
    for t in rows:
        by_seq.setdefault(int(seqs[t]), []).append(t)
    for b, ts in by_seq.items():
        ref_pool = oracle_pool(wl, slots=sequence_slots(wl, b))
        ref = oracle.decode_step(
            lo, ref_pool, 0, latent_new=bits(wl.new_latent), rope_new=bits(wl.new_rope), idxk_new=npy(wl.new_idx_k),
            idxs_new=npy(wl.new_idx_s), slot_mapping=npy(wl.slot_mapping), q=bits(wl.q), q_pe=bits(wl.q_pe),
            q_idx=npy(wl.q_idx), w=npy(wl.w), block_table=npy(wl.block_table), seq_lens=npy(wl.seq_lens),
            query_start_loc=npy(wl.query_start_loc), top_k=wl.dims.top_k, sigma=wl.dims.softmax_scale, rows=ts)
        for t in ts:
            n = int(pos[t]) + 1
            got = scores[t, :n].cpu().numpy()
            assert np.array_equal(G.canon(got), G.canon(ref[t]["scores"])), f"config {cfg} scores row {t}"
            assert np.array_equal(res["topk"][t], ref[t]["topk"]), f"config {cfg} topk row {t}"
            G.assert_attention_close(res["out"][t], res["lse"][t], ref[t]["out"], ref[t]["lse"], f"config {cfg} row {t}")
    _check_every_row_attention(wl, lo, res, seqs, f"config {cfg}")


def _check_every_row_attention(wl, lo, res, seqs, what):
    """Every row's out/lse against oracle.sparse_attend over the row's (property-checked) selection."""
    bs = wl.dims.block_size
    bt = npy(wl.block_table)
    topk = res["topk"]
    rows = np.repeat(np.asarray(seqs, np.int64)[:, None], topk.shape[1], axis=1)
    sel = topk >= 0
    slots = np.unique(bt[rows[sel], topk[sel] // bs].astype(np.int64) * bs + topk[sel] % bs)
    new_slots = npy(wl.slot_mapping)
    ref_pool = oracle_pool(wl, slots=np.setdiff1d(slots, new_slots))
    oracle.kvpack_store(lo, ref_pool, 0, bits(wl.new_latent), bits(wl.new_rope), npy(wl.new_idx_k),
                        npy(wl.new_idx_s), new_slots)
    q, q_pe = bits(wl.q), bits(wl.q_pe)
    out_ref = np.empty(res["out"].shape, np.float64)
    lse_ref = np.empty(res["lse"].shape, np.float64)
    for t in range(wl.n_tokens):
        out_ref[t], lse_ref[t] = oracle.sparse_attend(lo, ref_pool, 0, oracle.bf16_bits_to_f64(q[t]),
                                                      oracle.bf16_bits_to_f64(q_pe[t]), topk[t], bt[seqs[t]],
                                                      wl.dims.softmax_scale)
    G.assert_attention_close(res["out"], res["lse"], out_ref, lse_ref, f"{what}, every row")
