"""Pins for the oracle's indexer scores and top-k selection (CPU only)."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from paged_sparse_mla_gb300.workloads import TINY, build_workload, make_config
from tests.oracle_helpers import bits, layout_of, npy, oracle_pool


def _int_values(codes_u8: torch.Tensor) -> np.ndarray:
    """E4M3 codes holding integers -> int64 through torch's own fp8 cast."""
    v = codes_u8.view(torch.float8_e4m3fn).to(torch.float64)
    assert torch.equal(v, v.round())
    return v.to(torch.int64).numpy()


def test_scores_equal_integer_recomputation():
    """Integer inputs: 4*I = sum_h (4 w_h) * max(0, q_h . k) exactly, in int64."""
    wl = make_config(1)
    lay = layout_of(wl)
    pool = oracle_pool(wl)
    oracle.kvpack_store(lay, pool, 0, bits(wl.new_latent), bits(wl.new_rope), npy(wl.new_idx_k),
                        npy(wl.new_idx_s), npy(wl.slot_mapping))
    src = wl.slot_idx_k.clone()
    src[wl.slot_mapping] = wl.new_idx_k
    seqs, pos = oracle.query_positions(npy(wl.seq_lens), npy(wl.query_start_loc))
    w4 = (npy(wl.w) * 4).astype(np.int64)
    q = _int_values(wl.q_idx)
    for t in range(len(seqs)):
        b, p = seqs[t], pos[t]
        got = oracle.index_scores_row(lay, pool, 0, npy(wl.q_idx[t]), npy(wl.w[t]),
                                      npy(wl.block_table[b]), p)
        slots = oracle.context_slots(npy(wl.block_table[b]), p + 1, lay.block_size)
        k = _int_values(src[torch.as_tensor(slots)])
        dots = q[t] @ k.T                               # int64 [H_I, n]
        ref4 = (w4[t][:, None] * np.maximum(dots, 0)).sum(axis=0)
        assert np.array_equal(got.astype(np.float64) * 4, ref4.astype(np.float64))


def test_scores_brute_force_loops_tiny():
    dims = TINY
    wl = build_workload("bf", dims, [37, 5], [2, 1], seed=11, idx_scale=[0.5, 2.0, 1.0])
    lay = layout_of(wl)
    pool = oracle_pool(wl)
    # the step's own tokens are stored first
    oracle.kvpack_store(lay, pool, 0, np.zeros((3, dims.d_latent), np.uint16),
                        np.zeros((3, dims.d_rope), np.uint16), npy(wl.new_idx_k), npy(wl.new_idx_s),
                        npy(wl.slot_mapping))
    seqs, pos = oracle.query_positions(npy(wl.seq_lens), npy(wl.query_start_loc))
    assert list(pos) == [35, 36, 4]
    qv = wl.q_idx.view(torch.float8_e4m3fn).double().numpy()
    for t in range(3):
        b, p = seqs[t], pos[t]
        got = oracle.index_scores_row(lay, pool, 0, npy(wl.q_idx[t]), npy(wl.w[t]),
                                      npy(wl.block_table[b]), p)
        assert got.size == p + 1
        for j in range(p + 1):
            blk = int(wl.block_table[b, j // dims.block_size])
            slot = blk * dims.block_size + j % dims.block_size
            is_new = (wl.slot_mapping == slot).nonzero()
            src_k = wl.new_idx_k[is_new[0, 0]] if is_new.numel() else wl.slot_idx_k[slot]
            src_s = float(wl.new_idx_s[is_new[0, 0]] if is_new.numel() else wl.slot_idx_s[slot])
            kv = src_k.view(torch.float8_e4m3fn).double().tolist()
            total = 0.0
            for h in range(dims.n_idx_heads):
                dot = 0.0
                for d in range(dims.d_index):
                    dot += qv[t, h, d] * kv[d]
                total += float(wl.w[t, h]) * max(dot, 0.0)
            assert got[j] == np.float32(total * src_s), (t, j)


def test_scores_invariant_under_block_relocation():
    wl = make_config(1)
    lay = layout_of(wl)
    pool = oracle_pool(wl)
    rng = np.random.default_rng(3)
    perm = rng.permutation(wl.num_blocks)
    moved = np.zeros_like(pool)
    bs = lay.block_stride
    for old, new in enumerate(perm):
        moved[new * bs:(new + 1) * bs] = pool[old * bs:(old + 1) * bs]
    bt = npy(wl.block_table).astype(np.int64)
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    for b in range(2):
        a = oracle.index_scores_row(lay, pool, 0, npy(wl.q_idx[b]), npy(wl.w[b]), bt[b], 200)
        c = oracle.index_scores_row(lay, moved, 0, npy(wl.q_idx[b]), npy(wl.w[b]), bt2[b], 200)
        assert np.array_equal(a, c)


def _sorted_topk(scores, k):
    order = sorted(range(len(scores)), key=lambda j: (-float(scores[j]), j))
    keep = sorted(order[:k])
    return keep + [-1] * (k - len(keep))


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_python_sort_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 400))
    s = (rng.integers(0, 12, size=n) * 0.25).astype(np.float32)     # heavy ties
    for k in (1, 7, 64, 500):
        assert list(oracle.topk_select(s, k)) == _sorted_topk(s, k)


def test_topk_special_cases():
    s = np.full(100, 3.5, dtype=np.float32)
    assert list(oracle.topk_select(s, 10)) == list(range(10))              # all equal -> first k
    assert list(oracle.topk_select(s[:5], 8)) == [0, 1, 2, 3, 4, -1, -1, -1]  # n <= k
    r = np.random.default_rng(1).normal(size=50).astype(np.float32)
    r[[7, 30]] = r.max() + 1
    assert list(oracle.topk_select(r, 1)) == [int(np.argmax(r))] == [7]   # k=1: argmax, lowest index
    z = np.array([0.0, -0.0, 0.0, -1.0], dtype=np.float32)
    assert list(oracle.topk_select(z, 2)) == [0, 1]                        # -0.0 == +0.0
    assert list(oracle.topk_select(np.array([-np.inf, 1, -np.inf], np.float32), 2)) == [0, 1]


def test_topk_exhaustive_tiny():
    for n in range(1, 6):
        for vals in itertools.product([0.0, 1.0, 2.0], repeat=n):
            s = np.array(vals, dtype=np.float32)
            for k in range(1, 7):
                assert list(oracle.topk_select(s, k)) == _sorted_topk(s, k)
