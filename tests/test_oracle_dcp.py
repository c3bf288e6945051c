"""Pins of the split-context oracle (CPU): the shard decomposition must equal the unsharded path.

The candidate merge is checked against the textbook top-k of the whole row, the
LSE merge against softmax attention over the whole key set (a closed form: the
partition of a softmax sum), and the shard visibility rule against brute force.
"""
import numpy as np
import pytest

import oracle
from oracle import dcp


@pytest.mark.parametrize("n_shards", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("n,k", [(1, 4), (7, 4), (64, 16), (300, 64), (1000, 128), (129, 128)])
def test_topk_merge_equals_unsharded_topk(n_shards, n, k):
    rng = np.random.default_rng(1000 * n_shards + n + k)
    # heavy ties: few distinct values, and -0 / +0 both present
    s = rng.integers(-3, 4, size=n).astype(np.float32) * np.float32(0.5)
    s[rng.random(n) < 0.05] = np.float32(-0.0)
    shard_rows = [s[r::n_shards] for r in range(n_shards)]
    shard_topk = [oracle.topk_select(row, k) for row in shard_rows]
    glob, per = dcp.topk_merge(shard_rows, shard_topk, n_shards, k)
    assert np.array_equal(glob, oracle.topk_select(s, k))
    # the per-shard lists are the global selection in local coordinates
    sel = glob[glob >= 0]
    for r in range(n_shards):
        loc = per[r][per[r] >= 0]
        assert np.array_equal(loc, np.sort(sel[sel % n_shards == r] // n_shards))
        assert np.all(per[r][loc.size:] == -1)


def test_topk_merge_with_short_shards_pads():
    s = np.array([5, 1, 4], dtype=np.float32)        # 3 positions over 4 shards: shard 3 is empty
    rows = [s[r::4] for r in range(4)]
    tk = [oracle.topk_select(row, 4) for row in rows]
    glob, per = dcp.topk_merge(rows, tk, 4, 4)
    assert glob.tolist() == [0, 1, 2, -1]
    assert per[3].tolist() == [-1, -1, -1, -1]


@pytest.mark.parametrize("n_shards", [1, 2, 3, 5])
def test_lse_merge_equals_attention_over_all_keys(n_shards):
    rng = np.random.default_rng(7 + n_shards)
    H, DL, DR, n = 4, 16, 8, 37
    q, qpe = rng.normal(size=(H, DL)), rng.normal(size=(H, DR))
    lat, rope = rng.normal(size=(n, DL)), rng.normal(size=(n, DR))
    sigma = 1 / np.sqrt(DL + DR)
    out_all, lse_all = oracle.attend(q, qpe, lat, rope, sigma)
    part = rng.integers(0, n_shards, size=n)          # an arbitrary partition of the keys
    outs, lses = [], []
    for r in range(n_shards):
        m = part == r
        o, l = oracle.attend(q, qpe, lat[m], rope[m], sigma)
        outs.append(o)
        lses.append(l)
    out, lse = dcp.lse_merge(np.stack(outs), np.stack(lses))
    assert np.allclose(out, out_all, rtol=0, atol=1e-12)
    assert np.allclose(lse, lse_all, rtol=0, atol=1e-12)


def test_lse_merge_identity_and_empty_parts():
    rng = np.random.default_rng(3)
    o = rng.normal(size=(1, 2, 5))
    l = np.array([[0.3, -1.2]])
    out, lse = dcp.lse_merge(o, l)
    assert np.allclose(out, o[0]) and np.allclose(lse, l[0])
    # an empty part (out 0, lse -inf) changes nothing
    out2, lse2 = dcp.lse_merge(np.concatenate([o, np.zeros_like(o)]), np.concatenate([l, np.full_like(l, -np.inf)]))
    assert np.allclose(out2, o[0]) and np.allclose(lse2, l[0])
    # all parts empty: out 0, lse -inf
    out3, lse3 = dcp.lse_merge(np.zeros((3, 2, 5)), np.full((3, 2), -np.inf))
    assert np.all(out3 == 0) and np.all(lse3 == -np.inf)
    # two equal parts: the mean, and lse + ln 2
    out4, lse4 = dcp.lse_merge(np.stack([o[0], o[0]]), np.stack([l[0], l[0]]))
    assert np.allclose(out4, o[0]) and np.allclose(lse4, l[0] + np.log(2))


@pytest.mark.parametrize("n_shards", [1, 2, 3, 4])
def test_shard_visibility_by_brute_force(n_shards):
    for p in range(0, 40):
        for r in range(n_shards):
            brute = sum(1 for j in range(p + 1) if j % n_shards == r)
            assert dcp.shard_visible(p, r, n_shards) == brute


@pytest.mark.parametrize("n_shards", [2, 4])
def test_sharded_sparse_attention_equals_unsharded(n_shards):
    """Scores, local top-k, candidate merge, per-shard attention and LSE merge reproduce the one-shard result."""
    rng = np.random.default_rng(11 * n_shards)
    H, DL, DR, n, k = 4, 16, 8, 203, 32
    q, qpe = rng.normal(size=(H, DL)), rng.normal(size=(H, DR))
    lat, rope = rng.normal(size=(n, DL)), rng.normal(size=(n, DR))
    scores = rng.integers(-20, 21, size=n).astype(np.float32)
    sigma = 1 / np.sqrt(DL + DR)
    sel = oracle.topk_select(scores, k)
    sel = sel[sel >= 0]
    out_ref, lse_ref = oracle.attend(q, qpe, lat[sel], rope[sel], sigma)
    rows = [scores[r::n_shards] for r in range(n_shards)]
    glob, per = dcp.topk_merge(rows, [oracle.topk_select(row, k) for row in rows], n_shards, k)
    outs, lses = [], []
    for r in range(n_shards):
        loc = per[r][per[r] >= 0]
        j = loc * n_shards + r
        o, l = oracle.attend(q, qpe, lat[j], rope[j], sigma)
        outs.append(o)
        lses.append(l)
    out, lse = dcp.lse_merge(np.stack(outs), np.stack(lses))
    assert np.array_equal(np.sort(glob[glob >= 0]), np.sort(sel))
    assert np.allclose(out, out_ref, rtol=0, atol=1e-12) and np.allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_workload_shard_rule_matches_oracle():
    """The workload builder's shard visibility (used to build GPU shard pools) follows the oracle's rule."""
    from paged_sparse_mla_gb300 import workloads
    for n_shards in (1, 2, 3, 8):
        for p in range(50):
            for r in range(n_shards):
                assert workloads.shard_visible(p, r, n_shards) == dcp.shard_visible(p, r, n_shards)
