"""Pins of the top-k property check used by the full-size GPU tests.

The check must accept the oracle's selection on every row, including rows
with heavy ties, rows shorter than k and rows with -0/+0 scores, and reject
each kind of wrong selection planted below.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.topk_properties import CHECKS, topk_violations


def _rows(seed, T=40, S=300, k=32, levels=6):
    rng = np.random.default_rng(seed)
    n = rng.integers(1, S + 1, size=T)
    n[:3] = [1, k, k + 1]                                   # shorter than, equal to and just above k
    scores = np.full((T, S), np.nan, dtype=np.float32)      # positions past n are never read
    for t in range(T):
        scores[t, :n[t]] = rng.integers(-levels, levels + 1, size=n[t]).astype(np.float32) * 0.5
    scores[3, :n[3]] = 0.0
    scores[3, 1:n[3]:2] = -0.0                              # -0 and +0 tie as values
    topk = np.stack([oracle.topk_select(scores[t, :n[t]], k) for t in range(T)])
    return torch.from_numpy(scores), torch.from_numpy(topk), torch.from_numpy(n), k


def _only(bad, check):
    return [c for c in CHECKS if bad[c]] == [check]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_selection_passes_every_check(seed):
    s, tk, n, k = _rows(seed)
    bad = topk_violations(s, tk, n, k, rows_per_chunk=7)
    assert not any(bad.values()), bad


def _row_with_left_out(s, tk, n, k, need_tie=False):
    for t in range(tk.shape[0]):
        if n[t] <= k:
            continue
        kept = tk[t][tk[t] >= 0]
        thr = s[t, kept].min()
        left = np.setdiff1d(np.arange(int(n[t])), kept.numpy())
        tied_left = left[(s[t, left] == thr).numpy()]
        if not need_tie or tied_left.size:
            return t, kept.numpy(), left, thr, tied_left
    raise AssertionError("no suitable row")


def test_catches_a_lower_score_kept_instead_of_a_higher_one():
    s, tk, n, k = _rows(0)
    t, kept, left, thr, _ = _row_with_left_out(s, tk, n, k)
    s[t, kept[0]] = float(thr) - 100.0                      # the kept position now scores below every other
    bad = topk_violations(s, tk, n, k)
    assert t in bad["threshold"]


def test_catches_a_tie_resolved_to_the_higher_position():
    s, tk, n, k = _rows(1, levels=2)
    t, kept, left, thr, tied_left = _row_with_left_out(s, tk, n, k, need_tie=True)
    kept_at = kept[(s[t, kept] == thr).numpy()]
    new = np.sort(np.concatenate([np.setdiff1d(kept, [kept_at.max()]), [tied_left.max()]]))
    tk[t, :new.size] = torch.from_numpy(new.astype(np.int32))
    bad = topk_violations(s, tk, n, k)
    assert _only({c: [r for r in v if r == t] for c, v in bad.items()}, "ties")


def test_catches_a_dropped_entry_unsorted_output_and_out_of_range_position():
    s, tk, n, k = _rows(2)
    full = [t for t in range(tk.shape[0]) if n[t] > k]
    a, b, c = full[:3]
    tk[a, k - 1] = -1                                        # one slot short
    tk[b, [0, 1]] = tk[b, [1, 0]]                            # two positions swapped
    tk[c, k - 1] = int(n[c])                                 # past the visible context
    bad = topk_violations(s, tk, n, k)
    assert a in bad["count"] and b in bad["ascending"] and c in bad["in_range"]


def test_catches_a_gap_before_the_padding():
    s, tk, n, k = _rows(0)
    t = 0                                                    # n = 1: one kept position, then padding
    tk[t, 0], tk[t, 1] = -1, 0
    bad = topk_violations(s, tk, n, k)
    assert t in bad["prefix"]
