"""GPU parity of smla_topk on rows that take each of its exact fallback paths.

The fast path collects the positions whose score reaches a threshold taken from
an evenly spread sample of the row, into one list per warp (each warp scans its
own contiguous segment of the row, 512 entries per list), and falls back to an
exact radix select over the whole row when:

  overflow   one warp's list overflows: the top scores cluster in one segment
             (a contiguous run of high scores, the top k in the last 1/16 of the
             row, a monotone row); the hits are then collected once more into
             lists packed one after another, or, beyond the buffer, the row
             takes the radix select;
  miss       the sample overestimates the threshold and fewer than k positions
             reach it: the highest scores sit exactly at the sampled positions;
  plateau    more positions reach the threshold than the candidate buffer holds
             (8,192): a plateau of equal top scores;
  large k    k is above the fast path's limit (4,096);
  unaligned  the row does not start on a 16-byte boundary (an odd row stride).

Each case is checked row for row against oracle.topk_select, with heavy ties,
through the one-CTA-per-row path and through the split-segment path (long rows
of a small batch, where the clustered segment overflows in the first stage and
the clustered candidates in the second).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_sparse_mla_gb300 as smla
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

SAMPLE_RUNS = 2048  # the fast path samples 2,048 runs of 4 consecutive positions


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


def _background(rng, n):
    return rng.integers(-60, 61, size=n).astype(np.float32) * np.float32(0.25)


def clustered_row(rng, n, lo, hi):
    """Background scores with a run of high, heavily tied scores on positions [lo, hi)."""
    s = _background(rng, n)
    s[lo:hi] = np.float32(100.0) + rng.integers(0, 40, size=hi - lo).astype(np.float32)
    return s


def monotone_row(n, increasing=True):
    s = np.arange(n, dtype=np.float32) if increasing else np.arange(n, 0, -1, dtype=np.float32)
    return s * np.float32(0.5)


def sample_aligned_row(rng, m, ties):
    """A row of n = (SAMPLE_RUNS - 1) * m + 4 positions whose highest scores sit exactly on the
    positions the fast path samples (runs of 4 starting every m positions), so that the sample's
    threshold is reached by far fewer than k positions."""
    n = (SAMPLE_RUNS - 1) * m + 4
    s = _background(rng, n)
    starts = np.arange(SAMPLE_RUNS) * m
    pos = (starts[:, None] + np.arange(4)[None, :]).ravel()
    if ties:
        s[pos] = np.float32(1000.0) + rng.integers(0, 100, size=pos.size).astype(np.float32)
    else:
        s[pos] = np.float32(1000.0) + rng.permutation(pos.size).astype(np.float32)
    return s


def _run_topk(rows, k, split=False, stride=None):
    """smla_topk over the given rows (one sequence per row, one query token each)."""
    R = len(rows)
    lens = [r.size for r in rows]
    if stride is None:
        stride = (max(lens) + 3) // 4 * 4
    scores = np.full((R, stride), np.float32(-1e30), dtype=np.float32)
    for t, r in enumerate(rows):
        scores[t, :r.size] = r
    prm = smla.make_params(64, 64, k, 1.0)
    ws = None
    if split:
        ws = torch.empty(smla.topk_workspace_size(prm, R), dtype=torch.uint8, device="cuda")
        assert ws.numel() > 0
    out = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qsl = torch.arange(R + 1, dtype=torch.int32, device="cuda")
    smla.smla_topk(prm, torch.as_tensor(scores, device="cuda"), seq_lens, qsl, out, workspace=ws)
    assert smla.smla_get_last_error() == 0
    return out.cpu().numpy()


def _check(rows, got, k, what):
    for t, r in enumerate(rows):
        assert np.array_equal(got[t], oracle.topk_select(r, k)), f"{what}: row {t}"


def test_overflow_of_one_warp_list():
    rng = np.random.default_rng(201)
    n = 100_000
    rows = [
        clustered_row(rng, n, 40_000, 43_000),          # inside one warp's segment
        clustered_row(rng, n, n - n // 16, n),          # the top k in the last 1/16 of the row
        clustered_row(rng, n, 0, 2_600),                # at the start
        monotone_row(n, increasing=True),
        monotone_row(n, increasing=False),
        clustered_row(rng, 250_001, 120_000, 126_000),  # a longer, odd-length row
    ]
    _check(rows, _run_topk(rows, 2048), 2048, "overflow")


@pytest.mark.parametrize("ties", [False, True])
def test_sample_misses_the_threshold(ties):
    rng = np.random.default_rng(202 + ties)
    rows = [sample_aligned_row(rng, m, ties) for m in (50, 64, 97)]
    _check(rows, _run_topk(rows, 2048), 2048, "sample miss")


def test_plateau_of_ties_beyond_the_candidate_buffer():
    rng = np.random.default_rng(207)
    n = 120_000
    rows = []
    a = _background(rng, n)
    a[rng.choice(n, 10_000, replace=False)] = np.float32(50.0)         # spread plateau
    rows.append(a)
    b = _background(rng, n)
    b[30_000:42_000] = np.float32(50.0)                                # contiguous plateau
    rows.append(b)
    c = _background(rng, n)
    c[rng.choice(n, 9_000, replace=False)] = np.float32(50.0)          # plateau with 1,000 above it
    c[rng.choice(n, 1_000, replace=False)] = np.float32(60.0) + rng.integers(0, 5, 1_000).astype(np.float32)
    rows.append(c)
    _check(rows, _run_topk(rows, 2048), 2048, "plateau")


def test_k_above_the_fast_path_limit():
    rng = np.random.default_rng(204)
    k = 4100
    rows = [_background(rng, 60_000), clustered_row(rng, 30_001, 10_000, 16_000), _background(rng, 4_100),
            _background(rng, 4_000), monotone_row(9_000, increasing=False)]
    _check(rows, _run_topk(rows, k), k, "k = 4100")


def test_rows_off_the_16_byte_boundary():
    rng = np.random.default_rng(205)
    rows = [_background(rng, 10_001), clustered_row(rng, 10_001, 100, 3_000), _background(rng, 9_999),
            _background(rng, 10_000)]
    got = _run_topk(rows, 2048, stride=10_001)          # rows 1 and 3 start 4 bytes past a boundary
    _check(rows, got, 2048, "unaligned")


def test_clustered_rows_on_the_split_segment_path():
    """Few long rows with a scratch: stage 1 selects each segment on its own CTA (the clustered
    segment overflows there), stage 2 selects over the segments' candidates (the cluster's
    candidates are contiguous and overflow again)."""
    rng = np.random.default_rng(206)
    rows = [clustered_row(rng, 300_000, 150_000, 156_000), clustered_row(rng, 200_000, 190_000, 200_000),
            monotone_row(260_000, increasing=True), sample_aligned_row(rng, 120, ties=True), _background(rng, 90_000)]
    _check(rows, _run_topk(rows, 2048, split=True), 2048, "split")
