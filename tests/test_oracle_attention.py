"""Pins for the oracle's attention (CPU only)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests.oracle_helpers import layout_of, npy, oracle_pool, oracle_step, bits
from paged_sparse_mla_gb300.workloads import make_config, build_workload, TINY


def _rand(shape, seed):
    return np.random.default_rng(seed).normal(size=shape)


@pytest.mark.parametrize("n", [1, 3, 64, 300])
def test_attend_matches_torch_sdpa(n):
    h, dl, dr = 8, 64, 16
    q, qpe, lat, rope = _rand((h, dl), 1), _rand((h, dr), 2), _rand((n, dl), 3), _rand((n, dr), 4)
    sigma = 1 / math.sqrt(80)
    out, lse = oracle.attend(q, qpe, lat, rope, sigma)
    qq = torch.from_numpy(np.concatenate([q, qpe], 1))[None, :, None, :]      # [1, H, 1, D]
    kk = torch.from_numpy(np.concatenate([lat, rope], 1))[None, None].expand(1, h, n, dl + dr)
    vv = torch.from_numpy(lat)[None, None].expand(1, h, n, dl)
    ref = F.scaled_dot_product_attention(qq, kk, vv, scale=sigma)[0, :, 0]
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    ref_lse = torch.logsumexp(sigma * (qq[0, :, 0] @ kk[0, 0].T), dim=1)
    assert np.allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_single_key_returns_that_key():
    lat, rope = _rand((1, 64), 5), _rand((1, 16), 6)
    q, qpe = _rand((8, 64), 7), _rand((8, 16), 8)
    out, lse = oracle.attend(q, qpe, lat, rope, 0.3)
    assert np.allclose(out, np.repeat(lat, 8, 0), rtol=0, atol=1e-15)
    assert np.allclose(lse, 0.3 * (q @ lat[0] + qpe @ rope[0]), rtol=1e-14)


def test_zero_query_gives_mean_and_log_n():
    lat, rope = _rand((37, 64), 9), _rand((37, 16), 10)
    out, lse = oracle.attend(np.zeros((4, 64)), np.zeros((4, 16)), lat, rope, 0.5)
    assert np.allclose(out, lat.mean(0)[None].repeat(4, 0), rtol=1e-13, atol=1e-14)
    assert np.allclose(lse, math.log(37), rtol=1e-14)


def test_empty_set():
    out, lse = oracle.attend(np.ones((2, 4)), np.ones((2, 2)), np.zeros((0, 4)), np.zeros((0, 2)), 1.0)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_dominant_key():
    lat, rope = _rand((10, 8), 11), np.zeros((10, 2))
    q = np.zeros((1, 8))
    q[0] = lat[4] * 50
    out, _ = oracle.attend(q, np.zeros((1, 2)), lat, rope, 1.0)
    assert np.allclose(out[0], lat[4], atol=1e-8)


def test_sparse_equals_dense_when_topk_covers_context():
    """Prompts inside the top-k still take the sparse kernel: results must match dense."""
    wl = make_config(1)
    pool = oracle_pool(wl)
    res = oracle_step(wl, pool, top_k=256)
    lay = layout_of(wl)
    for t, r in res.items():
        assert (r["topk"] >= 0).sum() == r["pos"] + 1
        out, lse = oracle.dense_attend(lay, pool, 0, oracle.bf16_bits_to_f64(bits(wl.q[t])),
                                       oracle.bf16_bits_to_f64(bits(wl.q_pe[t])),
                                       npy(wl.block_table[r["seq"]]), r["pos"], wl.dims.softmax_scale)
        assert np.allclose(r["out"], out, rtol=1e-12, atol=1e-13)
        assert np.allclose(r["lse"], lse, rtol=1e-12, atol=1e-13)


def test_sparse_differs_from_dense_when_topk_smaller():
    wl = make_config(1)
    pool = oracle_pool(wl)
    res = oracle_step(wl, pool)
    lay = layout_of(wl)
    r = res[0]
    assert (r["topk"] >= 0).sum() == 64
    out, _ = oracle.dense_attend(lay, pool, 0, oracle.bf16_bits_to_f64(bits(wl.q[0])),
                                 oracle.bf16_bits_to_f64(bits(wl.q_pe[0])), npy(wl.block_table[0]),
                                 r["pos"], wl.dims.softmax_scale)
    assert not np.allclose(r["out"], out, atol=1e-3)
