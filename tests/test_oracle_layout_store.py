"""Pins for the packed layout and the FP8 store (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.store import quantize_latent, bf16_bits_to_f64
from paged_sparse_mla_gb300.workloads import FULL, TINY, make_config
from tests.oracle_helpers import bits, layout_of, npy, oracle_pool


def test_record_sizes_match_shapes():
    full = oracle.PoolLayout(64, 1, 512, 64, 128, 128, 10)
    assert full.rec_bytes == 656 and full.rec_stride == 656
    assert full.idx_key_off == 41_984 and full.idx_scale_off == 50_176
    assert full.block_stride == 50_432
    tiny = oracle.PoolLayout(16, 1, 64, 16, 64, 32, 10)
    assert tiny.rec_bytes == 100 and tiny.rec_stride == 112


@pytest.mark.parametrize("n_layers", [1, 2, 3])
@pytest.mark.parametrize("dims", [FULL, TINY])
def test_regions_tile_the_pool_without_overlap(dims, n_layers):
    lay = oracle.PoolLayout(dims.block_size, n_layers, dims.d_latent, dims.d_rope, dims.quant_tile,
                            dims.d_index, 3)
    owner = np.full(lay.pool_bytes, -1, dtype=np.int64)
    tag = 0
    for layer in range(n_layers):
        for slot in range(3 * dims.block_size):
            for start, size in ((lay.record_offset(slot, layer), lay.rec_bytes),
                                (lay.index_key_offset(slot, layer), dims.d_index),
                                (lay.index_scale_offset(slot, layer), 4)):
                assert (owner[start:start + size] == -1).all()
                owner[start:start + size] = tag
                tag += 1
        for blk in range(3):
            base = blk * lay.block_stride + layer * lay.layer_stride
            for off in (lay.rec_off, lay.idx_key_off, lay.idx_scale_off):
                assert (base + off) % 256 == 0
    assert lay.block_stride % 256 == 0


def test_quantize_matches_torch_fp32_route():
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(64, 512, generator=g) * torch.exp(torch.randn(64, 1, generator=g) * 3)).to(torch.bfloat16)
    codes, scales = quantize_latent(bits(x), 128)
    xf = x.float().view(64, 4, 128)
    amax = xf.abs().amax(dim=2)
    ref_scale = amax / 448.0
    ref_scale = torch.where(ref_scale == 0, torch.ones_like(ref_scale), ref_scale)
    ref_codes = (xf / ref_scale[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(64, 512)
    assert np.array_equal(scales, ref_scale.numpy())
    assert np.array_equal(codes, ref_codes.numpy())


def test_quantize_error_bound_and_amax_code():
    g = torch.Generator().manual_seed(6)
    x = torch.randn(32, 512, generator=g).to(torch.bfloat16)
    codes, scales = quantize_latent(bits(x), 128)
    xv = bf16_bits_to_f64(bits(x)).reshape(32, 4, 128)
    deq = oracle.e4m3_decode(codes).reshape(32, 4, 128) * scales.astype(np.float64)[:, :, None]
    # RNE to 3 mantissa bits: relative error <= 2^-4 for normals, absolute <= 2^-10 * scale below 2^-6
    bound = np.maximum(np.abs(xv) * 2.0 ** -4, scales.astype(np.float64)[:, :, None] * 2.0 ** -10)
    assert (np.abs(deq - xv) <= bound * (1 + 1e-6)).all()
    # the element holding the tile's amax maps to +-448
    idx = np.abs(xv).argmax(axis=2)
    top = np.take_along_axis(oracle.e4m3_decode(codes).reshape(32, 4, 128), idx[:, :, None], axis=2)
    assert (np.abs(top) == 448.0).all()


def test_zero_tile_gets_unit_scale():
    x = torch.zeros(2, 128, dtype=torch.bfloat16)
    codes, scales = quantize_latent(bits(x), 64)
    assert (scales == 1.0).all() and (codes == 0).all()


def test_store_then_read_returns_quantised_inputs():
    wl = make_config(1)
    lay = layout_of(wl)
    pool = oracle_pool(wl)
    s = npy(wl.cached_slots)
    st = torch.as_tensor(s)
    lat, rope = oracle.read_record(lay, pool, 0, s)
    codes, scales = quantize_latent(bits(wl.slot_latent[st]), lay.quant_tile)
    expect = (oracle.e4m3_decode(codes).reshape(len(s), -1, lay.quant_tile)
              * scales.astype(np.float64)[:, :, None]).reshape(len(s), -1).astype(np.float32)
    assert np.array_equal(lat, expect.astype(np.float64))
    assert np.array_equal(rope, wl.slot_rope[st].double().numpy())
    keys, ks = oracle.read_index_key(lay, pool, 0, s)
    assert np.array_equal(keys, wl.slot_idx_k[st].view(torch.float8_e4m3fn).double().numpy())
    assert np.array_equal(ks, wl.slot_idx_s[st].double().numpy())


def test_full_record_round_trip_within_the_e4m3_bound():
    """Four per-128 scale tiles: every element comes back within the E4M3 rounding bound of its
    bf16 input, scaled by its own tile's scale (a read with another tile's scale breaks the bound)."""
    from paged_sparse_mla_gb300.workloads import build_workload
    wl = build_workload("round-trip", FULL, [300, 200], [1, 1], seed=11)
    lay = layout_of(wl)
    pool = oracle_pool(wl)
    s = npy(wl.cached_slots)
    st = torch.as_tensor(s)
    lat, rope = oracle.read_record(lay, pool, 0, s)
    x = bf16_bits_to_f64(bits(wl.slot_latent[st])).reshape(len(s), 4, 128)
    amax = np.abs(x).max(axis=2, keepdims=True)
    scale = amax / 448.0
    bound = np.maximum(np.abs(x) * 2.0 ** -4, scale * 2.0 ** -10) * (1 + 1e-6)
    assert (np.abs(lat.reshape(len(s), 4, 128) - x) <= bound).all()
    assert np.array_equal(rope, bf16_bits_to_f64(bits(wl.slot_rope[st])))


def test_store_skips_negative_slots_and_touches_only_its_bytes():
    wl = make_config(1)
    lay = layout_of(wl)
    pool = np.zeros(lay.pool_bytes, dtype=np.uint8)
    sm = npy(wl.slot_mapping).copy()
    sm[0] = -1
    oracle.kvpack_store(lay, pool, 0, bits(wl.new_latent), bits(wl.new_rope), npy(wl.new_idx_k),
                        npy(wl.new_idx_s), sm)
    touched = np.zeros(lay.pool_bytes, dtype=bool)
    for slot in sm[sm >= 0]:
        r = lay.record_offset(slot, 0)
        touched[r:r + lay.rec_bytes] = True
        k = lay.index_key_offset(slot, 0)
        touched[k:k + lay.d_index] = True
        c = lay.index_scale_offset(slot, 0)
        touched[c:c + 4] = True
    assert (pool[~touched] == 0).all()
    r0 = lay.record_offset(npy(wl.slot_mapping)[0], 0)
    assert (pool[r0:r0 + lay.rec_bytes] == 0).all()
