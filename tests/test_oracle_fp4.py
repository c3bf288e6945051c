"""Pins for the oracle's FP4 (E2M1) indexer keys: codec, packing, layout and scores (CPU only).

The codec is pinned to the MX specification's value table and to the (separately
pinned) E4M3 codec; the packing to a golden byte table; the layout to its closed
form; the scores to an int64 recomputation and to the E4M3 path on the same
key values.  Planted mistakes (nibble order, exponent bias) must fail them.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.fp4
import oracle.store
from paged_sparse_mla_gb300.workloads import make_config
from tests.oracle_helpers import bits, layout_of, npy, oracle_pool

HERE = os.path.dirname(__file__)


def _golden(name, cols):
    rows = []
    for line in open(os.path.join(HERE, "golden", name)):
        line = line.strip()
        if line and not line.startswith("#"):
            parts = line.split()
            rows.append((int(parts[0], 16), *[float(v) for v in parts[1:1 + cols]]))
    return rows


def _spec_table():
    """code -> value from the spec's table (independent of the oracle's decoder)."""
    t = np.zeros(16, np.float64)
    for code, val in _golden("e2m1_spec_values.txt", 1):
        t[code] = val
    return t


def test_decode_matches_spec_values():
    rows = _golden("e2m1_spec_values.txt", 1)
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1_decode(np.uint8(code))
        assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_every_e2m1_value_is_an_e4m3_value():
    """FP4 keys lose nothing when held as E4M3: every E2M1 value round-trips through the E4M3 codec."""
    v = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    back = oracle.e4m3_decode(oracle.e4m3_encode(v.astype(np.float32)))
    assert np.array_equal(back, v) and np.array_equal(np.signbit(back), np.signbit(v))


def test_encode_round_trip_every_code():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(oracle.e2m1_encode(oracle.e2m1_decode(codes)), codes)


@pytest.mark.parametrize("x,code", [
    (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4),   # halfway: to the even mantissa bit
    (2.5, 0x4), (3.5, 0x6), (5.0, 0x6), (-5.0, 0xE),
    (6.5, 0x7), (1e9, 0x7), (-1e9, 0xF), (float("inf"), 0x7),  # saturate to +-6
    (-0.1, 0x8),                                            # rounds to zero, keeps the sign
])
def test_encode_ties_and_saturation(x, code):
    assert int(oracle.e2m1_encode(x)) == code


def test_encode_is_nearest():
    rng = np.random.default_rng(3)
    x = rng.uniform(-6.5, 6.5, size=20_000)
    got = oracle.e2m1_decode(oracle.e2m1_encode(x))
    table = _spec_table()
    best = np.abs(x[:, None] - table[None, :]).min(axis=1)    # distance to the nearest E2M1 value
    assert np.array_equal(np.abs(x - got), best)


def test_packing_matches_golden_bytes():
    table = _spec_table()
    for byte, first, second in _golden("e2m1_packing.txt", 2):
        codes = oracle.e2m1_unpack(np.array([[byte]], np.uint8))[0]
        vals = table[codes]
        assert vals[0] == first and vals[1] == second and np.signbit(vals[1]) == np.signbit(second), hex(byte)
        assert int(oracle.e2m1_pack(codes[None, :])[0, 0]) == byte


def test_fp4_layout_closed_form():
    """DeepSeek shape, one layer: 64 keys x 64 packed bytes after the 41,984 record bytes."""
    e4 = oracle.PoolLayout(64, 1, 512, 64, 128, 128, 10)
    f4 = oracle.PoolLayout(64, 1, 512, 64, 128, 128, 10, "e2m1")
    assert f4.key_bytes == 64 and e4.key_bytes == 128
    assert f4.idx_key_off == 41984 and f4.idx_scale_off == 41984 + 64 * 64 and f4.block_stride == 46336
    assert e4.block_stride == 50432
    # per token: 656 + 64 + 4 instead of 656 + 128 + 4 bytes, 8.1% of the block
    assert abs(1 - f4.block_stride / e4.block_stride - 0.0812) < 1e-3
    for n_layers in (1, 2, 3):
        lo = oracle.PoolLayout(16, n_layers, 64, 16, 64, 32, 5, "e2m1")
        assert lo.idx_key_off % 256 == 0 and lo.idx_scale_off % 256 == 0 and lo.layer_stride % 256 == 0
        assert lo.idx_key_off >= lo.block_size * lo.rec_stride
        assert lo.idx_scale_off >= lo.idx_key_off + lo.block_size * 16
        assert lo.layer_stride >= lo.idx_scale_off + 4 * lo.block_size


def _fp4_setup(scale=0.004, cfg=2):
    wl = make_config(cfg, scale=scale, key_format="e2m1")
    lay = layout_of(wl)
    pool = oracle_pool(wl)
    oracle.kvpack_store(lay, pool, 0, bits(wl.new_latent), bits(wl.new_rope), npy(wl.new_idx_k),
                        npy(wl.new_idx_s), npy(wl.slot_mapping))
    return wl, lay, pool


def test_fp4_scores_equal_integer_recomputation():
    """8*I = sum_h (4 w_h) * max(0, q_h . (2 k)) exactly in int64, with k decoded through the spec table
    and the packing golden rule (element 2i = low nibble)."""
    wl, lay, pool = _fp4_setup()
    table2 = (_spec_table() * 2).astype(np.int64)                       # every E2M1 value x2 is an integer
    src = npy(wl.slot_idx_k).copy()
    src[npy(wl.slot_mapping)] = npy(wl.new_idx_k)
    q = wl.q_idx.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(q, np.round(q))
    q = q.astype(np.int64)
    w4 = (npy(wl.w) * 4).astype(np.int64)
    seqs, pos = oracle.query_positions(npy(wl.seq_lens), npy(wl.query_start_loc))
    for t in range(len(seqs)):
        b, p = seqs[t], pos[t]
        got = oracle.index_scores_row(lay, pool, 0, npy(wl.q_idx[t]), npy(wl.w[t]), npy(wl.block_table[b]), p)
        slots = oracle.context_slots(npy(wl.block_table[b]), p + 1, lay.block_size)
        packed = src[slots]
        k2 = np.empty((packed.shape[0], 2 * packed.shape[1]), np.int64)
        k2[:, 0::2] = table2[packed & 0xF]
        k2[:, 1::2] = table2[packed >> 4]
        ref8 = (w4[t][:, None] * np.maximum(q[t] @ k2.T, 0)).sum(axis=0)
        assert np.array_equal(got.astype(np.float64) * 8, ref8.astype(np.float64)), f"row {t}"


def test_fp4_scores_equal_e4m3_scores_of_the_same_key_values():
    """Storing the same key values as E4M3 (torch's own fp8 cast) in an E4M3 layout gives identical
    scores: the FP4 path reduces to the pinned FP8 one."""
    wl, lay, pool = _fp4_setup(scale=0.003)
    table = _spec_table()
    vals = lambda packed: np.stack([table[packed & 0xF], table[packed >> 4]], axis=-1).reshape(packed.shape[0], -1)
    as_e4m3 = lambda packed: torch.from_numpy(vals(npy(packed)).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    lay8 = oracle.PoolLayout(lay.block_size, lay.n_layers, lay.d_latent, lay.d_rope, lay.quant_tile, lay.d_index,
                             lay.num_blocks)
    pool8 = np.zeros(lay8.pool_bytes, np.uint8)
    sc = npy(wl.cached_slots)
    oracle.kvpack_store(lay8, pool8, 0, bits(wl.slot_latent[wl.cached_slots]), bits(wl.slot_rope[wl.cached_slots]),
                        as_e4m3(wl.slot_idx_k[wl.cached_slots]), npy(wl.slot_idx_s[wl.cached_slots]), sc)
    oracle.kvpack_store(lay8, pool8, 0, bits(wl.new_latent), bits(wl.new_rope), as_e4m3(wl.new_idx_k),
                        npy(wl.new_idx_s), npy(wl.slot_mapping))
    seqs, pos = oracle.query_positions(npy(wl.seq_lens), npy(wl.query_start_loc))
    for t in range(len(seqs)):
        b, p = seqs[t], pos[t]
        a = oracle.index_scores_row(lay, pool, 0, npy(wl.q_idx[t]), npy(wl.w[t]), npy(wl.block_table[b]), p)
        c = oracle.index_scores_row(lay8, pool8, 0, npy(wl.q_idx[t]), npy(wl.w[t]), npy(wl.block_table[b]), p)
        assert np.array_equal(a, c), f"row {t}"
    # the two pools hold the same records; only the key region (and so the block stride) differs
    assert lay.block_stride < lay8.block_stride


def test_fp4_store_copies_packed_keys_verbatim():
    wl, lay, pool = _fp4_setup(scale=0.002)
    sm = npy(wl.slot_mapping)
    for i, slot in enumerate(sm):
        off = lay.index_key_offset(int(slot), 0)
        assert np.array_equal(pool[off:off + lay.key_bytes], npy(wl.new_idx_k[i]))


def test_fp4_whole_step_runs_and_selects():
    """The oracle's whole step on an FP4-key layout: scores, an exact top-k and attention."""
    wl, lay, pool = _fp4_setup(scale=0.003, cfg=3)
    ref = oracle.decode_step(lay, pool, 0, latent_new=bits(wl.new_latent), rope_new=bits(wl.new_rope),
                             idxk_new=npy(wl.new_idx_k), idxs_new=npy(wl.new_idx_s),
                             slot_mapping=npy(wl.slot_mapping), q=bits(wl.q), q_pe=bits(wl.q_pe),
                             q_idx=npy(wl.q_idx), w=npy(wl.w), block_table=npy(wl.block_table),
                             seq_lens=npy(wl.seq_lens), query_start_loc=npy(wl.query_start_loc),
                             top_k=wl.dims.top_k, sigma=wl.dims.softmax_scale, rows=[0, 5], store=False)
    for t, r in ref.items():
        assert r["scores"].size == r["pos"] + 1
        assert np.array_equal(r["topk"], oracle.topk_select(r["scores"], wl.dims.top_k))
        assert np.isfinite(r["lse"]).all()


# ---------------------------------------------------------------- planted mistakes

def _unpack_high_first(packed):
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b >> 4
    out[..., 1::2] = b & 0x0F
    return out


def _decode_bias0(codes):
    c = np.asarray(codes, dtype=np.uint8)
    e = (c >> 1) & 3
    m = c & 1
    s = np.where(c & 8, -1.0, 1.0)
    return s * np.where(e == 0, m / 2.0, 2.0 ** e * (1 + m / 2.0))


def test_planted_nibble_order_is_caught(monkeypatch):
    monkeypatch.setattr(oracle.store, "e2m1_unpack", _unpack_high_first)
    monkeypatch.setattr(oracle, "e2m1_unpack", _unpack_high_first)
    with pytest.raises(AssertionError):
        test_packing_matches_golden_bytes()
    with pytest.raises(AssertionError):
        test_fp4_scores_equal_integer_recomputation()


def test_planted_exponent_bias_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "e2m1_decode", _decode_bias0)
    monkeypatch.setattr(oracle.store, "e2m1_decode", _decode_bias0)
    with pytest.raises(AssertionError):
        test_decode_matches_spec_values()
    with pytest.raises(AssertionError):
        test_fp4_scores_equal_integer_recomputation()
