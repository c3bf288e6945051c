"""Planted mistakes in the oracle (CPU only) must be caught by its pins.

Each case patches one oracle function with a plausible bug and checks that a
pin test then fails.
"""
import numpy as np
import pytest

import oracle
import oracle.attention
import oracle.indexer
import oracle.topk
import oracle.store
import oracle.pipeline
from tests import test_oracle_attention as ta
from tests import test_oracle_indexer_topk as ti
from tests import test_oracle_layout_store as ts
from tests import test_oracle_dcp as td
import oracle.dcp


def _attend_no_rope(q, q_pe, lat, rope, sigma):
    return _orig_attend(q, 0 * q_pe, lat, rope, sigma)


def _attend_lse_log2(q, q_pe, lat, rope, sigma):
    out, lse = _orig_attend(q, q_pe, lat, rope, sigma)
    return out, lse / np.log(2)


def _topk_ties_high(scores_row, k):
    s = np.asarray(scores_row, dtype=np.float32)
    j = np.arange(s.size)
    order = np.lexsort((-j, -s.astype(np.float64)))
    out = np.full(k, -1, dtype=np.int32)
    keep = np.sort(order[:min(k, s.size)])
    out[:keep.size] = keep
    return out


_orig_attend = oracle.attention.attend
_orig_scores = oracle.indexer.index_scores_row


def _scores_no_relu(layout, pool, layer, q_codes, w, bt_row, p, chunk=1 << 17):
    n = int(p) + 1
    q = oracle.e4m3_decode(q_codes)
    slots = oracle.context_slots(bt_row, n, layout.block_size)
    keys, s = oracle.read_index_key(layout, pool, layer, slots)
    return ((np.asarray(w, np.float64)[:, None] * (q @ keys.T)).sum(0) * s).astype(np.float32)



_orig_lse_merge = oracle.dcp.lse_merge
_orig_topk_merge = oracle.dcp.topk_merge


def _lse_merge_unweighted(parts_out, parts_lse):
    out, lse = _orig_lse_merge(parts_out, parts_lse)
    return np.asarray(parts_out, np.float64).mean(axis=0), lse


def _lse_merge_max_only(parts_out, parts_lse):
    out, _ = _orig_lse_merge(parts_out, parts_lse)
    return out, np.asarray(parts_lse, np.float64).max(axis=0)


def _topk_merge_local_order(shard_scores, shard_topk, n_shards, k):
    # mistake: ties broken by shard first, then local position, instead of by global position
    glob, per = _orig_topk_merge(shard_scores, shard_topk, n_shards, k)
    cand = []
    for r in range(n_shards):
        loc = np.asarray(shard_topk[r], np.int64)
        loc = loc[loc >= 0]
        for i in loc:
            cand.append((-float(np.asarray(shard_scores[r], np.float32)[i]), r, int(i), int(i) * n_shards + r))
    cand.sort()
    keep = np.sort(np.array([c[3] for c in cand[:k]], dtype=np.int64))
    g = np.full(k, -1, dtype=np.int32)
    g[:keep.size] = keep
    return g, per


CASES = [
    ("merge without lse weights", oracle.dcp, "lse_merge", _lse_merge_unweighted,
     lambda: td.test_lse_merge_equals_attention_over_all_keys(3)),
    ("merged lse as the max", oracle.dcp, "lse_merge", _lse_merge_max_only,
     lambda: td.test_lse_merge_identity_and_empty_parts()),
    ("candidate ties by shard", oracle.dcp, "topk_merge", _topk_merge_local_order,
     lambda: td.test_topk_merge_equals_unsharded_topk(3, 300, 64)),
    ("attention drops rope", oracle.attention, "attend", _attend_no_rope,
     lambda: ta.test_attend_matches_torch_sdpa(64)),
    ("lse in log2", oracle.attention, "attend", _attend_lse_log2,
     lambda: ta.test_zero_query_gives_mean_and_log_n()),
    ("top-k ties to higher index", oracle.topk, "topk_select", _topk_ties_high,
     lambda: ti.test_topk_special_cases()),
    ("indexer without ReLU", oracle.indexer, "index_scores_row", _scores_no_relu,
     lambda: ti.test_scores_equal_integer_recomputation()),
]


@pytest.mark.parametrize("name,mod,attr,bad,pin", CASES, ids=[c[0] for c in CASES])
def test_pin_catches_planted_mistake(monkeypatch, name, mod, attr, bad, pin):
    monkeypatch.setattr(mod, attr, bad)
    for m in (oracle, oracle.pipeline, ta, ti, td.dcp):
        if hasattr(m, attr):
            monkeypatch.setattr(m, attr, bad, raising=False)
    with pytest.raises(AssertionError):
        pin()


def test_pin_catches_dequant_with_the_first_tile_scale(monkeypatch):
    def bad_read(layout, pool, layer, slots):
        lat, rope = orig(layout, pool, layer, slots)
        rec = oracle.store._offsets(layout, slots, layer, "record")[:, None]
        codes = pool[rec + np.arange(layout.d_latent)]
        s0 = np.ascontiguousarray(pool[rec + layout.d_latent + np.arange(4)]).view(np.float32)
        return (oracle.e4m3_decode(codes) * s0.astype(np.float64)).astype(np.float32).astype(np.float64), rope
    orig = oracle.store.read_record
    monkeypatch.setattr(oracle.store, "read_record", bad_read)
    monkeypatch.setattr(oracle, "read_record", bad_read)
    with pytest.raises(AssertionError):
        ts.test_full_record_round_trip_within_the_e4m3_bound()


def test_pin_catches_wrong_scale_rounding(monkeypatch):
    def bad_quant(latent_bits, quant_tile):
        codes, scale = orig(latent_bits, quant_tile)
        return codes, (scale * np.float32(1.0000001)).astype(np.float32)
    orig = oracle.store.quantize_latent
    monkeypatch.setattr(oracle.store, "quantize_latent", bad_quant)
    monkeypatch.setattr(ts, "quantize_latent", bad_quant)
    with pytest.raises(AssertionError):
        ts.test_quantize_matches_torch_fp32_route()
