"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Bit-exact: pool bytes after the store, indexer scores (integer-valued FP8
inputs make every fp32 partial sum exact), top-k indices.  Attention: max
|err| <= 2e-2 and mean |err| <= 2e-3 on out and lse against the float64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300.workloads import FULL, TINY, build_workload, make_config
from tests.oracle_helpers import bits, layout_of, npy, oracle_pool, oracle_step, sequence_slots
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


def _small_cases():
    return {
        "tiny": lambda: make_config(1),
        "decode-b32-scaled": lambda: make_config(2, scale=0.1),
        "agentic-mtp-scaled": lambda: make_config(3, scale=0.02),
        "longctx-scaled": lambda: make_config(4, scale=0.004),
        "prefill-scaled": lambda: make_config(5, scale=1 / 64),
        "short-contexts-tiny": lambda: build_workload("short", TINY, [1, 2, 17, 64, 65, 100, 16], [1, 1, 2, 1, 3, 4, 1],
                                                      seed=31, slack_blocks=3),
        "short-contexts-full": lambda: build_workload("shortf", FULL, [1, 5, 2048, 2049, 2177, 4100], [1, 1, 1, 4, 2, 3],
                                                      seed=32, slack_blocks=5),
        "pow2-key-scales": lambda: build_workload("pow2", FULL, [3000, 700], [2, 1], seed=33,
                                                  idx_scale=[0.5, 1.0, 2.0, 4.0]),
    }


CASES = _small_cases()


def _compare_all(wl, res_gpu, res_ref, what):
    seqs, pos = oracle.query_positions(npy(wl.seq_lens), npy(wl.query_start_loc))
    for t in range(wl.n_tokens):
        r = res_ref[t]
        n = r["pos"] + 1
        if "scores" in res_gpu:
            assert np.array_equal(G.canon(res_gpu["scores"][t, :n]), G.canon(r["scores"])), f"{what} scores row {t}"
        assert np.array_equal(res_gpu["topk"][t], r["topk"]), f"{what} topk row {t}"
    out_ref = np.stack([res_ref[t]["out"] for t in range(wl.n_tokens)])
    lse_ref = np.stack([res_ref[t]["lse"] for t in range(wl.n_tokens)])
    G.assert_attention_close(res_gpu["out"], res_gpu["lse"], out_ref, lse_ref, what)


@pytest.mark.parametrize("name", list(CASES))
def test_stages_match_oracle(name):
    wl = CASES[name]()
    ref_pool = oracle_pool(wl)
    ref = oracle_step(wl, ref_pool)                     # also stores the new tokens into ref_pool
    g = G.cuda_wl(CASES[name]())
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    res = G.run_stages(g, pool, lay, prm)
    assert res["err"] == 0
    assert np.array_equal(pool.cpu().numpy(), ref_pool), f"{name}: pool bytes differ after the store"
    _compare_all(wl, res, ref, name)


@pytest.mark.parametrize("name", ["tiny", "agentic-mtp-scaled", "prefill-scaled", "short-contexts-full"])
def test_fused_decode_equals_stages(name):
    g = G.cuda_wl(CASES[name]())
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    a = G.run_stages(g, G.gpu_pool(g, lay), lay, prm)
    b = G.run_decode(g, G.gpu_pool(g, lay), lay, prm)
    assert a["err"] == 0 and b["err"] == 0
    assert np.array_equal(a["topk"], b["topk"])
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


def test_prefill_chunk_matches_oracle_and_decode():
    """smla_prefill_chunk: a causal chunk on a cached prefix, checked against the oracle and smla_decode."""
    wl = CASES["prefill-scaled"]()
    ref_pool = oracle_pool(wl)
    ref = oracle_step(wl, ref_pool)
    g = G.cuda_wl(CASES["prefill-scaled"]())
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    d = g.dims
    T = g.n_tokens
    ws = torch.empty(smla.workspace_size(lay, prm, T, g.max_ctx), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    topk = torch.empty((T, prm.top_k), dtype=torch.int32, device="cuda")
    smla.smla_prefill_chunk(lay, prm, pool, 0, g.new_latent, g.new_rope, g.new_idx_k, g.new_idx_s, g.slot_mapping, g.q,
                            g.q_pe, g.q_idx, g.w, g.block_table, g.seq_lens, g.query_start_loc, g.max_q, g.max_ctx,
                            out, lse, ws, topk_idx_out=topk)
    assert smla.smla_get_last_error() == 0
    assert np.array_equal(pool.cpu().numpy(), ref_pool)
    res = dict(topk=topk.cpu().numpy(), out=out.float().cpu().numpy(), lse=lse.cpu().numpy())
    _compare_all(wl, res, ref, "prefill_chunk")
    b = G.run_decode(g, G.gpu_pool(g, lay), lay, prm)
    assert np.array_equal(res["topk"], b["topk"]) and np.array_equal(res["out"], b["out"])


def test_sparse_equals_dense_when_topk_covers_context():
    """Prompts inside the top-k take the sparse kernel; it must reproduce dense attention."""
    wl = make_config(1)
    ref_pool = oracle_pool(wl)
    ref = oracle_step(wl, ref_pool, top_k=256)
    lay_o = layout_of(wl)
    g = G.cuda_wl(make_config(1))
    lay, prm = G.gpu_layout(g), G.gpu_params(g, top_k=256)
    res = G.run_decode(g, G.gpu_pool(g, lay), lay, prm)
    assert res["err"] == 0
    for t, r in ref.items():
        out_d, lse_d = oracle.dense_attend(lay_o, ref_pool, 0, oracle.bf16_bits_to_f64(bits(wl.q[t])),
                                           oracle.bf16_bits_to_f64(bits(wl.q_pe[t])), npy(wl.block_table[r["seq"]]),
                                           r["pos"], wl.dims.softmax_scale)
        assert (res["topk"][t] >= 0).sum() == r["pos"] + 1
        G.assert_attention_close(res["out"][t], res["lse"][t], out_d, lse_d, f"dense row {t}")


def test_block_permutation_gives_identical_outputs():
    base = G.cuda_wl(make_config(2, scale=0.05))
    lay, prm = G.gpu_layout(base), G.gpu_params(base)
    a = G.run_decode(base, G.gpu_pool(base, lay), lay, prm)
    perm = torch.as_tensor(np.random.default_rng(5).permutation(base.num_blocks), device="cuda")
    bs = base.dims.block_size
    moved = G.cuda_wl(make_config(2, scale=0.05))
    moved.block_table = torch.where(base.block_table >= 0, perm[base.block_table.clamp(min=0).long()].int(), -1)
    slot_perm = (perm[:, None] * bs + torch.arange(bs, device="cuda")).reshape(-1)
    inv = torch.empty_like(slot_perm)
    inv[slot_perm] = torch.arange(slot_perm.numel(), device="cuda")
    moved.slot_mapping = slot_perm[base.slot_mapping]
    moved.cached_slots = slot_perm[base.cached_slots]
    for name in ("slot_latent", "slot_rope", "slot_idx_k", "slot_idx_s"):
        setattr(moved, name, getattr(base, name)[inv])
    b = G.run_decode(moved, G.gpu_pool(moved, lay), lay, prm)
    assert a["err"] == 0 and b["err"] == 0
    assert np.array_equal(a["topk"], b["topk"])
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


def test_prefix_sharing_equals_private_copies():
    base = G.cuda_wl(make_config(1))
    lay, prm = G.gpu_layout(base), G.gpu_params(base)
    a = G.run_decode(base, G.gpu_pool(base, lay), lay, prm)
    priv = G.cuda_wl(make_config(1))
    used = set(npy(base.block_table).ravel().tolist()) - {-1}
    free = [x for x in range(base.num_blocks) if x not in used][:8]
    bs = base.dims.block_size
    bt = base.block_table.clone()
    for i, fb in enumerate(free):
        old = int(bt[1, i])
        bt[1, i] = fb
        for name in ("slot_latent", "slot_rope", "slot_idx_k", "slot_idx_s"):
            getattr(priv, name)[fb * bs:(fb + 1) * bs] = getattr(base, name)[old * bs:(old + 1) * bs]
    priv.block_table = bt
    extra = torch.as_tensor([fb * bs + o for fb in free for o in range(bs)], dtype=torch.int64, device="cuda")
    priv.cached_slots = torch.cat([base.cached_slots, extra])
    b = G.run_decode(priv, G.gpu_pool(priv, lay), lay, prm)
    assert np.array_equal(a["topk"], b["topk"])
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


def test_all_equal_scores_select_first_positions():
    g = G.cuda_wl(build_workload("eq", FULL, [5000, 3000], [1, 2], seed=41))
    g.q_idx.zero_()
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    res = G.run_stages(g, G.gpu_pool(g, lay), lay, prm)
    assert res["err"] == 0
    for t in range(g.n_tokens):
        assert list(res["topk"][t]) == list(range(2048))


def test_single_position_returns_its_record():
    g = G.cuda_wl(build_workload("one", FULL, [1, 1], [1, 1], seed=42))
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    res = G.run_decode(g, G.gpu_pool(g, lay), lay, prm)
    assert res["err"] == 0
    lo = layout_of(g)
    ref_pool = np.zeros(lo.pool_bytes, np.uint8)
    oracle.kvpack_store(lo, ref_pool, 0, bits(g.new_latent), bits(g.new_rope), npy(g.new_idx_k), npy(g.new_idx_s),
                        npy(g.slot_mapping))
    lat, _ = oracle.read_record(lo, ref_pool, 0, npy(g.slot_mapping))
    for t in range(2):
        assert list(res["topk"][t][:2]) == [0, -1]
        e = np.abs(res["out"][t] - lat[t][None, :])
        assert e.max() <= G.MAX_ERR


def test_bad_block_id_is_reported_not_faulted():
    g = G.cuda_wl(make_config(1))
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    g.block_table[0, 3] = g.num_blocks + 7        # out of the pool
    res = G.run_stages(g, pool, lay, prm, store=False)
    assert res["err"] == 4                          # SMLA_ERR_BAD_INDEX
    assert G.smla.smla_get_last_error() == 0        # cleared by the read


def test_position_past_the_block_table_row_is_reported_not_read():
    """A caller-supplied top-k entry at or beyond bt_stride * block_size has no block-table entry:
    the attention latches SMLA_ERR_BAD_INDEX and treats its record as zeros, and the other rows
    are unaffected."""
    g = G.cuda_wl(make_config(1))
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    base = G.run_stages(g, pool, lay, prm, store=False)
    assert base["err"] == 0
    topk = torch.as_tensor(base["topk"], device="cuda")
    bad = topk.clone()
    bad[0, 0] = g.block_table.shape[1] * g.dims.block_size + 3      # past the last block-table column
    T, d = g.n_tokens, g.dims
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    smla.smla_attend(lay, prm, pool, 0, g.q, g.q_pe, bad, g.block_table, g.query_start_loc, out, lse)
    assert smla.smla_get_last_error() == 4                          # SMLA_ERR_BAD_INDEX
    o = out.float().cpu().numpy()
    assert np.array_equal(o[1:], base["out"][1:])                   # other rows untouched


def test_wait_that_never_completes_times_out_and_context_survives():
    """A bounded wait on an mbarrier nothing arrives at gives up, reports SMLA_ERR_TIMEOUT and returns."""
    import time
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    G.smla.smla_selftest_wait(50_000_000)           # 50 ms
    assert G.smla.smla_get_last_error() == 5        # SMLA_ERR_TIMEOUT, read and cleared
    assert time.perf_counter() - t0 >= 0.05
    assert G.smla.smla_get_last_error() == 0
    # the context still runs the path, with the oracle's result
    wl = make_config(1)
    ref = oracle_step(wl, oracle_pool(wl))
    g = G.cuda_wl(make_config(1))
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    res = G.run_decode(g, G.gpu_pool(g, lay), lay, prm)
    assert res["err"] == 0
    for t in range(g.n_tokens):
        assert np.array_equal(res["topk"][t], ref[t]["topk"])


@pytest.mark.parametrize("lens", [[20000, 9000, 300, 1], [70000, 40000, 33000, 24000, 15000, 8200, 4097, 2049]])
def test_split_attention_matches_oracle_and_one_cta_path(lens):
    """Few query tokens and a scratch: each token's selection is split into contiguous ranges over
    CTAs (short rows leave empty ranges), the fp32 partials are merged by their lse.  Within the
    attention tolerance of the oracle, and close to the one-CTA-per-token path."""
    wl = build_workload("split", FULL, lens, [1] * len(lens), seed=93, slack_blocks=2)
    ref = oracle_step(wl, oracle_pool(wl))
    g = G.cuda_wl(build_workload("split", FULL, lens, [1] * len(lens), seed=93, slack_blocks=2))
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    res = G.run_stages(g, pool, lay, prm, split=False)    # one CTA per token (no scratch)
    assert res["err"] == 0
    T, d = g.n_tokens, g.dims
    topk = torch.as_tensor(res["topk"], device="cuda")
    ws = torch.empty(smla.attend_workspace_size(lay, prm, T), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    smla.smla_attend(lay, prm, pool, 0, g.q, g.q_pe, topk, g.block_table, g.query_start_loc, out, lse, workspace=ws)
    assert smla.smla_get_last_error() == 0
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    out_ref = np.stack([ref[t]["out"] for t in range(T)])
    lse_ref = np.stack([ref[t]["lse"] for t in range(T)])
    G.assert_attention_close(o, l, out_ref, lse_ref, "split")
    # the two paths round differently (bf16 probabilities summed per tile vs fp32 partials merged
    # by lse); both are held to the oracle above, and to each other well inside that tolerance
    assert np.abs(l - res["lse"]).max() <= 1e-3
    assert np.abs(o - res["out"]).max() <= 1e-2


@pytest.mark.parametrize("n_rows", [160, 200])
def test_balanced_attention_matches_oracle_and_one_cta_path(n_rows):
    """More rows than SMs with a short last round (on 152 SMs: 8 or 48 rows): with a scratch every
    CTA takes the same number of tiles, a row that straddles two CTAs is finished from two partials
    merged by their lse.  Ragged rows (contexts below k leave empty tiles, and some parts empty) must match the
    oracle, and the one-CTA-per-row path within the attention tolerance."""
    rng = np.random.default_rng(95 + n_rows)
    lens = rng.choice([1, 7, 100, 1500, 2048, 2049, 3000, 6000, 9000], size=n_rows).tolist()
    wl = build_workload("bal", FULL, lens, [1] * n_rows, seed=96, slack_blocks=2)
    ref = oracle_step(wl, oracle_pool(wl))
    g = G.cuda_wl(build_workload("bal", FULL, lens, [1] * n_rows, seed=96, slack_blocks=2))
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    res = G.run_stages(g, pool, lay, prm, split=False)      # one CTA per row (no scratch)
    assert res["err"] == 0
    T, d = g.n_tokens, g.dims
    topk = torch.as_tensor(res["topk"], device="cuda")
    ws = torch.empty(smla.attend_workspace_size(lay, prm, T), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    smla.smla_attend(lay, prm, pool, 0, g.q, g.q_pe, topk, g.block_table, g.query_start_loc, out, lse, workspace=ws)
    assert smla.smla_get_last_error() == 0
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    for t in range(T):
        assert np.array_equal(res["topk"][t], ref[t]["topk"]), f"topk row {t}"
    out_ref = np.stack([ref[t]["out"] for t in range(T)])
    lse_ref = np.stack([ref[t]["lse"] for t in range(T)])
    G.assert_attention_close(o, l, out_ref, lse_ref, "balanced")
    assert np.abs(l - res["lse"]).max() <= 1e-3
    assert np.abs(o - res["out"]).max() <= 1e-2


@pytest.mark.parametrize("lens", [[140000, 61000, 30000, 9000], [300000], [200000, 150000, 5000, 1, 3000]])
def test_topk_rows_split_into_segments(lens):
    """Few long rows and a scratch: each row's segments are selected on their own CTAs and the
    candidates merged.  Heavy ties (across segment boundaries too): every row equals the oracle's."""
    rng = np.random.default_rng(97 + len(lens))
    R, L, k = len(lens), max(lens), 2048
    stride = (L + 3) // 4 * 4
    scores = rng.integers(-60, 61, size=(R, stride)).astype(np.float32) * np.float32(0.25)
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qsl = torch.arange(R + 1, dtype=torch.int32, device="cuda")
    prm = smla.make_params(64, 64, k, 1.0)
    ws = torch.empty(smla.topk_workspace_size(prm, R), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    out = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    smla.smla_topk(prm, torch.as_tensor(scores, device="cuda"), seq_lens, qsl, out, workspace=ws)
    assert smla.smla_get_last_error() == 0
    got = out.cpu().numpy()
    for t in range(R):
        assert np.array_equal(got[t], oracle.topk_select(scores[t, :lens[t]], k)), f"row {t}"


def test_topk_more_rows_than_one_wave():
    """1,000 causal rows of one sequence: the top-k grid is one resident wave and each CTA takes
    a front row and a back row in alternate passes; every row must still equal the oracle's."""
    rng = np.random.default_rng(91)
    R, L, k = 1000, 12000, 2048
    stride = L
    scores = (rng.integers(-40, 41, size=(R, stride)).astype(np.float32) * np.float32(0.5))
    seq_lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    qsl = torch.tensor([0, R], dtype=torch.int32, device="cuda")
    prm = smla.make_params(64, 64, k, 1.0)
    out = torch.full((R, k), -7, dtype=torch.int32, device="cuda")
    smla.smla_topk(prm, torch.as_tensor(scores, device="cuda"), seq_lens, qsl, out)
    assert smla.smla_get_last_error() == 0
    got = out.cpu().numpy()
    for t in range(R):
        n = L - R + t + 1
        assert np.array_equal(got[t], oracle.topk_select(scores[t, :n], k)), f"row {t}"


def test_bad_slot_is_reported_and_skipped():
    g = G.cuda_wl(make_config(1))
    lay = G.gpu_layout(g)
    pool = torch.zeros(lay.pool_bytes, dtype=torch.uint8, device="cuda")
    sm = g.slot_mapping.clone()
    sm[0] = g.num_blocks * g.dims.block_size       # one past the pool
    G.smla.kvpack_store(lay, pool, 0, g.new_latent, g.new_rope, g.new_idx_k, g.new_idx_s, sm)
    assert G.smla.smla_get_last_error() == 4
    assert int(pool.count_nonzero()) > 0           # the valid token was still stored


def test_two_layers_are_independent():
    wl = make_config(1)
    d = wl.dims
    g = G.cuda_wl(make_config(1))
    lay = G.smla.layout_init(d.block_size, 2, d.d_latent, d.d_rope, d.quant_tile, d.d_index, g.num_blocks)
    prm = G.gpu_params(g)
    pool = torch.zeros(lay.pool_bytes, dtype=torch.uint8, device="cuda")
    s = g.cached_slots
    for layer in (0, 1):
        G.smla.kvpack_store(lay, pool, layer, g.slot_latent[s].contiguous(), g.slot_rope[s].contiguous(),
                            g.slot_idx_k[s].contiguous(), g.slot_idx_s[s].contiguous(), s)
    lo = oracle.PoolLayout(d.block_size, 2, d.d_latent, d.d_rope, d.quant_tile, d.d_index, wl.num_blocks)
    ref = np.zeros(lo.pool_bytes, np.uint8)
    for layer in (0, 1):
        sc = npy(wl.cached_slots)
        oracle.kvpack_store(lo, ref, layer, bits(wl.slot_latent[sc]), bits(wl.slot_rope[sc]), npy(wl.slot_idx_k[sc]),
                            npy(wl.slot_idx_s[sc]), sc)
    assert np.array_equal(pool.cpu().numpy(), ref)
    r1 = G.run_stages(g, pool, lay, prm, layer=1)
    ref_pool1 = oracle_pool(wl)
    ref1 = oracle_step(wl, ref_pool1)
    _compare_all(wl, r1, ref1, "layer 1")
