"""The seeded input recipe: shapes, length mixes and prefix sharing of the five workloads.

The recipe stands in for the pages' traces: uniform 8K-32K decode contexts,
an agentic prefix tree (lognormal lengths around 142K, forked children that
share at least 96% of their parent's blocks), 1M-token contexts and a 131K
prefix with an 8K prefill chunk.  These checks run on metadata and on scaled
copies, so they need neither a GPU nor the full-size tensors.
"""
import numpy as np
import pytest

from paged_sparse_mla_gb300.workloads import FULL, TINY, agentic_tree, build_workload, make_config


def test_agentic_tree_shape_and_sharing():
    lens, share = agentic_tree(2)
    assert len(lens) == 64
    parents = [b for b, (p, _) in enumerate(share) if p < 0]
    assert len(parents) == 13
    kids = {p: sum(1 for q, _ in share if q == p) for p in parents}
    assert min(kids.values()) >= 1
    for b, (p, ns) in enumerate(share):
        if p < 0:
            assert 16_384 <= lens[b] <= 262_144
            continue
        assert p < b and share[p][0] < 0                  # children fork from parents
        assert lens[p] <= lens[b] <= lens[p] * 1.04 + 1
        # the shared blocks cover at least 96% of the child's tokens, to within the two partial blocks
        assert ns * 64 >= 0.96 * lens[b] - 2 * 64, (b, ns, lens[b])
        assert ns * 64 <= lens[p] - 4 and ns * 64 <= lens[b] - 4  # never a block holding new tokens
    med = float(np.median([lens[b] for b in parents]))
    assert 80_000 < med < 250_000                          # lognormal around 142K (13 draws)


def test_agentic_tree_is_seeded():
    assert agentic_tree(2) == agentic_tree(2)
    assert agentic_tree(2) != agentic_tree(3)


def test_tiny_workload_shares_eight_blocks():
    wl = make_config(1)
    bt = wl.block_table.numpy()
    assert wl.batch == 2 and wl.n_tokens == 2 and wl.num_blocks == 32
    assert list(wl.seq_lens.numpy()) == [256, 256]
    assert np.array_equal(bt[0, :8], bt[1, :8]) and not np.intersect1d(bt[0, 8:], bt[1, 8:]).size
    assert wl.dims == TINY


def test_scaled_workloads_keep_their_structure():
    wl = make_config(2, scale=0.01)
    assert wl.batch == 32 and wl.max_q == 1 and wl.dims == FULL
    wl = make_config(3, scale=0.01)
    assert wl.batch == 64 and wl.max_q == 4 and wl.n_tokens == 256
    wl = make_config(4, scale=0.001)
    assert wl.batch == 8 and len(set(wl.seq_lens.numpy().tolist())) == 1
    wl = make_config(5, scale=0.01)
    assert wl.batch == 1 and wl.n_tokens == 81 and int(wl.seq_lens[0]) == 1310 + 81


def test_full_size_decode_workload():
    wl = make_config(2)
    lens = wl.seq_lens.numpy()
    assert wl.batch == 32 and lens.min() >= 8192 and lens.max() <= 32768 and wl.max_ctx == lens.max()
    bt = wl.block_table.numpy()
    used = bt[bt >= 0]
    assert used.size == np.unique(used).size == wl.num_blocks  # no sharing; ids a permutation of the pool
    assert not np.array_equal(used, np.sort(used))


def test_block_ids_are_a_permutation_and_new_slots_are_free():
    lens, share = agentic_tree(2, ctx_scale=0.01)
    wl = build_workload("a", FULL, lens, [4] * len(lens), seed=2, share=share)
    bt = wl.block_table.numpy()
    used = np.unique(bt[bt >= 0])
    assert used.min() >= 0 and used.max() < wl.num_blocks
    assert used.size == wl.num_blocks                      # every pool block belongs to some sequence
    assert not np.isin(wl.slot_mapping.numpy(), wl.cached_slots.numpy()).any()
    assert np.array_equal(np.sort(wl.slot_mapping.numpy()), np.unique(wl.slot_mapping.numpy()))


def test_softmax_scales():
    # the tiny workload's text fixes 1/sqrt(80); the DeepSeek shape takes 1/sqrt(D_L + D_R) = 1/sqrt(576)
    assert TINY.softmax_scale == pytest.approx(80 ** -0.5, rel=1e-15)
    assert FULL.softmax_scale == pytest.approx(576 ** -0.5, rel=1e-15)
