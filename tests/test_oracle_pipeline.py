"""Whole-step invariants of the oracle (CPU only)."""
import numpy as np
import torch

import oracle
from paged_sparse_mla_gb300.workloads import TINY, build_workload, make_config
from tests.oracle_helpers import layout_of, npy, oracle_pool, oracle_step


def _same(a, b):
    assert a.keys() == b.keys()
    for t in a:
        for key in ("scores", "topk", "out", "lse"):
            assert np.array_equal(a[t][key], b[t][key]), (t, key)


def test_step_invariant_under_physical_block_permutation():
    wl = make_config(1)
    base = oracle_step(wl, oracle_pool(wl))
    perm = torch.as_tensor(np.random.default_rng(9).permutation(wl.num_blocks))
    bs = wl.dims.block_size
    wl2 = make_config(1)
    wl2.block_table = torch.where(wl.block_table >= 0, perm[wl.block_table.clamp(min=0).long()].int(), -1)
    slot_perm = (perm[:, None] * bs + torch.arange(bs)).reshape(-1)
    inv = torch.empty_like(slot_perm)
    inv[slot_perm] = torch.arange(slot_perm.numel())
    wl2.slot_mapping = slot_perm[wl.slot_mapping]
    wl2.cached_slots = slot_perm[wl.cached_slots]
    for name in ("slot_latent", "slot_rope", "slot_idx_k", "slot_idx_s"):
        setattr(wl2, name, getattr(wl, name)[inv])
    _same(base, oracle_step(wl2, oracle_pool(wl2)))


def test_prefix_sharing_equals_private_copies():
    wl = make_config(1)
    shared = oracle_step(wl, oracle_pool(wl))
    # give sequence 1 private copies of the 8 shared blocks (use the 8 slack blocks)
    used = set(npy(wl.block_table).ravel().tolist()) - {-1}
    free = [b for b in range(wl.num_blocks) if b not in used][:8]
    wl2 = make_config(1)
    bt = wl.block_table.clone()
    bs = wl.dims.block_size
    for i, fb in enumerate(free):
        old = int(bt[1, i])
        bt[1, i] = fb
        for name in ("slot_latent", "slot_rope", "slot_idx_k", "slot_idx_s"):
            getattr(wl2, name)[fb * bs:(fb + 1) * bs] = getattr(wl, name)[old * bs:(old + 1) * bs]
    wl2.block_table = bt
    extra = torch.as_tensor([fb * bs + o for fb in free for o in range(bs)], dtype=torch.int64)
    wl2.cached_slots = torch.cat([wl.cached_slots, extra])
    assert not set(npy(bt[0]).tolist()) & set(npy(bt[1]).tolist())
    _same(shared, oracle_step(wl2, oracle_pool(wl2)))


def test_mtp_queries_see_only_their_prefix():
    wl = build_workload("mtp", TINY, [90, 70], [4, 3], seed=21)
    lay = layout_of(wl)
    base = oracle_step(wl, oracle_pool(wl))
    assert [base[t]["pos"] for t in range(7)] == [86, 87, 88, 89, 67, 68, 69]
    # perturb the last new token of sequence 0 (position 89): only query 3 may change
    wl2 = build_workload("mtp", TINY, [90, 70], [4, 3], seed=21)
    wl2.new_idx_k[3] = torch.full_like(wl2.new_idx_k[3], 0x48)        # 4.0 everywhere
    wl2.new_latent[3] = 100.0
    pert = oracle_step(wl2, oracle_pool(wl2))
    for t in (0, 1, 2, 4, 5, 6):
        for key in ("scores", "topk", "out", "lse"):
            assert np.array_equal(base[t][key], pert[t][key]), (t, key)
    assert not np.array_equal(base[3]["scores"], pert[3]["scores"])


def test_topk_selection_drives_attention():
    """Replacing an unselected record leaves the output unchanged; a selected one changes it."""
    wl = make_config(1)
    pool = oracle_pool(wl)
    base = oracle_step(wl, pool.copy())
    lay = layout_of(wl)
    sel = set(base[0]["topk"].tolist())
    unsel = next(j for j in range(base[0]["pos"]) if j not in sel)
    chosen = next(iter(sel - {-1}))
    for j, should_change in ((unsel, False), (chosen, True)):
        p2 = pool.copy()
        slot = int(wl.block_table[0, j // lay.block_size]) * lay.block_size + j % lay.block_size
        r = lay.record_offset(slot, 0)
        p2[r:r + lay.d_latent] = 0x38                                   # latent codes -> 1.0
        res = oracle_step(wl, p2, rows=[0])
        assert np.array_equal(res[0]["topk"], base[0]["topk"])
        assert (not np.array_equal(res[0]["out"], base[0]["out"])) == should_change
