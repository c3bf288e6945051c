"""GPU parity of the host-tier record gather (smla_attend_hisparse).

The records of a random part of the blocks are moved to a pinned host buffer
and wiped from the HBM pool (the indexer keys stay); attention over the same
selection must then give exactly the all-HBM result, and the oracle's within
the attention tolerance.  A map entry past the host buffer is reported, not
dereferenced.
"""
import numpy as np
import pytest
import torch

import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300.workloads import make_config
from tests.oracle_helpers import oracle_pool, oracle_step
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


def _evict(pool, lay, blocks):
    """Move the record regions of `blocks` (every layer) to a pinned host buffer; zero them in the pool."""
    per_layer = lay.block_size * lay.rec_stride
    host = torch.empty(len(blocks) * lay.n_layers * per_layer, dtype=torch.uint8).pin_memory()
    hmap = torch.full((lay.num_blocks,), -1, dtype=torch.int32)
    for h, b in enumerate(blocks):
        hmap[b] = h
        for layer in range(lay.n_layers):
            off = b * lay.block_stride + layer * lay.layer_stride + lay.rec_off
            dst = (h * lay.n_layers + layer) * per_layer
            host[dst:dst + per_layer].copy_(pool[off:off + per_layer].cpu())
            pool[off:off + per_layer] = 0
    return host, hmap.cuda()


def _attend(g, lay, prm, pool, topk, host=None, hmap=None):
    d = g.dims
    T = g.n_tokens
    out = torch.empty((T, d.n_heads, d.d_latent), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, d.n_heads), dtype=torch.float32, device="cuda")
    if host is None:
        smla.smla_attend(lay, prm, pool, 0, g.q, g.q_pe, topk, g.block_table, g.query_start_loc, out, lse)
    else:
        smla.smla_attend_hisparse(lay, prm, pool, 0, host, hmap, g.q, g.q_pe, topk, g.block_table,
                                  g.query_start_loc, out, lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), smla.smla_get_last_error()


@pytest.mark.parametrize("name,factory,frac", [
    ("tiny", lambda: make_config(1), 0.5),
    ("agentic-mtp-scaled", lambda: make_config(3, scale=0.02), 0.5),
    ("agentic-mtp-scaled-all-host", lambda: make_config(3, scale=0.02), 1.0),
])
def test_host_tier_equals_hbm_and_oracle(name, factory, frac):
    wl = factory()
    ref = oracle_step(wl, oracle_pool(wl))
    g = G.cuda_wl(factory())
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    res = G.run_stages(g, pool, lay, prm)                 # stores this step's tokens; top-k from the library
    assert res["err"] == 0
    topk = torch.as_tensor(res["topk"], device="cuda")
    out0, lse0, e0 = _attend(g, lay, prm, pool, topk)
    assert e0 == 0
    used = np.unique(g.block_table.cpu().numpy())
    used = used[used >= 0]                                # the table pads with -1
    rng = np.random.default_rng(3)
    moved = used[rng.random(used.size) < frac] if frac < 1 else used
    host, hmap = _evict(pool, lay, [int(b) for b in moved])
    out1, lse1, e1 = _attend(g, lay, prm, pool, topk, host, hmap)
    assert e1 == 0
    assert np.array_equal(out1, out0) and np.array_equal(lse1, lse0), f"{name}: host tier differs from HBM"
    out_ref = np.stack([ref[t]["out"] for t in range(g.n_tokens)])
    lse_ref = np.stack([ref[t]["lse"] for t in range(g.n_tokens)])
    G.assert_attention_close(out1, lse1, out_ref, lse_ref, name)


def test_host_map_entry_out_of_range_is_reported():
    g = G.cuda_wl(make_config(1))
    lay, prm = G.gpu_layout(g), G.gpu_params(g)
    pool = G.gpu_pool(g, lay)
    res = G.run_stages(g, pool, lay, prm)
    topk = torch.as_tensor(res["topk"], device="cuda")
    host, hmap = _evict(pool, lay, [int(g.block_table[0, 0])])
    hmap[int(g.block_table[0, 0])] = 5          # only one host block exists
    _, _, err = _attend(g, lay, prm, pool, topk, host, hmap)
    assert err == 4                              # SMLA_ERR_BAD_INDEX
