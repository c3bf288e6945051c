"""GPU parity of kvpack_store's two access paths against the CPU oracle, through the C ABI.

The store reads a token's latent as 16-byte vectors and its rope and indexer key as 32-bit words,
and writes each lane's 16 E4M3 codes as one 16-byte store, when every base and stride allows it
(the launcher checks the pool, latent, rope and key pointers and the layout's strides); otherwise
it uses 2- and 1-byte accesses.  Tensors that torch allocates are aligned, so the full-size tests
take the vector path; here each input in turn, and the pool, sits a few bytes past an aligned
address, which sends the launch down the other path.  Either way the pool bytes must equal the
oracle's store of the same tokens, for E4M3 and for packed E2M1 indexer keys.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import paged_sparse_mla_gb300 as smla
from paged_sparse_mla_gb300.workloads import FULL, build_workload
from tests.oracle_helpers import bits, layout_of, npy
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    G.ensure_built()


def _shifted(t, elems):
    """The values of t, contiguous, `elems` elements past the start of an allocation."""
    flat = t.reshape(-1)
    buf = torch.zeros(flat.numel() + elems, dtype=t.dtype, device="cuda")
    view = buf[elems:]
    view.copy_(flat)
    return view.view(t.shape)


@pytest.mark.parametrize("key_format", ["e4m3", "e2m1"])
@pytest.mark.parametrize("moved", ["none", "latent", "rope", "idx_k", "pool"])
def test_store_paths_match_the_oracle(moved, key_format):
    dims = replace(FULL, key_format=key_format)
    # three sequences, 7 new tokens; ragged contexts so that the new slots fall in several blocks
    wl = G.cuda_wl(build_workload("store-paths", dims, [640, 130, 70], [4, 1, 2], seed=11))
    lay = G.gpu_layout(wl)
    lat, rope, key = wl.new_latent, wl.new_rope, wl.new_idx_k
    if moved == "latent":
        lat = _shifted(lat, 1)   # 2 bytes past a 16-byte boundary
    elif moved == "rope":
        rope = _shifted(rope, 1)  # 2 bytes past a 4-byte boundary
    elif moved == "idx_k":
        key = _shifted(key, 1)   # 1 byte past a 4-byte boundary
    pool_buf = torch.zeros(lay.pool_bytes + 16, dtype=torch.uint8, device="cuda")
    off = 8 if moved == "pool" else 0
    pool = pool_buf[off:off + lay.pool_bytes]
    smla.kvpack_store(lay, pool, 0, lat, rope, key, wl.new_idx_s, wl.slot_mapping)
    torch.cuda.synchronize()
    assert smla.smla_get_last_error() == 0
    lo = layout_of(wl)
    ref = np.zeros(lo.pool_bytes, np.uint8)
    oracle.kvpack_store(lo, ref, 0, bits(wl.new_latent), bits(wl.new_rope), npy(wl.new_idx_k), npy(wl.new_idx_s),
                        npy(wl.slot_mapping))
    got = pool.cpu().numpy()
    assert np.array_equal(got, ref), f"{moved}: {int((got != ref).sum())} pool bytes differ"
    assert int(pool_buf[:off].sum()) == 0 and int(pool_buf[off + lay.pool_bytes:].sum()) == 0, "wrote outside the pool"
