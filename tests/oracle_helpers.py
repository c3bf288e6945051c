"""Helpers shared by the oracle tests: numpy views of generated workloads."""
import numpy as np
import torch

import oracle


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def npy(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def layout_of(wl) -> "oracle.PoolLayout":
    d = wl.dims
    return oracle.PoolLayout(d.block_size, d.n_layers, d.d_latent, d.d_rope, d.quant_tile,
                             d.d_index, wl.num_blocks, d.key_format)


def oracle_pool(wl, layer: int = 0, slots=None, chunk: int = 1 << 17) -> np.ndarray:
    """Pool holding the cached context, written by the oracle's own store."""
    lay = layout_of(wl)
    pool = np.zeros(lay.pool_bytes, dtype=np.uint8)
    s = npy(wl.cached_slots) if slots is None else np.asarray(slots, dtype=np.int64)
    for c0 in range(0, s.size, chunk):
        sc = s[c0:c0 + chunk]
        st = torch.as_tensor(sc, device=wl.slot_latent.device)
        oracle.kvpack_store(lay, pool, layer, bits(wl.slot_latent[st]), bits(wl.slot_rope[st]),
                            npy(wl.slot_idx_k[st]), npy(wl.slot_idx_s[st]), sc)
    return pool


def oracle_step(wl, pool, layer: int = 0, rows=None, top_k=None):
    d = wl.dims
    return oracle.decode_step(
        layout_of(wl), pool, layer,
        latent_new=bits(wl.new_latent), rope_new=bits(wl.new_rope), idxk_new=npy(wl.new_idx_k),
        idxs_new=npy(wl.new_idx_s), slot_mapping=npy(wl.slot_mapping), q=bits(wl.q),
        q_pe=bits(wl.q_pe), q_idx=npy(wl.q_idx), w=npy(wl.w), block_table=npy(wl.block_table),
        seq_lens=npy(wl.seq_lens), query_start_loc=npy(wl.query_start_loc),
        top_k=d.top_k if top_k is None else top_k, sigma=d.softmax_scale, rows=rows)


def sequence_slots(wl, b: int) -> np.ndarray:
    """Physical slots of every cached position of sequence b (before this step's tokens)."""
    bs = wl.dims.block_size
    n_q = int(wl.query_start_loc[b + 1] - wl.query_start_loc[b])
    n = int(wl.seq_lens[b]) - n_q
    return oracle.context_slots(npy(wl.block_table[b]), n, bs)
