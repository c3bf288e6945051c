"""Latent MQA attention over a set of cached positions.

[AgentX "Kimi K3"], [GLM-5.3 "What is new"]: MLA compresses KV into one latent
shared by all 64 query heads, so attention is MQA over the latent.
[AgentX "DeepSeek V4"]: sparse MLA attends only over the top-k entries.
[AgentX "Kimi K3"] (DCP): partial outputs carry log-sum-exp statistics.
[GLM-5.3 "How to try"] (sparse_mla_force_mqa): a prompt that fits inside the
top-k still takes the sparse kernel, so sparse must equal dense attention when
every position is selected.

reading: with K[j] = dequantised latent (D_L) and kpe[j] = rope part (D_R),
    s[h, j]  = sigma * (q[h] . K[j] + q_pe[h] . kpe[j])
    P[h, :]  = softmax_j s[h, :]
    out[h]   = sum_j P[h, j] * K[j]          (V is the latent itself)
    lse[h]   = ln sum_j exp(s[h, j])
in float64.  An empty set gives out = 0 and lse = -inf.
"""

import numpy as np

from .indexer import context_slots
from .store import read_record


def attend(q, q_pe, lat, rope, sigma: float):
    """Textbook softmax attention.  q [H, D_L], q_pe [H, D_R], lat [n, D_L], rope [n, D_R]."""
    h = q.shape[0]
    if lat.shape[0] == 0:
        return np.zeros((h, lat.shape[1]), dtype=np.float64), np.full(h, -np.inf)
    s = float(sigma) * (q @ lat.T + q_pe @ rope.T)           # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=1, keepdims=True)
    out = (e / z) @ lat
    lse = (m + np.log(z))[:, 0]
    return out, lse


def sparse_attend(layout, pool, layer, q, q_pe, topk_row, block_table_row, sigma: float):
    """Attention over the positions listed in ``topk_row`` (-1 entries ignored)."""
    sel = np.asarray(topk_row, dtype=np.int64)
    sel = sel[sel >= 0]
    bt = np.asarray(block_table_row, dtype=np.int64)
    slots = bt[sel // layout.block_size] * layout.block_size + sel % layout.block_size
    lat, rope = read_record(layout, pool, layer, slots)
    return attend(q, q_pe, lat, rope, sigma)


def dense_attend(layout, pool, layer, q, q_pe, block_table_row, p: int, sigma: float):
    """Attention over every position 0..p."""
    slots = context_slots(block_table_row, int(p) + 1, layout.block_size)
    lat, rope = read_record(layout, pool, layer, slots)
    return attend(q, q_pe, lat, rope, sigma)
