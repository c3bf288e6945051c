"""Indexer scores over the cached context.

[AgentX "DeepSeek V4"]: the indexer has 64 heads but yields a single global
top-k selection per token.  [GLM-5.3 "What is new"]: the indexer chooses
2,048 tokens and its cost grows quadratically with the prompt.

reading (score function): for query token t and every cached position j it
may see,
    I[t, j] = s_I[j] * sum_h  w[t, h] * ReLU( sum_d qI[t, h, d] * kI[j, d] )
with qI decoded E4M3 values, kI decoded E4M3 values (or FP4 E2M1 values for a
layout with FP4 keys, [AgentX "Hybrid KV cache management"]), one indexer key
per cached token shared by all indexer heads, w the per-(token, head) weight
and s_I[j] the key's fp32 scale.  Accumulated in float64 and rounded once to
float32.

reading (query positions): ``seq_lens[b]`` counts this step's tokens, which
are stored before the scores are taken; query i of the n_q tokens of sequence b
sits at position p = seq_lens[b] - n_q + i and sees positions 0..p (itself
included).
"""

import numpy as np

from .fp8 import e4m3_decode
from .store import read_index_key


def query_positions(seq_lens, query_start_loc):
    """Per query token: (sequence index b, position p)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    seqs, pos = [], []
    for b in range(seq_lens.size):
        n_q = qsl[b + 1] - qsl[b]
        for i in range(n_q):
            seqs.append(b)
            pos.append(seq_lens[b] - n_q + i)
    return np.array(seqs, dtype=np.int64), np.array(pos, dtype=np.int64)


def context_slots(block_table_row, n: int, block_size: int) -> np.ndarray:
    """Physical slots of logical positions 0..n-1 through one block-table row."""
    j = np.arange(n, dtype=np.int64)
    blocks = np.asarray(block_table_row, dtype=np.int64)[j // block_size]
    return blocks * block_size + j % block_size


def index_scores_row(layout, pool, layer, q_codes, w, block_table_row, p: int,
                     chunk: int = 1 << 17) -> np.ndarray:
    """Scores I[t, 0..p] (float32) of one query token.

    q_codes: [H_I, D_I] uint8 E4M3; w: [H_I] fp32.
    """
    n = int(p) + 1
    if n <= 0:
        return np.zeros(0, dtype=np.float32)
    q = e4m3_decode(q_codes)                                   # [H_I, D_I]
    wt = np.asarray(w, dtype=np.float32).astype(np.float64)    # [H_I]
    slots = context_slots(block_table_row, n, layout.block_size)
    out = np.empty(n, dtype=np.float32)
    for c0 in range(0, n, chunk):
        keys, s = read_index_key(layout, pool, layer, slots[c0:c0 + chunk])
        dots = q @ keys.T                                      # [H_I, n_c], exact in float64
        head_sum = (wt[:, None] * np.maximum(dots, 0.0)).sum(axis=0)
        out[c0:c0 + chunk] = (head_sum * s).astype(np.float32)
    return out


def index_scores(layout, pool, layer, q_codes, w, block_table, seq_lens, query_start_loc,
                 max_ctx: int, rows=None) -> np.ndarray:
    """Scores [T, max_ctx] float32; -inf beyond each token's position p.

    ``rows`` restricts the computation to those query tokens (others stay -inf).
    """
    seqs, pos = query_positions(seq_lens, query_start_loc)
    t_all = seqs.size
    out = np.full((t_all, max_ctx), -np.inf, dtype=np.float32)
    for t in (range(t_all) if rows is None else rows):
        row = index_scores_row(layout, pool, layer, q_codes[t], w[t], block_table[seqs[t]], pos[t])
        out[t, :row.size] = row
    return out
