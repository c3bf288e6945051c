"""The whole step: store -> indexer scores -> top-k -> sparse attention.

[GLM-5.3 "What is new", "Config and numbers"]: decode steps carry MTP draft
tokens (MTP3: one token plus three drafts) and prefill runs on a long cached
prefix; [AgentX "Head-of-line blocking"] chunked prefill appends new tokens to
a cached prefix.  Both are the same computation per query token; only the
number of query tokens per sequence differs.

reading: the step's new tokens are written to the pool first (through
``slot_mapping``), then every query token is scored against positions
0..p, its top-k is taken and attention runs over the selected positions.
"""

import numpy as np

from .indexer import index_scores_row, query_positions
from .store import kvpack_store, bf16_bits_to_f64
from .topk import topk_select
from .attention import sparse_attend


def decode_step(layout, pool, layer, *, latent_new, rope_new, idxk_new, idxs_new, slot_mapping,
                q, q_pe, q_idx, w, block_table, seq_lens, query_start_loc, top_k: int,
                sigma: float, rows=None, store: bool = True):
    """Run the step for query tokens ``rows`` (all if None).

    ``pool`` is modified in place by the store when ``store`` is true.  bf16
    inputs (latent_new, rope_new, q, q_pe) are uint16 bit patterns.
    Returns {t: dict(scores=fp32[p+1], topk=int32[k], out=f64[H, D_L], lse=f64[H])}.
    """
    if store:
        kvpack_store(layout, pool, layer, latent_new, rope_new, idxk_new, idxs_new, slot_mapping)
    seqs, pos = query_positions(seq_lens, query_start_loc)
    result = {}
    for t in (range(seqs.size) if rows is None else rows):
        b, p = int(seqs[t]), int(pos[t])
        scores = index_scores_row(layout, pool, layer, q_idx[t], w[t], block_table[b], p)
        sel = topk_select(scores, top_k)
        out, lse = sparse_attend(layout, pool, layer, bf16_bits_to_f64(q[t]), bf16_bits_to_f64(q_pe[t]),
                                 sel, block_table[b], sigma)
        result[t] = dict(scores=scores, topk=sel, out=out, lse=lse, seq=b, pos=p)
    return result
