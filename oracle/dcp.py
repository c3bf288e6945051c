"""Split-context (DCP-style) sparse attention: token shards, candidate merge, LSE merge.

[AgentX "Kimi K3"]: decode context parallelism spreads one long context over
ranks; each rank attends over its part and the partial outputs are combined
with their log-sum-exp statistics.  [GLM-5.3 "What is new"] runs the same idea
(DCP8) for decode.  The pages give no formulas; what follows is the plainest
statement of that decomposition over this path's steps.

reading (token shards): with N shards, global position j of a sequence lives
in shard r = j mod N at local position i = j div N (round-robin).  A query at
global position p sees, in shard r, the local positions 0 .. (p - r) div N
(none when p < r).

reading (candidate merge): each shard scores its own positions and keeps its
local top-k; the union of those candidates, as (score, global j), is reduced to
the k highest by (score desc, j asc) -- the same rule as the unsharded top-k,
so the result equals it whenever every shard keeps k candidates (a position in
the global top-k is also in its shard's top-k).  Each shard then attends over
its selected local positions.

reading (LSE merge): partial results (out_r normalised within shard r, lse_r)
combine as  lse = ln sum_r exp(lse_r),  out = sum_r exp(lse_r - lse) out_r;
a shard with no selected position has lse_r = -inf and weight 0.
"""

import numpy as np


def shard_of(j, n_shards: int):
    """(shard, local position) of global positions ``j``."""
    j = np.asarray(j, dtype=np.int64)
    return j % n_shards, j // n_shards


def shard_visible(p: int, r: int, n_shards: int) -> int:
    """How many local positions of shard r a query at global position p sees."""
    return 0 if p < r else (p - r) // n_shards + 1


def topk_merge(shard_scores, shard_topk, n_shards: int, k: int):
    """Global top-k from the shards' local candidates, for one query token.

    shard_scores[r]: the shard's score row over its local positions.
    shard_topk[r]: the shard's local top-k (local positions, -1 padded).
    Returns (global [k] int32 ascending, -1 padded; per-shard [N, k] int32 local
    positions ascending, -1 padded).
    """
    cand_s, cand_j = [], []
    for r in range(n_shards):
        loc = np.asarray(shard_topk[r], dtype=np.int64)
        loc = loc[loc >= 0]
        cand_s.append(np.asarray(shard_scores[r], dtype=np.float32)[loc].astype(np.float64))
        cand_j.append(loc * n_shards + r)
    s = np.concatenate(cand_s) if cand_s else np.zeros(0)
    j = np.concatenate(cand_j) if cand_j else np.zeros(0, dtype=np.int64)
    order = np.lexsort((j, -s))            # score desc, then global position asc
    keep = np.sort(j[order[:min(k, j.size)]])
    glob = np.full(k, -1, dtype=np.int32)
    glob[:keep.size] = keep
    per = np.full((n_shards, k), -1, dtype=np.int32)
    r_of, i_of = shard_of(keep, n_shards)
    for r in range(n_shards):
        loc = np.sort(i_of[r_of == r])
        per[r, :loc.size] = loc
    return glob, per


def lse_merge(parts_out, parts_lse):
    """Combine partial attention results.  parts_out [N, H, D], parts_lse [N, H] -> (out [H, D], lse [H])."""
    o = np.asarray(parts_out, dtype=np.float64)
    l = np.asarray(parts_lse, dtype=np.float64)
    m = l.max(axis=0)                                        # [H]
    finite = np.isfinite(m)
    mm = np.where(finite, m, 0.0)
    wts = np.where(np.isfinite(l), np.exp(l - mm[None, :]), 0.0)   # [N, H]
    z = wts.sum(axis=0)                                      # [H]
    out = np.zeros(o.shape[1:], dtype=np.float64)
    nz = z > 0
    out[nz] = np.einsum("nh,nhd->hd", wts, o)[nz] / z[nz, None]
    lse = np.where(nz, mm + np.log(np.where(nz, z, 1.0)), -np.inf)
    return out, lse
