"""Top-k selection of cached positions.

[GLM-5.3 "What is new"]: the indexer selects 2,048 tokens.  [AgentX
"DeepSeek V4"]: one global top-k per token; scanning and gathering the top-k
entries dominates sparse MLA.

reading (ties and output form): the k highest scores among positions
0..p are kept, equal scores going to the lower position; if p+1 <= k every
position is kept.  The kept positions are returned in ascending order, padded
with -1 to length k.  Scores compare as float32 values (so -0.0 == +0.0).
"""

import numpy as np


def topk_select(scores_row, k: int) -> np.ndarray:
    """Indices [k] int32 for one query token; ``scores_row`` holds positions 0..p."""
    s = np.asarray(scores_row, dtype=np.float32)
    n = s.size
    j = np.arange(n, dtype=np.int64)
    order = np.lexsort((j, -s.astype(np.float64)))   # primary: score desc, secondary: j asc
    keep = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[:keep.size] = keep
    return out
