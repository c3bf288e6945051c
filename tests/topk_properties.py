"""Property check of a top-k selection against the score rows it was taken from.

A selection of row t (visible positions 0..n_t-1, k slots) is THE top-k of the
row under the rule "k highest scores, equal scores to the lower position,
ascending, -1 padded" exactly when:

  count       it keeps min(k, n_t) positions;
  prefix      the kept positions fill the first slots, -1 after them;
  ascending   the kept positions increase strictly;
  in_range    every kept position is < n_t;
  threshold   no position left out scores above the lowest kept score T;
  ties        every kept position scoring T lies below every left-out
              position scoring T.

Scores compare as float32 values (-0 == +0).  This holds at any size, so the
full-size tests check every row with it, while the oracle recomputes sampled
rows one by one.  Works on CPU and CUDA tensors alike.
"""
import torch

CHECKS = ("count", "prefix", "ascending", "in_range", "threshold", "ties")


def topk_violations(scores: torch.Tensor, topk: torch.Tensor, n_visible: torch.Tensor, k: int,
                    rows_per_chunk: int = 256) -> dict:
    """Rows failing each check, as {check: [row, ...]}; every list empty means the selection is exact."""
    bad = {c: [] for c in CHECKS}
    T, S = scores.shape
    dev = scores.device
    for r0 in range(0, T, rows_per_chunk):
        r1 = min(T, r0 + rows_per_chunk)
        s = scores[r0:r1].float() + 0.0                      # folds -0 onto +0
        tk = topk[r0:r1].long()
        n = n_visible[r0:r1].long().to(dev)
        R = r1 - r0
        valid = tk >= 0
        cnt = valid.sum(1)
        want = torch.clamp(n, max=k)
        ok = {}
        ok["count"] = cnt == want
        ok["prefix"] = ~(valid[:, 1:] & ~valid[:, :-1]).any(1)
        ok["ascending"] = ((tk[:, 1:] > tk[:, :-1]) | ~valid[:, 1:]).all(1)
        ok["in_range"] = (~valid | (tk < n[:, None])).all(1)
        # membership of each visible position (invalid slots land in a spare column)
        member = torch.zeros((R, S + 1), dtype=torch.bool, device=dev)
        member.scatter_(1, torch.where(valid & (tk < S), tk, torch.full_like(tk, S)), True)
        member = member[:, :S]
        cols = torch.arange(S, device=dev)
        visible = cols[None, :] < n[:, None]
        kept = member & visible
        left = visible & ~member
        inf = torch.tensor(float("inf"), device=dev)
        thr = torch.where(kept, s, inf).amin(1)               # lowest kept score
        top_left = torch.where(left, s, -inf).amax(1)         # highest score left out
        ok["threshold"] = (top_left <= thr) | ~left.any(1)
        at_thr = s == thr[:, None]
        last_kept_at = torch.where(kept & at_thr, cols[None, :], torch.full_like(cols, -1)[None, :]).amax(1)
        first_left_at = torch.where(left & at_thr, cols[None, :], torch.full_like(cols, S)[None, :]).amin(1)
        ok["ties"] = last_kept_at < first_left_at
        for c in CHECKS:
            rows = (~ok[c]).nonzero().flatten()
            bad[c].extend(int(x) + r0 for x in rows.cpu())
    return bad


def assert_topk_exact(scores, topk, n_visible, k, what=""):
    bad = topk_violations(scores, topk, n_visible, k)
    failed = {c: v[:5] for c, v in bad.items() if v}
    assert not failed, f"{what}: top-k violates {failed} (first rows shown)"
