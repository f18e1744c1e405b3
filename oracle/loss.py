"""Packed next-token targets, token-weighted objective and constructed-logit probe
(test infrastructure only).

"Pack sequences without joining their contexts", "Keep the same nine-target
objective": the packed loss is the raw sum of the negative log likelihoods of
all eligible targets divided once by their count N (token weighting).  The
probe gives every non-gold logit 0 and the gold logit z_y = ln((V-1) q / (1-q)),
so softmax assigns probability q to the gold class; the mean-loss logit
gradient is (p_ic - [c == y_i]) / N, and cells that are not eligible are
skipped before any arithmetic.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


def stream_targets(token_ids, cu_seqlens, ignore_index: int = IGNORE_INDEX):
    """Next-token targets of a packed stream of whole documents, pairs formed inside each
    document ("Form pairs inside each source range"): position t of segment [s, e) predicts
    token t + 1 when t + 1 < e; the last position of every segment has no target
    (``ignore_index``), so no pair crosses a boundary ("A's final input still predicts its
    own EOS; it does not predict B's BOS")."""
    ids = np.asarray(token_ids, dtype=np.int64).reshape(-1)
    cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
    out = np.full(ids.size, ignore_index, dtype=np.int64)
    for b in range(cu.size - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        for t in range(s, e - 1):
            out[t] = ids[t + 1]
    return out


def constructed_logits(targets, eligible, q_of_cell, vocab: int):
    """Logits [cells, V] of the probe; non-eligible rows stay all zero (skipped later)."""
    targets = np.asarray(targets).reshape(-1)
    eligible = np.asarray(eligible, dtype=bool).reshape(-1)
    q = np.asarray(q_of_cell, dtype=np.float64).reshape(-1)
    z = np.zeros((targets.size, vocab))
    for c in range(targets.size):
        if eligible[c]:
            z[c, targets[c]] = np.log((vocab - 1) * q[c] / (1.0 - q[c]))
    return z


def token_weighted_loss(logits, targets, eligible):
    """(loss_sum, mean, grad) of the token-weighted mean cross entropy.

    Only eligible cells are touched; ``grad`` is d(mean)/d(logits), zero on
    excluded cells.  Zero eligible targets is an error (no denominator).
    """
    logits = np.asarray(logits, dtype=np.float64)
    targets = np.asarray(targets).reshape(-1)
    eligible = np.asarray(eligible, dtype=bool).reshape(-1)
    idx = np.nonzero(eligible)[0]
    N = idx.size
    if N == 0:
        raise ValueError("no eligible targets: the mean has no denominator")
    z = logits[idx]
    mx = z.max(axis=1, keepdims=True)
    logz = mx[:, 0] + np.log(np.exp(z - mx).sum(axis=1))
    nll = logz - z[np.arange(N), targets[idx]]
    loss_sum = float(nll.sum())
    p = np.exp(z - logz[:, None])
    onehot = np.zeros_like(p)
    onehot[np.arange(N), targets[idx]] = 1.0
    grad = np.zeros_like(logits)
    grad[idx] = (p - onehot) / N
    return loss_sum, loss_sum / N, grad
