"""Exact per-segment causal attention in float64 (test infrastructure only).

Definition followed ("Packing与 FlashAttention Varlen", section 1: a packed
stream with boundaries [0, 5, 8, 12] is three independent attentions, i.e.
block-diagonal causal attention; section 5: each logical sequence b is the
slice [cu[b], cu[b+1]) of the flat Q/K/V axis and its output is written back at
the same offsets).  The permission rule is the one of "Pack sequences without
joining their contexts", "Permission depends on the example": query i may use
key j iff both are real tokens of the same segment and pos(j) <= pos(i).

For one segment of length l, a q head h and its kv head hk = h // (Hq / Hkv):

    s_ij  = scale * q_i . k_j                      (visible j only)
    LSE_i = ln sum_j exp(s_ij)                     (natural log)
    P_ij  = exp(s_ij - LSE_i),  O_i = sum_j P_ij v_j

Backward, given dO (analytic gradient of the definition above):

    D_i   = dO_i . O_i
    dV_j  = sum_i P_ij dO_i          dP_ij = dO_i . v_j
    dS_ij = P_ij (dP_ij - D_i)
    dQ_i  = scale sum_j dS_ij k_j    dK_j  = scale sum_i dS_ij q_i

and dK, dV sum over the q heads that share a kv head.

Local window ("Packing与 FlashAttention Varlen", section 5: a local window further
narrows the key blocks a query block may see): with ``window = w`` (causal only),
query i sees the keys i - w <= j <= i of its segment, i.e. itself and the w keys
before it (FlashAttention's left window size; its right size is 0 under causality).

Cross-attention (``cu_k`` given, blog section 3: cu_q and cu_k cut Q and K/V separately,
the b-th Q slice and K/V slice belong to the same sample; section 5: the causal bound is
aligned bottom-right, (m+1)*BM + seqlen_k - seqlen_q): query i of a segment sees the keys
j <= i + (lk - lq) of the same segment.  Reading taken here: causal cross-attention needs
lq <= lk in every segment (every query then sees at least one key); other lengths are
rejected rather than given empty softmax rows.

The GQA head mapping h -> h // (Hq/Hkv) is not on the pages; it is the plainest
reading (consecutive q heads share a kv head).  Rows of long segments are
processed in blocks only to bound memory; each block computes full rows.
"""
from __future__ import annotations

import numpy as np

_BLOCK_BYTES = 256 * 1024 * 1024


def _row_block(l: int, heads: int) -> int:
    return max(1, min(l, _BLOCK_BYTES // max(1, 8 * heads * l)))


def check_cu_seqlens(cu, T: int) -> np.ndarray:
    """The boundary contract of blog section 3: int, first 0, last T, strictly increasing."""
    cu = np.asarray(cu, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 2:
        raise ValueError("cu_seqlens needs at least two entries")
    if cu[0] != 0 or cu[-1] != T:
        raise ValueError("cu_seqlens must start at 0 and end at T")
    if np.any(np.diff(cu) <= 0):
        raise ValueError("cu_seqlens must be strictly increasing")
    return cu


def _expand(x: np.ndarray, g: int) -> np.ndarray:
    # [l, Hkv, d] -> [Hq, l, d]; q head h reads kv head h // g
    return np.repeat(x, g, axis=1).transpose(1, 0, 2)


def _visible(i, j, causal: bool, window, off: int = 0):
    """Permission of query rows i (column vector) on key columns j (row vector); off is the
    bottom-right causal offset lk - lq (0 for self-attention)."""
    if not causal:
        return np.ones(np.broadcast(i, j).shape, dtype=bool)
    vis = j <= i + off
    if window is not None:
        vis = vis & (j >= i - window)
    return vis


def _check_window(causal: bool, window):
    if window is not None and (not causal or window < 0):
        raise ValueError("a local window needs causal attention and window >= 0")


def segment_forward(q, k, v, scale: float, causal: bool = True, window=None):
    """One segment, all heads.  q [lq,Hq,d], k/v [lk,Hkv,d] (float64); lq == lk unless
    cross-attention (bottom-right causal alignment, lq <= lk when causal).

    Returns (o [lq,Hq,d], lse [Hq,lq]).
    """
    _check_window(causal, window)
    l, Hq, d = q.shape
    lk = k.shape[0]
    off = lk - l
    if causal and off < 0:
        raise ValueError("causal cross-attention needs lq <= lk")
    if window is not None and off != 0:
        raise ValueError("a local window is for self-attention")
    g = Hq // k.shape[1]
    Q = q.transpose(1, 0, 2)
    K = _expand(k, g)
    V = _expand(v, g)
    o = np.empty((Hq, l, v.shape[2]))
    lse = np.empty((Hq, l))
    rb = _row_block(l, Hq)
    for r0 in range(0, l, rb):
        r1 = min(l, r0 + rb)
        kend = r1 + off if causal else lk
        s = scale * (Q[:, r0:r1] @ K[:, :kend].transpose(0, 2, 1))
        if causal:
            i = np.arange(r0, r1)[:, None]
            j = np.arange(kend)[None, :]
            s = np.where(_visible(i, j, causal, window, off), s, -np.inf)
        mx = s.max(axis=2, keepdims=True)
        e = np.exp(s - mx)
        z = e.sum(axis=2, keepdims=True)
        o[:, r0:r1] = (e / z) @ V[:, :kend]
        lse[:, r0:r1] = (mx + np.log(z))[..., 0]
    return o.transpose(1, 0, 2), lse


def segment_backward(q, k, v, o, lse, do, scale: float, causal: bool = True, window=None):
    """Analytic backward of ``segment_forward`` for one segment.

    ``o``/``lse`` are this oracle's own forward results.  Returns (dq, dk, dv)
    with the shapes of q, k, v.
    """
    _check_window(causal, window)
    l, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    lk = k.shape[0]
    off = lk - l
    if causal and off < 0:
        raise ValueError("causal cross-attention needs lq <= lk")
    Q = q.transpose(1, 0, 2)
    K = _expand(k, g)
    V = _expand(v, g)
    dO = do.transpose(1, 0, 2)
    D = (do * o).sum(axis=2).T                    # [Hq, l]
    dQ = np.zeros((Hq, l, d))
    dKx = np.zeros((Hq, lk, d))
    dVx = np.zeros((Hq, lk, v.shape[2]))
    rb = _row_block(l, Hq)
    for r0 in range(0, l, rb):
        r1 = min(l, r0 + rb)
        kend = r1 + off if causal else lk
        s = scale * (Q[:, r0:r1] @ K[:, :kend].transpose(0, 2, 1))
        p = np.exp(s - lse[:, r0:r1, None])
        if causal:
            i = np.arange(r0, r1)[:, None]
            j = np.arange(kend)[None, :]
            p = np.where(_visible(i, j, causal, window, off), p, 0.0)
        dVx[:, :kend] += p.transpose(0, 2, 1) @ dO[:, r0:r1]
        dp = dO[:, r0:r1] @ V[:, :kend].transpose(0, 2, 1)
        ds = p * (dp - D[:, r0:r1, None])
        dQ[:, r0:r1] = scale * (ds @ K[:, :kend])
        dKx[:, :kend] += scale * (ds.transpose(0, 2, 1) @ Q[:, r0:r1])
    dK = dKx.reshape(Hkv, g, lk, d).sum(axis=1)
    dV = dVx.reshape(Hkv, g, lk, v.shape[2]).sum(axis=1)
    return dQ.transpose(1, 0, 2), dK.transpose(1, 0, 2), dV.transpose(1, 0, 2)


def _head_slices(Hq: int, Hkv: int, kv_heads):
    g = Hq // Hkv
    if kv_heads is None:
        kv_heads = range(Hkv)
    kv_heads = list(kv_heads)
    return kv_heads, g


def varlen_forward(q, k, v, cu_seqlens, scale=None, causal=True, kv_heads=None, window=None,
                   cu_seqlens_k=None):
    """Packed forward: every segment of ``cu_seqlens`` is its own attention.

    q [T,Hq,d], k/v [T,Hkv,d] float64.  Returns (o [T,Hq,d], lse [Hq,T]).
    With ``kv_heads`` set, only those kv heads and their q-head groups are
    computed; every other entry is NaN.  With ``cu_seqlens_k`` (cross-attention) k/v are
    [Tk,Hkv,d] cut by their own boundaries.
    """
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    cu = check_cu_seqlens(cu_seqlens, T)
    cuk = cu if cu_seqlens_k is None else check_cu_seqlens(cu_seqlens_k, k.shape[0])
    if cuk.size != cu.size:
        raise ValueError("cu_seqlens and cu_seqlens_k need the same number of segments")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    kvh, g = _head_slices(Hq, Hkv, kv_heads)
    o = np.full((T, Hq, v.shape[2]), np.nan)
    lse = np.full((Hq, T), np.nan)
    for b in range(cu.size - 1):
        s, e = cu[b], cu[b + 1]
        sk, ek = cuk[b], cuk[b + 1]
        for hk in kvh:
            hq = slice(hk * g, (hk + 1) * g)
            ob, lb = segment_forward(q[s:e, hq], k[sk:ek, hk:hk + 1], v[sk:ek, hk:hk + 1],
                                     scale, causal, window)
            o[s:e, hq] = ob
            lse[hq, s:e] = lb
    return o, lse


def varlen_backward(q, k, v, o, lse, do, cu_seqlens, scale=None, causal=True,
                    kv_heads=None, window=None, cu_seqlens_k=None):
    """Packed backward (dq, dk, dv); entries of heads outside ``kv_heads`` are NaN."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu = check_cu_seqlens(cu_seqlens, T)
    cuk = cu if cu_seqlens_k is None else check_cu_seqlens(cu_seqlens_k, k.shape[0])
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    kvh, g = _head_slices(Hq, Hkv, kv_heads)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    for b in range(cu.size - 1):
        s, e = cu[b], cu[b + 1]
        sk, ek = cuk[b], cuk[b + 1]
        for hk in kvh:
            hq = slice(hk * g, (hk + 1) * g)
            a, bk, c = segment_backward(q[s:e, hq], k[sk:ek, hk:hk + 1], v[sk:ek, hk:hk + 1],
                                        o[s:e, hq], lse[hq, s:e], do[s:e, hq],
                                        scale, causal, window)
            dq[s:e, hq] = a
            dk[sk:ek, hk:hk + 1] = bk
            dv[sk:ek, hk:hk + 1] = c
    return dq, dk, dv


def rows_forward_backward(q, k, v, do, cu_seqlens, tokens, heads, scale=None,
                          causal=True):
    """O, LSE and dQ for single (token, q head) pairs, each computed from its own row.

    dQ_i needs only row i: P_i from LSE_i, dP_i = dO_i V^T, D_i = dO_i . O_i.
    Used to check outputs of large packs one row at a time.
    Returns (o [n,d], lse [n], dq [n,d]).
    """
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    cu = check_cu_seqlens(cu_seqlens, T)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    seg = np.searchsorted(cu, np.asarray(tokens), side="right") - 1
    n = len(tokens)
    o = np.empty((n, v.shape[2]))
    lse = np.empty(n)
    dq = np.empty((n, d))
    for r, (t, h, b) in enumerate(zip(tokens, heads, seg)):
        s0 = cu[b]
        kend = t + 1 if causal else cu[b + 1]
        hk = h // g
        K = k[s0:kend, hk]
        V = v[s0:kend, hk]
        sc = scale * (K @ q[t, h])
        mx = sc.max()
        e = np.exp(sc - mx)
        z = e.sum()
        p = e / z
        o[r] = p @ V
        lse[r] = mx + np.log(z)
        dp = V @ do[t, h]
        D = do[t, h] @ o[r]
        dq[r] = scale * ((p * (dp - D)) @ K)
    return o, lse, dq


def dense_permission_attention(q, k, v, segments, positions, valid, scale):
    """Brute force: materialise the [T, T] permission matrix and run masked softmax.

    allowed(i, j) = valid[i] and valid[j] and seg[i] == seg[j] and pos[j] <= pos[i]
    ("Pack sequences without joining their contexts", "Permission depends on
    the example").  A query with no allowed key (an inactive pad query) gets a
    zero mixture and LSE = -inf.  Works on torch float64 tensors so autograd
    can differentiate it.  Returns (o [T,Hq,d], lse [Hq,T], allowed [T,T]).
    """
    import torch

    segments = torch.as_tensor(segments)
    positions = torch.as_tensor(positions)
    valid = torch.as_tensor(valid, dtype=torch.bool)
    allowed = (valid[:, None] & valid[None, :]
               & (segments[:, None] == segments[None, :])
               & (positions[None, :] <= positions[:, None]))
    T, Hq, d = q.shape
    g = Hq // k.shape[1]
    K = k.repeat_interleave(g, dim=1)
    V = v.repeat_interleave(g, dim=1)
    s = scale * torch.einsum("ihc,jhc->hij", q, K)
    s = s.masked_fill(~allowed[None], float("-inf"))
    lse = torch.logsumexp(s, dim=2)
    safe = torch.where(torch.isfinite(lse), lse, torch.zeros_like(lse))
    p = torch.exp(s - safe[..., None]).masked_fill(~allowed[None], 0.0)
    o = torch.einsum("hij,jhc->ihc", p, V)
    return o, lse, allowed


def key_rows_backward(q, k, v, do, cu_seqlens, tokens, kv_head, scale=None, causal=True):
    """dK, dV for single (key token, kv head) pairs, from the queries that read them.

    dK_j and dV_j need P_ij for every query i that sees key j (i >= j in the
    segment when causal), and P_ij needs that query's full-row LSE_i and D_i.
    Cost is (queries after j) x (segment length) per key, so this is meant for
    keys near the end of long segments.  Returns (dk [n,d], dv [n,d]).
    """
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    cu = check_cu_seqlens(cu_seqlens, T)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    seg = np.searchsorted(cu, np.asarray(tokens), side="right") - 1
    dk = np.zeros((len(tokens), d))
    dv = np.zeros((len(tokens), v.shape[2]))
    cache = {}
    for r, (j, b) in enumerate(zip(tokens, seg)):
        s0, e0 = cu[b], cu[b + 1]
        first_q = j if causal else s0
        for h in range(kv_head * g, (kv_head + 1) * g):
            for i in range(first_q, e0):
                key = (i, h)
                if key not in cache:
                    kend = i + 1 if causal else e0
                    K = k[s0:kend, kv_head]
                    V = v[s0:kend, kv_head]
                    sc = scale * (K @ q[i, h])
                    mx = sc.max()
                    e = np.exp(sc - mx)
                    z = e.sum()
                    o_i = (e / z) @ V
                    cache[key] = (mx + np.log(z), do[i, h] @ o_i)
                lse_i, D_i = cache[key]
                p = np.exp(scale * (q[i, h] @ k[j, kv_head]) - lse_i)
                dp = do[i, h] @ v[j, kv_head]
                dv[r] += p * do[i, h]
                dk[r] += scale * p * (dp - D_i) * q[i, h]
    return dk, dv
