"""Segment-aware tile maps, plain Python (test infrastructure only).

Tile bounds follow "Packing与 FlashAttention Varlen", section 5: for segment b
of length l and q block m of BM rows, the block exists only while
m * BM < l, and its key blocks of BN columns run up to

    n_blocks = ceil(l / BN)                               (non-causal)
    n_blocks = min(ceil(l / BN), ceil((m + 1) * BM / BN)) (causal, cu_q == cu_k)

which equals ceil(min(l, (m + 1) * BM) / BN).  Blocks wholly outside a segment
or wholly above its causal diagonal are never listed.

Order (the pages do not fix one; reading taken here).  Records that read the
same K/V tiles sit together so that they run at the same time and share those
tiles through L2, and longer work goes first:

    key = (-class_b, b, h, -n_blocks, m),   class_b = floor(log2(C_b)),
    C_b = sum over the segment's q blocks of n_blocks

i.e. segments by cost class (a power-of-two bucket of their total tile count,
largest first; ties by segment index), then the segment's heads in order, then
its blocks with the most key tiles first.

The backward map lists kv blocks: for kv block n of BN rows the q blocks of BM
rows run from m_start = floor(n * BN / BM) (causal; 0 otherwise) to
ceil(l / BM) - 1; with C_b = sum over kv blocks of n_q its order is
(-class_b, b, h_kv, -n_q, n).

Token tiles (forward, causal, ``short > 0``).  A segment of l <= short tokens
would fill a q block of BM rows only l rows deep.  Maximal runs of consecutive
short segments are instead cut into row tiles of BM consecutive tokens that
may hold many segments; row i of such a tile sees the keys
[segment_start(i), i] -- the permission rule of "Pack sequences without joining
their contexts" ("Permission depends on the example": same segment and key not
later than the query) in its range form ("What the permission symbols mean").
A run [r0, r1) gives the tiles t0 = r0, r0 + BM, ... with rows = min(BM, r1 - t0)
rows; the keys a tile needs are [cu[f], t0 + rows) where f is the segment that
holds row t0.  Its record is (-1 - f, t0, h, rows), and the token records follow
every segment record, ordered by (t0, h).  Segments covered by token tiles have
no segment records.  The dK/dV map cuts the same runs into BN-row tiles of key
rows: key j of a tile is seen by the queries [j, end of its segment).

Cross-attention (``cu_k``, section 5: the causal bound is aligned bottom-right,
ceil(((m+1)*BM + lk - lq) / BN)): q block m of a segment with lq queries and lk keys has
ceil(min(lk, (m+1)*BM + lk - lq) / BN) key blocks (ceil(lk / BN) non-causal); kv block n has
its q blocks from floor(max(0, n*BN - (lk - lq)) / BM) (0 non-causal) to ceil(lq / BM) - 1.
The key-block cap lk can give the last q blocks of a causal segment equal counts, so causal
cross maps keep a segment's q blocks last-first (the same order whenever counts differ);
kv blocks and non-causal maps keep the self-attention order.  No token records.

Local window w (causal; section 5: "causal or local window further narrows
n_block_min/max"): q block m's key blocks run from n_min = floor(max(0, m*BM - w) / BN)
to its diagonal, count = n_max - n_min; kv block n's q blocks run from its diagonal
floor(n*BN / BM) to floor((n*BN + BN - 1 + w) / BM) (capped by the segment).  Window
maps have no token records and keep each segment's blocks in block order (q blocks
descending, kv blocks ascending), which is the no-window order as well.
"""
from __future__ import annotations

import numpy as np


def _ceil(a: int, b: int) -> int:
    return -(-a // b)


def _cost_class(c: int) -> int:
    return c.bit_length() - 1          # floor(log2(c)) for c >= 1


def window_key_start(m: int, BM: int, BN: int, window) -> int:
    """First key block of q block m under a local window (0 without one)."""
    return 0 if window is None else max(0, m * BM - window) // BN


def window_q_end(n: int, l: int, BM: int, BN: int, window) -> int:
    """One past the last q block that sees kv block n (the segment's last block without a window)."""
    Mq = _ceil(l, BM)
    return Mq if window is None else min(Mq, (n * BN + BN - 1 + window) // BM + 1)


def fwd_tile_map(cu_seqlens, Hq: int, BM: int, BN: int, causal: bool = True, short: int = 0, window=None,
                 cu_k=None):
    """Items as an int32 array [N, 4], in the order above: segment records
    (b, m, h, n_blocks), then (causal, short > 0) token records (-1 - f, t0, h, rows)."""
    cu = [int(x) for x in cu_seqlens]
    cuk = cu if cu_k is None else [int(x) for x in cu_k]
    B = len(cu) - 1
    tok = [causal and short > 0 and window is None and cu_k is None and cu[b + 1] - cu[b] <= short
           for b in range(B)]
    items = []
    for b in range(B):
        if tok[b]:
            continue
        l = cu[b + 1] - cu[b]
        lk = cuk[b + 1] - cuk[b]
        blocks = []
        for m in range(_ceil(l, BM)):
            nb = _ceil(min(lk, (m + 1) * BM + lk - l), BN) if causal else _ceil(lk, BN)
            blocks.append((m, nb - window_key_start(m, BM, BN, window)))
        cls = _cost_class(sum(nb for _, nb in blocks))
        for h in range(Hq):
            for m, nb in blocks:
                items.append(((-cls, b, h, -m if (window is not None or (causal and cu_k is not None)) else -nb, m),
                              (b, m, h, nb)))
    items.sort(key=lambda t: t[0])
    out = [r for _, r in items] + _token_records(cu, tok, Hq, BM)
    return np.asarray(out, dtype=np.int32).reshape(-1, 4)


def bwd_tile_map(cu_seqlens, Hkv: int, BM: int, BN: int, causal: bool = True, short: int = 0, window=None,
                 cu_k=None):
    """Items as an int32 array [N, 4], in the order above: segment records
    (b, n, h_kv, n_q), then (causal, short > 0) token records (-1 - f, t0, h_kv, rows)
    whose BN-row tiles hold the key rows [t0, t0 + rows) of a run of short segments."""
    cu = [int(x) for x in cu_seqlens]
    cuk = cu if cu_k is None else [int(x) for x in cu_k]
    B = len(cu) - 1
    tok = [causal and short > 0 and window is None and cu_k is None and cu[b + 1] - cu[b] <= short
           for b in range(B)]
    items = []
    for b in range(B):
        if tok[b]:
            continue
        l = cu[b + 1] - cu[b]
        lk = cuk[b + 1] - cuk[b]
        blocks = []
        for n in range(_ceil(lk, BN)):
            m_start = max(0, n * BN - (lk - l)) // BM if causal else 0
            blocks.append((n, window_q_end(n, l, BM, BN, window) - m_start))
        cls = _cost_class(sum(nq for _, nq in blocks))
        for h in range(Hkv):
            for n, nq in blocks:
                items.append(((-cls, b, h, n if window is not None else -nq, n), (b, n, h, nq)))
    items.sort(key=lambda t: t[0])
    return np.asarray([r for _, r in items] + _token_records(cu, tok, Hkv, BN), dtype=np.int32).reshape(-1, 4)


def _token_records(cu, tok, H, rows_per_tile):
    """Token records of every maximal run of short segments, by (t0, head)."""
    out, B, b = [], len(cu) - 1, 0
    while b < B:
        if not tok[b]:
            b += 1
            continue
        e = b
        while e < B and tok[e]:
            e += 1
        r0, r1 = cu[b], cu[e]
        for t0 in range(r0, r1, rows_per_tile):
            f = max(x for x in range(b, e) if cu[x] <= t0)
            for h in range(H):
                out.append((-1 - f, t0, h, min(rows_per_tile, r1 - t0)))
        b = e
    return out


def bwd_item_edges(cu_seqlens, item, BM: int, BN: int, window=None, cu_k=None):
    """(query, key) token pairs a backward kv item's tiles cover, in global indices (keys in
    the K/V stream's indices under cross-attention)."""
    b, n, _h, nq = (int(x) for x in item)
    cu = [int(x) for x in cu_seqlens]
    cuk = cu if cu_k is None else [int(x) for x in cu_k]
    if b < 0:                                     # token record: key rows [t0, t0 + rows)
        t0, rows = n, nq
        last = t0 + rows - 1
        end = min(cu[x + 1] for x in range(len(cu) - 1) if cu[x + 1] > last)
        return [(i, j) for j in range(t0, t0 + rows) for i in range(t0, end)]
    s, l = cu[b], cu[b + 1] - cu[b]
    sk, lk = cuk[b], cuk[b + 1] - cuk[b]
    m0 = window_q_end(n, l, BM, BN, window) - nq
    cols = range(sk + n * BN, sk + min(lk, (n + 1) * BN))
    rows = range(s + m0 * BM, s + min(l, (m0 + nq) * BM))
    return [(i, j) for i in rows for j in cols]


def fwd_item_edges(cu_seqlens, item, BM: int, BN: int, window=None, cu_k=None):
    """(query, key) token pairs a forward item's tiles cover, in global indices (keys in the
    K/V stream's indices under cross-attention)."""
    b, m, _h, nb = (int(x) for x in item)
    if b < 0:                                     # token record (-1 - f, t0, h, rows)
        t0, rows = m, nb
        kb = int(cu_seqlens[-1 - b])
        return [(i, j) for i in range(t0, t0 + rows) for j in range(kb, t0 + rows)]
    s = int(cu_seqlens[b])
    l = int(cu_seqlens[b + 1]) - s
    cuk = cu_seqlens if cu_k is None else cu_k
    sk, lk = int(cuk[b]), int(cuk[b + 1]) - int(cuk[b])
    n0 = window_key_start(m, BM, BN, window)
    rows = range(s + m * BM, s + min(l, (m + 1) * BM))
    cols = range(sk + n0 * BN, sk + min(lk, (n0 + nb) * BN))
    return [(i, j) for i in rows for j in cols]


def token_item_key_blocks(cu_seqlens, item, BN: int):
    """Key blocks of BN columns from cu[f] that a token record's rows need."""
    f, t0, _h, rows = (int(x) for x in item)
    return _ceil(t0 + rows - int(cu_seqlens[-1 - f]), BN)
