"""Segment-aware tile maps, plain Python (test infrastructure only).

Tile bounds follow "Packing与 FlashAttention Varlen", section 5: for segment b
of length l and q block m of BM rows, the block exists only while
m * BM < l, and its key blocks of BN columns run up to

    n_blocks = ceil(l / BN)                               (non-causal)
    n_blocks = min(ceil(l / BN), ceil((m + 1) * BM / BN)) (causal, cu_q == cu_k)

which equals ceil(min(l, (m + 1) * BM) / BN).  Blocks wholly outside a segment
or wholly above its causal diagonal are never listed.

Order (the pages do not fix one; reading taken here): longest first, ties by
segment, then block, then head -- key (-n_blocks, b, m, h).  Heads are last so
that q heads of one GQA group sit next to each other.

The backward map lists kv blocks: for kv block n of BN rows the q blocks of BM
rows run from m_start = floor(n * BN / BM) (causal; 0 otherwise) to
ceil(l / BM) - 1, ordered by (-n_q, b, n, h_kv).
"""
from __future__ import annotations

import numpy as np


def _ceil(a: int, b: int) -> int:
    return -(-a // b)


def fwd_tile_map(cu_seqlens, Hq: int, BM: int, BN: int, causal: bool = True):
    """Items (b, m, h, n_blocks) as an int32 array [N, 4], sorted longest first."""
    cu = [int(x) for x in cu_seqlens]
    items = []
    for b in range(len(cu) - 1):
        l = cu[b + 1] - cu[b]
        for m in range(_ceil(l, BM)):
            nb = _ceil(min(l, (m + 1) * BM), BN) if causal else _ceil(l, BN)
            for h in range(Hq):
                items.append((b, m, h, nb))
    items.sort(key=lambda t: (-t[3], t[0], t[1], t[2]))
    return np.asarray(items, dtype=np.int32).reshape(-1, 4)


def bwd_tile_map(cu_seqlens, Hkv: int, BM: int, BN: int, causal: bool = True):
    """Items (b, n, h_kv, n_q) as an int32 array [N, 4], sorted longest first."""
    cu = [int(x) for x in cu_seqlens]
    items = []
    for b in range(len(cu) - 1):
        l = cu[b + 1] - cu[b]
        Mq = _ceil(l, BM)
        for n in range(_ceil(l, BN)):
            m_start = (n * BN) // BM if causal else 0
            for h in range(Hkv):
                items.append((b, n, h, Mq - m_start))
    items.sort(key=lambda t: (-t[3], t[0], t[1], t[2]))
    return np.asarray(items, dtype=np.int32).reshape(-1, 4)


def fwd_item_edges(cu_seqlens, item, BM: int, BN: int):
    """(query, key) token pairs a forward item's tiles cover, in global indices."""
    b, m, _h, nb = (int(x) for x in item)
    s = int(cu_seqlens[b])
    l = int(cu_seqlens[b + 1]) - s
    rows = range(s + m * BM, s + min(l, (m + 1) * BM))
    cols = range(s, s + min(l, nb * BN))
    return [(i, j) for i in rows for j in cols]
