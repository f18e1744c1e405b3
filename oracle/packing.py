"""Packing planners and boundary metadata, plain Python (test infrastructure only).

* ``next_fit``  -- order-preserving next-fit ("Packing与 FlashAttention Varlen",
  section 2, the ``sequential`` strategy; "Pack sequences without joining their
  contexts", "Fill only the current row" and "Extend the existing storage and
  decoder"): documents are read in order, a new pack starts when the document
  does not fit the space left in the current one, a document longer than the
  capacity is an error (never split), an exact fill opens no extra pack.
* ``best_fit_decreasing`` -- the default ``binpack`` strategy of blog section 2
  (maximise fill, may reorder).  The pages do not fix tie-breaking; the reading
  taken here: sort by length descending, ties by input index; put each document
  in the open pack with the least remaining space that still fits it, ties to
  the earliest-opened pack; otherwise open a new pack.  Packs keep their
  opening order and documents their insertion order.
* ``build_metadata`` -- blog section 3: cumulative boundaries ``cu_seqlens``
  (first 0, last T, strictly increasing), per-sample positions restarting at 0
  (blog section 2, ``packing_row`` when positions are absent), segment ids,
  ``max_seqlen = max diff(cu_seqlens)``.  A tail pad up to ``pad_to`` tokens is
  one extra segment with its own positions 0..p-1.
* ``cu_seqlens_from_position_ids`` -- blog section 3, both readings of the
  reset point (position == 0, and position == min(position)).
* ``packed_storage_rows`` -- the course's storage rows (inputs, targets,
  occurrence segments, local positions, validity) for next-fit placements
  ("Fill only the current row").
* ``unpad_index`` / ``gather_rows`` -- the padded-batch bridge of blog section 4
  (a 2-D attention mask: drop the padding, run the varlen kernel, scatter the output
  back to the padded shape).
"""
from __future__ import annotations

import numpy as np

PAD_CELL = -1
NO_SEGMENT = -1


def _check_lengths(lengths, capacity):
    for i, L in enumerate(lengths):
        if L <= 0:
            raise ValueError(f"document {i} has non-positive length {L}")
        if L > capacity:
            raise ValueError(f"document {i} of length {L} exceeds capacity {capacity}")


def next_fit(lengths, capacity: int):
    """Return packs as lists of document indices (input order kept)."""
    lengths = [int(x) for x in lengths]
    _check_lengths(lengths, capacity)
    packs, cur, used = [], [], 0
    for i, L in enumerate(lengths):
        if L > capacity - used:
            packs.append(cur)
            cur, used = [], 0
        cur.append(i)
        used += L
    if cur:
        packs.append(cur)
    return packs


def best_fit_decreasing(lengths, capacity: int):
    """Return packs as lists of document indices (see module docstring for ties)."""
    lengths = [int(x) for x in lengths]
    _check_lengths(lengths, capacity)
    order = sorted(range(len(lengths)), key=lambda i: (-lengths[i], i))
    remaining, packs = [], []
    for i in order:
        L = lengths[i]
        best = -1
        for b, rem in enumerate(remaining):
            if rem >= L and (best < 0 or rem < remaining[best]):
                best = b
        if best < 0:
            remaining.append(capacity - L)
            packs.append([i])
        else:
            remaining[best] -= L
            packs[best].append(i)
    return packs


def build_metadata(lengths, pad_to: int = 0):
    """cu_seqlens, position_ids, segment_ids, max_seqlen for one pack.

    ``lengths`` are the segment lengths in stream order.  If ``pad_to`` exceeds
    their sum, a tail pad segment of the difference is appended.
    """
    lengths = [int(x) for x in lengths]
    if any(L <= 0 for L in lengths):
        raise ValueError("segment lengths must be positive")
    total = sum(lengths)
    if pad_to and pad_to < total:
        raise ValueError("pad_to is smaller than the packed tokens")
    if pad_to > total:
        lengths = lengths + [pad_to - total]
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    position_ids = []
    segment_ids = []
    for b, L in enumerate(lengths):
        position_ids.extend(range(L))
        segment_ids.extend([b] * L)
    return (np.asarray(cu, dtype=np.int32), np.asarray(position_ids, dtype=np.int32),
            np.asarray(segment_ids, dtype=np.int32), max(lengths) if lengths else 0)


def cu_seqlens_from_position_ids(position_ids, reset_at_min: bool = False):
    """Boundary compilation of blog section 3.

    Reset points are the indices whose position equals 0 (or, with
    ``reset_at_min``, equals the minimum position); the total token count is
    appended.  Returns (cu_seqlens int32, max_seqlen).
    """
    p = np.asarray(position_ids).reshape(-1)
    sentinel = p.min() if reset_at_min else 0
    starts = [i for i in range(p.size) if p[i] == sentinel]
    cu = np.asarray(starts + [p.size], dtype=np.int32)
    return cu, int(np.diff(cu).max())


def boundary_plane_ok(position_ids, reset_at_min: bool = False, strict: bool = False) -> bool:
    """Contract check of a position plane used as the boundary carrier.

    The page (blog section 3) states the contract on the compiled array: int32,
    first value 0, last value T, strictly increasing.  Reset indices are
    distinct and below T, so the only way a plane breaks it is a first token
    that is not a reset point (cu[0] would not be 0), or an empty plane.
    ``strict`` adds the reading taken here for the repeated-values lesson of
    the mRoPE section (a plane that repeats coordinates inside a sample cannot
    carry boundaries): between resets the positions must count up by one.
    """
    p = np.asarray(position_ids).reshape(-1)
    if p.size == 0:
        return False
    sentinel = p.min() if reset_at_min else 0
    if p[0] != sentinel:
        return False
    if strict:
        for i in range(1, p.size):
            if p[i] != sentinel and p[i] != p[i - 1] + 1:
                return False
    return True


def packed_storage_rows(inputs, targets, capacity: int):
    """Course storage rows for next-fit placement of (input, target) pair lists.

    ``inputs[i]`` / ``targets[i]`` are the already formed pairs of document i.
    Returns a dict of row lists: inputs, targets, segments, positions,
    input_valid, target_valid (every real target is supervised here).
    """
    lengths = [len(x) for x in inputs]
    packs = next_fit(lengths, capacity)
    rows = {key: [] for key in ("inputs", "targets", "segments", "positions",
                                "input_valid", "target_valid")}
    for pack in packs:
        r_in = [PAD_CELL] * capacity
        r_tg = [PAD_CELL] * capacity
        r_seg = [NO_SEGMENT] * capacity
        r_pos = [0] * capacity
        r_val = [False] * capacity
        col = 0
        for doc in pack:
            for j, (a, t) in enumerate(zip(inputs[doc], targets[doc])):
                r_in[col] = a
                r_tg[col] = t
                r_seg[col] = doc
                r_pos[col] = j
                r_val[col] = True
                col += 1
        rows["inputs"].append(r_in)
        rows["targets"].append(r_tg)
        rows["segments"].append(r_seg)
        rows["positions"].append(r_pos)
        rows["input_valid"].append(r_val)
        rows["target_valid"].append(list(r_val))
    return rows


def unpad_index(mask):
    """Padded batch -> packed stream (blog section 4, the padded-batch path).

    ``mask`` [Bp, S]: nonzero marks a real token.  Each row's real tokens, in order, become
    one segment; a row without a real token is an error (it would be an empty segment, and
    cu_seqlens must be strictly increasing, blog section 3).  Returns (indices [Bp*S]:
    flat positions r*S + s of the T real tokens in row-major order, then -1 for the padding
    slots; inverse [Bp*S]: packed index of each position or -1; cu_seqlens [Bp+1]; T;
    max_seqlen).
    """
    m = np.asarray(mask).astype(bool)
    Bp, S = m.shape
    lens = m.sum(axis=1)
    if (lens == 0).any():
        raise ValueError("a row without real tokens would be an empty segment")
    real = [r * S + s for r in range(Bp) for s in range(S) if m[r, s]]
    T = len(real)
    indices = np.full(Bp * S, -1, dtype=np.int64)
    indices[:T] = real
    inverse = np.full(Bp * S, -1, dtype=np.int64)
    for i, flat in enumerate(real):
        inverse[flat] = i
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return indices, inverse, cu, T, int(lens.max())


def gather_rows(src, row_map):
    """dst[i] = src[row_map[i]] for row_map[i] >= 0, else a zero row (unpad with the indices,
    pad with the inverse map)."""
    src = np.asarray(src)
    dst = np.zeros((len(row_map),) + src.shape[1:], dtype=src.dtype)
    for i, r in enumerate(row_map):
        if r >= 0:
            dst[i] = src[r]
    return dst
