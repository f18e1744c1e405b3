"""Test helpers: the oracle-side view of each workload's packs, and comparisons.

Pack lengths here come from the ORACLE planner (the GPU-side planner is checked
against it separately); tensors come from ``seeded_inputs``.
"""
from __future__ import annotations

import numpy as np

import seeded_inputs as si
from oracle import packing as op

# Tolerances for the GPU path against the float64 oracle on the same bf16 inputs.
O_MAX_ABS = 2e-2
LSE_MAX_ABS = 1e-3
GRAD_REL_L2 = 1e-2


def real_packs(name: str):
    """(document lengths, pad_to) per pack: what the metadata kernel receives."""
    w = si.WORKLOADS[name]
    lengths = si.raw_lengths(name).tolist()
    if w.strategy == "fixed":
        groups = [list(range(len(lengths)))]
    elif w.strategy == "next_fit":
        groups = op.next_fit(lengths, w.capacity)
    else:
        groups = op.best_fit_decreasing(lengths, w.capacity)
    if w.packs_used:
        groups = groups[:w.packs_used]   # e.g. tiny4k: the first 131072-token row
    return [([lengths[i] for i in g], w.pad_to) for g in groups]


def packs(name: str):
    """All packs of a workload as lists of segment lengths (tail pad segment included)."""
    out = []
    for segs, pad_to in real_packs(name):
        segs = list(segs)
        if pad_to and sum(segs) < pad_to:
            segs.append(pad_to - sum(segs))
        out.append(segs)
    return out


def pack(name: str, index: int = 0):
    return packs(name)[index]


def most_segments_pack(name: str) -> int:
    p = packs(name)
    return int(np.argmax([len(x) for x in p]))


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_close_outputs(o, lse, ref_o, ref_lse):
    m = ~np.isnan(ref_o)
    err = np.abs(o[m] - ref_o[m]).max()
    assert err <= O_MAX_ABS, f"O max-abs {err}"
    ml = ~np.isnan(ref_lse)
    err = np.abs(lse[ml] - ref_lse[ml]).max()
    assert err <= LSE_MAX_ABS, f"LSE max-abs {err}"


def assert_close_grads(grads, refs):
    for name, a, b in zip(("dq", "dk", "dv"), grads, refs):
        m = ~np.isnan(b)
        r = rel_l2(a[m], b[m])
        assert r <= GRAD_REL_L2, f"{name} rel-L2 {r}"


def assert_close_grads_chunked(grads, refs, rows: int = 64, tol: float = 2 * GRAD_REL_L2):
    """Relative L2 per chunk of `rows` consecutive token rows, so that an error confined to a
    few rows (a mask off by one at a tile edge) is not averaged away.  A chunk's norm is
    floored at a tenth of the mean chunk norm: chunks whose gradient is (nearly) zero, such
    as dQ of single-token segments, are compared in absolute terms."""
    for name, a, b in zip(("dq", "dk", "dv"), grads, refs):
        n = a.shape[0] // rows * rows
        if n == 0:
            continue
        da = (a[:n] - b[:n]).reshape(n // rows, -1)
        nb = np.linalg.norm(b[:n].reshape(n // rows, -1), axis=1)
        err = np.linalg.norm(da, axis=1) / np.maximum(nb, 0.1 * nb.mean() + 1e-30)
        worst = int(np.argmax(err))
        assert err[worst] <= tol, f"{name} rows [{worst * rows}, {(worst + 1) * rows}) rel-L2 {err[worst]}"
