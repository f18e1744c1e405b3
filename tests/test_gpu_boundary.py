"""GPU parity for the boundary compiler (position_ids -> cu_seqlens), blog section 3.

Integer work: bit-exact against the oracle (cu_seqlens_from_position_ids,
boundary_plane_ok) on the same seeded positions.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import packing as op
import _workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    import packed_sequence_varlen_gb300 as pkg
    pkg._lib.load()
    return pkg


def run(va, positions, reset_at_min=False, strict=False):
    p = torch.tensor(np.asarray(positions, dtype=np.int32), device=DEV)
    cu, B, mx, st = va.cu_seqlens_from_position_ids(p, reset_at_min, strict)
    torch.cuda.synchronize()
    B = int(B.item())
    return cu[:B + 1].cpu().numpy(), B, int(mx.item()), int(st.item())


def expect(va, positions, reset_at_min=False, strict=False):
    cu, B, mx, st = run(va, positions, reset_at_min, strict)
    if op.boundary_plane_ok(positions, reset_at_min, strict):
        rcu, rmx = op.cu_seqlens_from_position_ids(positions, reset_at_min)
        assert st == 0
        assert np.array_equal(cu, rcu) and B == len(rcu) - 1 and mx == rmx
    else:
        assert st == 5 and B == 0 and mx == 0   # VA_ERR_BAD_SEQLENS


def test_page_example(va):
    """Blog section 3: positions 0..4 | 0..2 | 0..3 compile to [0, 5, 8, 12], max 5."""
    page = [0, 1, 2, 3, 4, 0, 1, 2, 0, 1, 2, 3]
    for at_min in (False, True):
        for strict in (False, True):
            cu, B, mx, st = run(va, page, at_min, strict)
            assert (cu.tolist(), B, mx, st) == ([0, 5, 8, 12], 3, 5, 0)
    shifted = [p + 1 for p in page]        # a scheme starting at 1 needs the minimum reading
    cu, B, mx, st = run(va, shifted, True, True)
    assert (cu.tolist(), B, mx, st) == ([0, 5, 8, 12], 3, 5, 0)
    assert run(va, shifted)[3] == 5        # reset-at-0: the first token is not a reset


@pytest.mark.parametrize("name", ["sft8k", "gqa16k", "long64k", "tiny4k"])
def test_workload_positions_round_trip(va, name):
    """Positions from the metadata builder compile back to its cu_seqlens, both readings."""
    for lengths in wl.packs(name)[:2]:
        cu, pos, _, mx = op.build_metadata(lengths)
        for at_min in (False, True):
            gcu, B, gmx, st = run(va, pos, at_min, True)
            assert st == 0 and np.array_equal(gcu, cu) and gmx == mx and B == len(lengths)
        # and from the GPU metadata kernel's own positions
        lens = torch.tensor(lengths, dtype=torch.int32, device=DEV)
        gcu0, gpos, _, _, _ = va.build_metadata(lens, pad_to=0, T_capacity=int(cu[-1]))
        c2, B2, m2, s2 = va.cu_seqlens_from_position_ids(gpos.contiguous(), False, True)
        torch.cuda.synchronize()
        assert int(s2.item()) == 0 and int(B2.item()) == len(lengths)
        assert torch.equal(c2[:len(lengths) + 1], gcu0[:len(lengths) + 1])


@pytest.mark.parametrize("seed", range(3))
def test_random_planes(va, seed):
    """Random lengths (1..300, many chunks per thread), and corrupted planes."""
    rng = np.random.default_rng(seed)
    lengths = rng.integers(1, 301, size=int(rng.integers(1, 3000))).tolist()
    _, pos, _, _ = op.build_metadata(lengths)
    base = int(rng.integers(0, 5))
    for at_min in (False, True):
        for strict in (False, True):
            expect(va, pos + (base if at_min else 0), at_min, strict)
    bad = pos.copy()
    i = int(rng.integers(1, bad.size)) if bad.size > 1 else 0
    bad[i] = bad[i] + 7                      # a jump inside a sample
    for strict in (False, True):
        expect(va, bad, False, strict)
    rep = np.repeat(np.arange(bad.size // 3 + 1), 3)[:bad.size].astype(np.int32)
    rep[0] = 0                               # repeated coordinates: 0 0 0 1 1 1 ...
    for strict in (False, True):
        expect(va, rep, False, strict)
    first = pos.copy()
    first[0] = 3                             # the first token is not a reset point
    expect(va, first, False, False)


def test_single_and_all_resets(va):
    expect(va, [0])
    expect(va, [0] * 5000, False, True)       # every token its own sample
    expect(va, [5, 5, 6], True, True)
    cu, B, mx, st = run(va, [0] * 5000)
    assert B == 5000 and mx == 1 and cu[-1] == 5000


def test_capacity_and_host_errors(va):
    lib = va._lib.load()
    p = torch.zeros(10, dtype=torch.int32, device=DEV)          # ten one-token samples
    cu = torch.empty(4, dtype=torch.int32, device=DEV)
    B, mx, st = (torch.empty(1, dtype=torch.int32, device=DEV) for _ in range(3))
    rc = lib.varlen_cu_seqlens_from_positions(va._ptr(p), 10, 0, 0, va._ptr(cu), 4, va._ptr(B), va._ptr(mx),
                                              va._ptr(st), va._stream(p.device))
    torch.cuda.synchronize()
    assert rc == 0 and int(st.item()) == 3 and int(B.item()) == 0   # VA_ERR_WORKSPACE
    rc = lib.varlen_cu_seqlens_from_positions(va._ptr(p), 0, 0, 0, va._ptr(cu), 4, va._ptr(B), va._ptr(mx),
                                              va._ptr(st), va._stream(p.device))
    assert rc == 1                                                 # VA_ERR_INVALID_ARG
    rc = lib.varlen_cu_seqlens_from_positions(None, 10, 0, 0, va._ptr(cu), 4, va._ptr(B), va._ptr(mx),
                                              va._ptr(st), va._stream(p.device))
    assert rc == 1
