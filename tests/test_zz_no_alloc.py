"""The allocation-free forward entry point, called through the C ABI.

varlen_attn_fwd_noalloc exists for callers that cannot allocate device memory
where they run attention (a plugin inside a runtime that owns every device
allocation, or a serving loop that must not call cudaMalloc because it can
synchronise the device).  Its scratch is a static device array shared by all
calls, so these tests check that consecutive calls -- a small shape, then
larger ones whose tile maps reach past the earlier records -- give results
bit-identical to the workspace-based entry point (same kernels, same map),
that the output also matches the oracle, that a contract violation is
reported through varlen_noalloc_read_status, and that the size limit is
exactly varlen_attn_workspace_size(shape, 0) <= 1 MiB.  The file is collected
last and passes alone in a fresh process or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention as oa
from oracle import packing as op

pytestmark = pytest.mark.gpu

SCRATCH = 1 << 20
O_MAX_ABS = 2e-2      # the forward tolerances of the parity tests
LSE_MAX_ABS = 1e-3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    from packed_sequence_varlen_gb300 import _lib
    return _lib.load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream(torch.device("cuda:0")).cuda_stream)


def _shape(lib, T, B, Hq, Hkv, d, mx):
    from packed_sequence_varlen_gb300 import _lib
    s = _lib.VaShape()
    lib.varlen_shape_contiguous(ctypes.byref(s), T, B, Hq, Hkv, d, mx)
    return s


def _largest_b_inside(lib, T, Hq, d):
    """The largest segment count whose forward workspace still fits the 1 MiB array."""
    lo, hi = 1, T
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if lib.varlen_attn_workspace_size(ctypes.byref(_shape(lib, T, mid, Hq, Hq, d, 1)), 0) <= SCRATCH:
            lo = mid
        else:
            hi = mid - 1
    return lo


def _noalloc_status(lib):
    st = ctypes.c_int32(-1)
    assert lib.varlen_noalloc_read_status(ctypes.byref(st), _stream()) == 0, lib.varlen_last_error()
    return st.value


def _workspace_forward(lib, q, k, v, cu, shape, scale):
    dev = q.device
    T, Hq = q.shape[0], q.shape[1]
    ws = torch.zeros(lib.varlen_attn_workspace_size(ctypes.byref(shape), 0), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    st = lib.varlen_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), ctypes.byref(shape), scale, 1,
                             _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream())
    assert st == 0, lib.varlen_last_error()
    return o, lse


def _boundary_lengths(T, B, seed):
    """B positive lengths summing to T (mostly short segments, one long remainder)."""
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(1, max(2, 2 * (T // B)), B - 1)]
    while sum(lengths) > T - 1:
        lengths = [max(1, x // 2) for x in lengths]
    return lengths + [T - sum(lengths)]


def test_noalloc_forward_bit_identical_to_workspace_forward(lib):
    dev = torch.device("cuda:0")
    # a small shape first, then larger ones: the later tile maps run past the earlier
    # records left in the shared array, and the last one sits at the size limit
    T_b, H_b, d_b = 65536, 8, 64
    B_b = _largest_b_inside(lib, T_b, H_b, d_b)
    cases = [([5, 3, 4], 2, 2, 64, True),
             ([300, 77, 129, 1000, 5], 4, 2, 128, True),
             (_boundary_lengths(T_b, B_b, 3), H_b, H_b, d_b, False)]
    for lengths, Hq, Hkv, d, oracle_check in cases:
        cu_h, _, _, mx = op.build_metadata(lengths)
        T = int(cu_h[-1])
        q, k, v = si.tensors(T, Hq, Hkv, d, seed_offset=31, with_dout=False)
        qd, kd, vd = (x.to(dev) for x in (q, k, v))
        cu = torch.tensor(cu_h, dtype=torch.int32, device=dev)
        shape = _shape(lib, T, len(lengths), Hq, Hkv, d, mx)
        assert lib.varlen_attn_workspace_size(ctypes.byref(shape), 0) <= SCRATCH
        scale = 1.0 / np.sqrt(d)
        o_ref, l_ref = _workspace_forward(lib, qd, kd, vd, cu, shape, scale)
        for _ in range(2):   # the static scratch keeps the last call's contents
            o = torch.full_like(qd, float("nan"))
            lse = torch.full((Hq, T), float("nan"), dtype=torch.float32, device=dev)
            st = lib.varlen_attn_fwd_noalloc(_ptr(qd), _ptr(kd), _ptr(vd), _ptr(cu), ctypes.byref(shape),
                                             scale, 1, _ptr(o), _ptr(lse), _stream())
            assert st == 0, lib.varlen_last_error()
            assert _noalloc_status(lib) == 0
            assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
        if oracle_check:
            ro, rl = oa.varlen_forward(si.to_f64(q), si.to_f64(k), si.to_f64(v), cu_h, scale)
            assert np.abs(o.double().cpu().numpy() - ro).max() <= O_MAX_ABS
            assert np.abs(lse.double().cpu().numpy() - rl).max() <= LSE_MAX_ABS


def test_noalloc_reports_a_bad_boundary_array(lib):
    dev = torch.device("cuda:0")
    T, H, d = 64, 2, 64
    q, k, v = (x.to(dev) for x in si.tensors(T, H, H, d, with_dout=False))
    shape = _shape(lib, T, 3, H, H, d, 40)
    bad = torch.tensor([0, 30, 20, 64], dtype=torch.int32, device=dev)   # not increasing
    out = torch.full_like(q, 7.0)
    lse = torch.full((H, T), 7.0, dtype=torch.float32, device=dev)
    st = lib.varlen_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(bad), ctypes.byref(shape), 0.125, 1,
                                     _ptr(out), _ptr(lse), _stream())
    assert st == 0, lib.varlen_last_error()
    assert _noalloc_status(lib) == 5        # VA_ERR_BAD_SEQLENS
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    good = torch.tensor([0, 30, 50, 64], dtype=torch.int32, device=dev)
    st = lib.varlen_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(good), ctypes.byref(shape), 0.125, 1,
                                     _ptr(out), _ptr(lse), _stream())
    assert st == 0 and _noalloc_status(lib) == 0   # the next call starts from a clean status


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    T, H, d = 65536, 8, 64
    B = _largest_b_inside(lib, T, H, d)
    past = _shape(lib, T, B + 1, H, H, d, 1)
    assert lib.varlen_attn_workspace_size(ctypes.byref(past), 0) > SCRATCH
    p = ctypes.c_void_p(256)
    st = lib.varlen_attn_fwd_noalloc(p, p, p, p, ctypes.byref(past), 0.1, 1, p, p, None)
    assert st == 3
    assert b"1048576" in lib.varlen_last_error()
    big = _shape(lib, 131072, 4000, 32, 32, 128, 64)
    assert lib.varlen_attn_fwd_noalloc(p, p, p, p, ctypes.byref(big), 0.1, 1, p, p, None) == 3
