"""The allocation-free forward entry point, called through the C ABI.

varlen_attn_fwd_noalloc exists for callers that cannot allocate device memory
where they run attention (a plugin inside a runtime that owns every device
allocation, or a serving loop that must not call cudaMalloc because it can
synchronise the device).  Its scratch is a static device array shared by all
calls; this test checks that two calls in a row give the same results as the
workspace-based entry point.  It lives in a file of its own that pytest
collects last, and it passes alone in a fresh process or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import packing as op

pytestmark = pytest.mark.gpu

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


def test_noalloc_forward_matches_workspace_forward_twice(lib):
    from packed_sequence_varlen_gb300 import _lib
    dev = torch.device("cuda:0")
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    cases = [([300, 77, 129, 1000, 5], 4, 2, 128), ([5, 3, 4], 2, 2, 64)]
    for lengths, Hq, Hkv, d in cases:
        cu_h, _, _, mx = op.build_metadata(lengths)
        T = int(cu_h[-1])
        q, k, v = (x.to(dev) for x in si.tensors(T, Hq, Hkv, d, seed_offset=31, with_dout=False))
        cu = torch.tensor(cu_h, dtype=torch.int32, device=dev)
        shape = _lib.VaShape()
        lib.varlen_shape_contiguous(ctypes.byref(shape), T, len(lengths), Hq, Hkv, d, mx)
        scale = 1.0 / np.sqrt(d)
        # the existing entry point, with a caller workspace
        ws = torch.zeros(lib.varlen_attn_workspace_size(ctypes.byref(shape), 0), dtype=torch.uint8,
                         device=dev)
        o_ref = torch.empty_like(q)
        l_ref = torch.empty((Hq, T), dtype=torch.float32, device=dev)
        st = lib.varlen_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), ctypes.byref(shape), scale, 1,
                                 _ptr(o_ref), _ptr(l_ref), _ptr(ws), ws.numel(), stream)
        assert st == 0, lib.varlen_last_error()
        for _ in range(2):   # the static scratch keeps the last call's contents
            o = torch.full_like(q, float("nan"))
            lse = torch.full((Hq, T), float("nan"), dtype=torch.float32, device=dev)
            st = lib.varlen_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), ctypes.byref(shape),
                                             scale, 1, _ptr(o), _ptr(lse), stream)
            assert st == 0, lib.varlen_last_error()
            torch.cuda.synchronize()
            assert float((o.float() - o_ref.float()).abs().max()) <= O_MAX_ABS
            assert float((lse - l_ref).abs().max()) <= LSE_MAX_ABS


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    from packed_sequence_varlen_gb300 import _lib
    shape = _lib.VaShape()
    # (T/256 + B) * Hq = (131072/256 + 4000) * 32 > 65520 records
    lib.varlen_shape_contiguous(ctypes.byref(shape), 131072, 4000, 32, 32, 128, 64)
    p = ctypes.c_void_p(256)
    st = lib.varlen_attn_fwd_noalloc(p, p, p, p, ctypes.byref(shape), 0.1, 1, p, p, None)
    assert st == 3
    assert b"1048576" in lib.varlen_last_error()
