"""varlen_validate_cu_seqlens through the C ABI against the oracle's contract check.

The contract ("Packing与 FlashAttention Varlen", section 3): int32 boundaries, first 0, last
T, strictly increasing; here also every length at most max_seqlen (the bound plans are
sized by).  A violation writes VA_ERR_BAD_SEQLENS (5) into the status word; a valid array
leaves the word exactly as the caller left it.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as oa

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SENTINEL = 12345   # a status value the kernel never writes


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    from packed_sequence_varlen_gb300 import _lib
    return _lib.load()


def oracle_verdict(cu, T, max_seqlen):
    try:
        c = oa.check_cu_seqlens(cu, T)
    except ValueError:
        return 5
    return 5 if int(np.diff(c).max()) > max_seqlen else SENTINEL


def run(lib, cu, T, max_seqlen, initial=SENTINEL):
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    status = torch.tensor([initial], dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream(torch.device(DEV)).cuda_stream)
    st = lib.varlen_validate_cu_seqlens(ctypes.c_void_p(cud.data_ptr()), len(cu) - 1, T, max_seqlen,
                                        ctypes.c_void_p(status.data_ptr()), stream)
    assert st == 0, lib.varlen_last_error()
    torch.cuda.synchronize()
    return int(status.item())


CASES = [
    ([0, 5, 8, 12], 12, 5, "the page's three samples"),
    ([0, 12], 12, 12, "one segment"),
    ([0, 5, 8, 12], 12, 4, "a length above max_seqlen"),
    ([0, 8, 5, 12], 12, 8, "not increasing"),
    ([1, 5, 8, 12], 12, 5, "first entry not 0"),
    ([0, 5, 8, 11], 12, 5, "last entry not T"),
    ([0, 5, 8, 13], 12, 5, "last entry past T"),
    ([0, 5, 5, 12], 12, 7, "a zero-length segment"),
    ([0, -3, 12], 12, 15, "a negative boundary"),
]


@pytest.mark.parametrize("cu,T,mx,what", CASES, ids=[c[3] for c in CASES])
def test_validate_small_cases(lib, cu, T, mx, what):
    assert run(lib, cu, T, mx) == oracle_verdict(cu, T, mx)


def test_validate_many_segments_and_corruptions(lib):
    """Thousands of boundaries (more than one thread's share of the block) with one corruption
    at a time, at the start, in the middle and at the end."""
    rng = np.random.default_rng(7)
    lengths = rng.integers(1, 65, 5000)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T, mx = int(cu[-1]), int(lengths.max())
    assert run(lib, cu.tolist(), T, mx) == SENTINEL
    assert run(lib, cu.tolist(), T, mx, initial=0) == 0     # a valid array writes nothing
    for at in (1, 2, 1234, 2500, 4999):
        bad = cu.copy()
        bad[at] = bad[at - 1]                                # zero-length segment
        assert run(lib, bad.tolist(), T, mx) == oracle_verdict(bad, T, mx) == 5
        bad = cu.copy()
        bad[at], bad[at + 1] = bad[at + 1], bad[at]          # two boundaries swapped
        assert run(lib, bad.tolist(), T, mx) == oracle_verdict(bad, T, mx) == 5
    assert run(lib, cu.tolist(), T, mx - 1) == 5             # max_seqlen one below the longest
