"""The device-detected failure path: a bounded wait that runs out.

Every mbarrier wait in the attention kernels gives up after a limit, writes VA_ERR_TIMEOUT
into the workspace status word, raises its CTA's abort flag, drains and frees its tensor
memory.  The test hook varlen_test_stall_next_forward makes that happen without any fault:
the next forward's producers publish one work item and load nothing, so no copy or MMA is
in flight when the consumers' waits (limited to a few milliseconds) run out.  The outputs
stay unwritten, and the next ordinary call on the same stream still matches the oracle.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention as oa
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


@pytest.mark.parametrize("d", [64, 128])
def test_bounded_wait_runs_out_and_reports_timeout(va, d):
    lengths = [300, 700, 129, 1000]          # mean length above the token-tile threshold
    cu_h, _, _, mx = op.build_metadata(lengths)
    T, Hq, Hkv = int(cu_h[-1]), 4, 2
    q, k, v, do = si.tensors(T, Hq, Hkv, d, seed_offset=55 + d)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    cu = torch.tensor(cu_h, dtype=torch.int32, device=DEV)
    lib = va._lib.load()
    ws = torch.zeros(va.workspace_size(T, len(lengths), Hq, Hkv, d, mx, False), dtype=torch.uint8, device=DEV)
    out = torch.full_like(qd, 7.0)
    lse = torch.full((Hq, T), 7.0, dtype=torch.float32, device=DEV)

    assert lib.varlen_test_stall_next_forward(20_000_000) == 0       # 20 ms
    va.varlen_attn_fwd(qd, kd, vd, cu, mx, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert va.read_status(ws) == 6                                   # VA_ERR_TIMEOUT
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())     # nothing was written

    # the hook is one-shot and the context is still usable: the next call is ordinary
    out2, lse2 = va.varlen_attn_fwd(qd, kd, vd, cu, mx, workspace=ws, check_status=True)
    dq, dk, dv = va.varlen_attn_bwd(qd, kd, vd, out2, lse2, dod, cu, mx, check_status=True)
    torch.cuda.synchronize()
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    ro, rl = oa.varlen_forward(qq, kk, vv, cu_h)
    rg = oa.varlen_backward(qq, kk, vv, ro, rl, dd, cu_h)
    wl.assert_close_outputs(out2.double().cpu().numpy(), lse2.double().cpu().numpy(), ro, rl)
    wl.assert_close_grads(tuple(x.double().cpu().numpy() for x in (dq, dk, dv)), rg)


def test_stall_hook_rejects_limits_outside_its_range(va):
    lib = va._lib.load()
    assert lib.varlen_test_stall_next_forward(10) == 1
    assert lib.varlen_test_stall_next_forward(5_000_000_000) == 1
