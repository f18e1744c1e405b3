"""GPU parity of the causal local window (query i sees keys i - w .. i of its segment)
against the float64 oracle: tile maps bit-exact, O / LSE / dQ / dK / dV within the
attention tolerances, and the closed form w = 0 (each query sees only itself: O = v)."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention as oa
from oracle import packing as op
from oracle import tiles as ot
import _workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
EDGE = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 1, 383, 384, 385]


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    import packed_sequence_varlen_gb300 as pkg
    pkg._lib.load()
    return pkg


def oracle_map(va, kind, cu, Hq, Hkv, d, w):
    BM, BN = va.tile_sizes(kind, d)
    if kind == 1:
        return ot.bwd_tile_map(cu, Hkv, BM, BN, True, 0, window=w)
    return ot.fwd_tile_map(cu, Hq, BM, BN, True, 0, window=w)


@pytest.mark.parametrize("w", [0, 1, 63, 64, 127, 128, 200, 512, 5000])
def test_window_maps_bit_exact(va, w):
    for lengths, Hq, Hkv, d in ((EDGE, 4, 2, 128), (wl.pack("sft8k", 0), 32, 32, 128),
                                (wl.pack("tiny4k")[:300], 8, 8, 64), (wl.pack("long64k"), 16, 16, 128)):
        cu, _, _, mx = op.build_metadata(lengths)
        cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
        for kind in (0, 1, 2):
            tm, n = va.plan(cud, int(cu[-1]), Hq, Hkv, d, mx, kind, True, window=w)
            ref = oracle_map(va, kind, cu, Hq, Hkv, d, w)
            assert n == len(ref)
            assert np.array_equal(tm.cpu().numpy(), ref)


def run_both(va, q, k, v, do, cu, mx, w):
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    o, lse = va.varlen_attn_fwd(qd, kd, vd, cud, mx, None, True, check_status=True, window=w)
    g = va.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cud, mx, None, True, check_status=True, window=w)
    torch.cuda.synchronize()
    return o.cpu().double().numpy(), lse.cpu().double().numpy(), tuple(x.cpu().double().numpy() for x in g)


@pytest.mark.parametrize("w", [0, 1, 100, 300])
@pytest.mark.parametrize("d,g", [(64, 1), (128, 2)])
def test_window_parity_ragged(va, w, d, g):
    cu, _, _, mx = op.build_metadata(EDGE)
    T, Hkv = int(cu[-1]), 2
    q, k, v, do = si.tensors(T, Hkv * g, Hkv, d, seed_offset=300 + w + d + g)
    o, lse, gr = run_both(va, q, k, v, do, cu, mx, w)
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    ro, rl = oa.varlen_forward(qq, kk, vv, cu, window=w)
    rg = oa.varlen_backward(qq, kk, vv, ro, rl, dd, cu, window=w)
    wl.assert_close_outputs(o, lse, ro, rl)
    if w == 0:
        # each query sees only itself: P = 1, so O is exactly its v row, dS = P (dP - D) = 0
        # (dQ = dK = 0 up to the rounding of dP - D) and dV = the group's dO
        assert np.array_equal(o, np.repeat(si.to_f64(v), g, axis=1))
        assert np.abs(gr[0]).max() < 1e-4 and np.abs(gr[1]).max() < 1e-4
        assert wl.rel_l2(gr[2], rg[2]) <= wl.GRAD_REL_L2
        return
    wl.assert_close_grads(gr, rg)
    wl.assert_close_grads_chunked(gr, rg)


def test_window_sft8k_pack(va):
    """One sft8k pack (segments up to 2048 tokens) with a 512-key window, all heads on the GPU,
    two kv heads against the oracle."""
    w_ = si.WORKLOADS["sft8k"]
    lengths = wl.pack("sft8k", 1)
    cu, _, _, mx = op.build_metadata(lengths)
    q, k, v, do = si.tensors(int(cu[-1]), w_.Hq, w_.Hkv, w_.d, seed_offset=901)
    o, lse, gr = run_both(va, q, k, v, do, cu, mx, 512)
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    ro, rl = oa.varlen_forward(qq, kk, vv, cu, kv_heads=[3, 20], window=512)
    rg = oa.varlen_backward(qq, kk, vv, ro, rl, dd, cu, kv_heads=[3, 20], window=512)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(gr, rg)


def test_window_autograd_and_rejections(va):
    cu, _, _, mx = op.build_metadata([70, 5, 200])
    T = int(cu[-1])
    q, k, v, do = si.tensors(T, 2, 2, 64, seed_offset=5)
    qd, kd, vd = (x.to(DEV).requires_grad_(True) for x in (q, k, v))
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out = va.varlen_attn(qd, kd, vd, cud, mx, window=33)
    out.backward(do.to(DEV))
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    ro, rl = oa.varlen_forward(qq, kk, vv, cu, window=33)
    rg = oa.varlen_backward(qq, kk, vv, ro, rl, dd, cu, window=33)
    assert np.abs(out.detach().cpu().double().numpy() - ro).max() <= wl.O_MAX_ABS
    wl.assert_close_grads(tuple(x.grad.cpu().double().numpy() for x in (qd, kd, vd)), rg)
    with pytest.raises(va.VarlenError):  # a window needs causal attention
        va.varlen_attn_fwd(qd.detach(), kd.detach(), vd.detach(), cud, mx, None, False, window=8)
