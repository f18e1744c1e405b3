"""GPU parity of cross-attention (Q and K/V cut by their own boundaries; causal aligned
bottom-right: query i of a segment sees keys j <= i + lk - lq) against the float64 oracle:
tile maps bit-exact, O / LSE / dQ / dK / dV within the attention tolerances."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import attention as oa
from oracle import tiles as ot
import _workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
VA_ERR_BAD_SEQLENS = 5
# query / key lengths: lq = lk, offsets that are and are not multiples of 64 / 128, a single
# query over many keys, 256 + 1 queries (a second q tile holding one row)
LQ = [1, 5, 17, 3, 40, 300, 129, 2, 257, 64]
LK = [1, 9, 17, 30, 41, 700, 129, 260, 300, 64]


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    import packed_sequence_varlen_gb300 as pkg
    pkg._lib.load()
    return pkg


def bounds(lq, lk):
    return [int(x) for x in np.cumsum([0] + lq)], [int(x) for x in np.cumsum([0] + lk)]


@pytest.mark.parametrize("causal", [True, False])
def test_cross_maps_bit_exact(va, causal):
    cuq, cuk = bounds(LQ, LK)
    cq, ck = (torch.tensor(x, dtype=torch.int32, device=DEV) for x in (cuq, cuk))
    for d, Hq, Hkv in ((128, 4, 2), (64, 8, 8)):
        for kind in (0, 1, 2):
            BM, BN = va.tile_sizes(kind, d)
            tm, n = va.plan_cross(cq, ck, cuq[-1], cuk[-1], Hq, Hkv, d, max(LQ), kind, causal)
            ref = (ot.bwd_tile_map(cuq, Hkv, BM, BN, causal, cu_k=cuk) if kind == 1
                   else ot.fwd_tile_map(cuq, Hq, BM, BN, causal, cu_k=cuk))
            assert n == len(ref)
            assert np.array_equal(tm.cpu().numpy(), ref)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d,g", [(64, 1), (128, 2)])
def test_cross_parity(va, causal, d, g):
    cuq, cuk = bounds(LQ, LK)
    Tq, Tk, Hkv = cuq[-1], cuk[-1], 2
    Hq = Hkv * g
    q, _, _, do = si.tensors(Tq, Hq, Hkv, d, seed_offset=500 + d + g)
    _, k, v, _ = si.tensors(Tk, Hq, Hkv, d, seed_offset=600 + d + g)
    cq, ck = (torch.tensor(x, dtype=torch.int32, device=DEV) for x in (cuq, cuk))
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, lse = va.varlen_attn_fwd_cross(qd, kd, vd, cq, ck, max(LQ), max(LK), None, causal, check_status=True)
    gr = va.varlen_attn_bwd_cross(qd, kd, vd, o, lse, dod, cq, ck, max(LQ), max(LK), None, causal,
                                  check_status=True)
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    ro, rl = oa.varlen_forward(qq, kk, vv, cuq, None, causal, cu_seqlens_k=cuk)
    rg = oa.varlen_backward(qq, kk, vv, ro, rl, dd, cuq, None, causal, cu_seqlens_k=cuk)
    wl.assert_close_outputs(o.cpu().double().numpy(), lse.cpu().double().numpy(), ro, rl)
    got = tuple(x.cpu().double().numpy() for x in gr)
    wl.assert_close_grads(got, rg)
    wl.assert_close_grads_chunked(got, rg)


def test_cross_equal_boundaries_match_self_attention(va):
    """cu_k = cu_q: the cross kernels give the self-attention kernels' results bit for bit (a pack
    whose mean segment length keeps the self path on segment records, as the cross path)."""
    lengths = [300, 117, 129, 100, 656]
    cu = [int(x) for x in np.cumsum([0] + lengths)]
    q, k, v, do = si.tensors(cu[-1], 4, 2, 128, seed_offset=77)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    o1, l1 = va.varlen_attn_fwd(qd, kd, vd, cud, 656, None, True)
    o2, l2 = va.varlen_attn_fwd_cross(qd, kd, vd, cud, cud, 656, 656, None, True, check_status=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = va.varlen_attn_bwd(qd, kd, vd, o1, l1, dod, cud, 656, None, True)
    g2 = va.varlen_attn_bwd_cross(qd, kd, vd, o2, l2, dod, cud, cud, 656, 656, None, True, check_status=True)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_cross_rejects_more_queries_than_keys(va):
    """Causal cross-attention needs lq <= lk in every segment: the device reports it."""
    cuq, cuk = bounds([5, 8], [9, 3])
    q, _, _, _ = si.tensors(13, 2, 2, 64, seed_offset=1)
    _, k, v, _ = si.tensors(12, 2, 2, 64, seed_offset=2)
    cq, ck = (torch.tensor(x, dtype=torch.int32, device=DEV) for x in (cuq, cuk))
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    va.varlen_attn_fwd_cross(q.to(DEV), k.to(DEV), v.to(DEV), cq, ck, 8, 9, None, True, workspace=ws)
    assert va.read_status(ws) == VA_ERR_BAD_SEQLENS
    va.varlen_attn_fwd_cross(q.to(DEV), k.to(DEV), v.to(DEV), cq, ck, 8, 9, None, False, workspace=ws)
    assert va.read_status(ws) == 0  # non-causal: any lengths
