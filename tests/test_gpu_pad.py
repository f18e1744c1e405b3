"""GPU parity of the padded-batch bridge (unpad, varlen attention, pad) against the oracle.

Index maps and cu_seqlens are bit-exact; gathered rows are copies (bit-exact); attention through
the bridge matches each row's own attention over its real tokens within the attention tolerances.
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


def make_mask(layout, lens, S, seed):
    rng = np.random.default_rng(seed)
    m = np.zeros((len(lens), S), dtype=np.int32)
    for r, L in enumerate(lens):
        if layout == "right":
            m[r, :L] = 1
        elif layout == "left":
            m[r, S - L:] = 1
        else:
            m[r, rng.choice(S, L, replace=False)] = 1
    return m


@pytest.mark.parametrize("layout", ["right", "left", "holes"])
def test_unpad_index_bit_exact(va, layout):
    """Maps and boundaries for rows spanning several 256-wide scan rounds, full and 1-token rows."""
    rng = np.random.default_rng(7)
    S = 700
    lens = [700, 1, 256, 257, 513, 3] + [int(x) for x in rng.integers(1, 701, 10)]
    m = make_mask(layout, lens, S, 8)
    idx, inv, cu, T, mx = va.unpad_index(torch.tensor(m, device=DEV))
    r_idx, r_inv, r_cu, r_T, r_mx = op.unpad_index(m)
    assert T == r_T and mx == r_mx
    assert np.array_equal(cu.cpu().numpy(), r_cu)
    assert np.array_equal(idx.cpu().numpy(), r_idx) and np.array_equal(inv.cpu().numpy(), r_inv)


def test_unpad_rejects_empty_row(va):
    m = torch.tensor([[1, 1, 0], [0, 0, 0]], dtype=torch.int32, device=DEV)
    with pytest.raises(va.VarlenError):
        va.unpad_index(m)


@pytest.mark.parametrize("layout,d,g", [("right", 128, 1), ("left", 64, 2), ("holes", 128, 2)])
def test_padded_batch_bridge(va, layout, d, g):
    """Padded Q/K/V [Bp, S, H, d] with a mask -> unpad -> varlen forward and backward -> pad:
    each row's output and gradients equal the oracle on that row's real tokens; padding is zero;
    pad(unpad(x)) is x on the real tokens, bit for bit."""
    Bp, S, Hkv = 5, 300, 2
    Hq = Hkv * g
    lens = [300, 17, 129, 1, 256]
    m = make_mask(layout, lens, S, 9)
    q, k, v, do = si.tensors(Bp * S, Hq, Hkv, d, seed_offset=31 + d + g)
    q, k, v, do = (x.reshape(Bp, S, x.shape[1], d) for x in (q, k, v, do))
    md = torch.tensor(m, device=DEV)
    idx, inv, cu, T, mx = va.unpad_index(md)
    pq, pk, pv, pdo = (va.unpad(x.to(DEV), idx, T) for x in (q, k, v, do))
    o, lse = va.varlen_attn_fwd(pq, pk, pv, cu, mx, None, True, check_status=True)
    dq, dk, dv = va.varlen_attn_bwd(pq, pk, pv, o, lse, pdo, cu, mx, None, True, check_status=True)
    outs = [va.pad(x, inv, Bp, S).cpu() for x in (o, dq, dk, dv)]
    back = va.pad(pq, inv, Bp, S).cpu()
    assert torch.equal(back, q * torch.tensor(m)[:, :, None, None].to(q.dtype))
    refs, gots = [[] for _ in range(4)], [[] for _ in range(4)]
    for r in range(Bp):  # the oracle on each row's own real tokens, one segment per row
        sel = m[r].astype(bool)
        rq, rk, rv, rdo = (si.to_f64(x[r][torch.tensor(sel)]) for x in (q, k, v, do))
        L = int(sel.sum())
        ro, rl = oa.varlen_forward(rq, rk, rv, [0, L])
        rg = oa.varlen_backward(rq, rk, rv, ro, rl, rdo, [0, L])
        for j, (a, b) in enumerate(zip(outs, (ro,) + tuple(rg))):
            gots[j].append(a[r][torch.tensor(sel)].double().numpy())
            refs[j].append(b)
            assert (a[r][torch.tensor(~sel)] == 0).all()   # padding stays zero
    got, ref = [np.concatenate(x) for x in gots], [np.concatenate(x) for x in refs]
    assert np.abs(got[0] - ref[0]).max() <= wl.O_MAX_ABS
    wl.assert_close_grads(tuple(got[1:]), tuple(ref[1:]))
