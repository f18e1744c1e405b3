"""Pins for the float64 attention oracle (CPU only).

Each pin checks the oracle against something other than itself: the dense
permission-matrix definition, torch's float64 SDPA and autograd, central
finite differences, closed forms and segment invariants.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import packing as op

TOL_ABS, TOL_REL = 1e-10, 1e-9   # course "Optional practice": abs 1e-10 + rel 1e-9


def close(a, b, abs_=TOL_ABS, rel=TOL_REL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.all(np.abs(a - b) <= abs_ + rel * np.maximum(np.abs(a), np.abs(b)))


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def random_pack(seed, T_max=40, Hq=4, Hkv=2, d=8):
    rng = np.random.default_rng(seed)
    lengths = []
    while sum(lengths) < T_max:
        lengths.append(int(rng.integers(1, 12)))
    cu, pos, seg, _ = op.build_metadata(lengths)
    T = int(cu[-1])
    q = rand((T, Hq, d), seed + 1)
    k = rand((T, Hkv, d), seed + 2)
    v = rand((T, Hkv, d), seed + 3)
    do = rand((T, Hq, d), seed + 4)
    return cu, pos, seg, q, k, v, do


@pytest.mark.parametrize("seed", range(8))
def test_matches_dense_permission_matrix(seed):
    """Per-segment oracle == brute-force [T,T] permission matrix, fwd and autograd bwd."""
    cu, pos, seg, q, k, v, do = random_pack(seed)
    T, Hq, d = q.shape
    scale = 0.37
    o, lse = oa.varlen_forward(q, k, v, cu, scale)
    dq, dk, dv = oa.varlen_backward(q, k, v, o, lse, do, cu, scale)

    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    valid = np.ones(T, dtype=bool)
    to, tl, allowed = oa.dense_permission_attention(tq, tk, tv, seg, pos, valid, scale)
    (to * torch.tensor(do)).sum().backward()
    assert close(o, to.detach().numpy(), 1e-12, 1e-12)
    assert close(lse, tl.detach().numpy(), 1e-12, 1e-12)
    assert close(dq, tq.grad.numpy(), 1e-12, 1e-10)
    assert close(dk, tk.grad.numpy(), 1e-12, 1e-10)
    assert close(dv, tv.grad.numpy(), 1e-12, 1e-10)
    # permission matrix: one causal block per segment
    for i in range(T):
        for j in range(T):
            same = seg[i] == seg[j]
            assert bool(allowed[i, j]) == (same and pos[j] <= pos[i])


def test_dense_brute_force_pad_query_zero_mixture():
    """An inactive pad query skips softmax and mixes nothing (course, 'Permission depends on the example')."""
    T, H, d = 6, 1, 4
    q, k, v = (torch.tensor(rand((T, H, d), s)) for s in (1, 2, 3))
    seg = [0, 0, 0, 1, 1, -1]
    pos = [0, 1, 2, 0, 1, 0]
    valid = [True] * 5 + [False]
    o, lse, allowed = oa.dense_permission_attention(q, k, v, seg, pos, valid, 0.5)
    assert torch.all(o[5] == 0) and torch.isinf(lse[0, 5])
    assert not allowed[5].any() and not allowed[:, 5].any()


@pytest.mark.parametrize("causal", [True, False])
def test_each_segment_equals_torch_sdpa_float64(causal):
    """Library special case: every slice equals torch SDPA on that slice alone (fwd and grads)."""
    cu, pos, seg, q, k, v, do = random_pack(11, T_max=60, Hq=4, Hkv=4, d=16)
    scale = 1.0 / np.sqrt(16)
    o, lse = oa.varlen_forward(q, k, v, cu, scale, causal)
    dq, dk, dv = oa.varlen_backward(q, k, v, o, lse, do, cu, scale, causal)
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        tq, tk, tv = (torch.tensor(x[s:e].transpose(1, 0, 2).copy(), requires_grad=True)
                      for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                              scale=scale)
        (to * torch.tensor(do[s:e].transpose(1, 0, 2).copy())).sum().backward()
        assert close(o[s:e], to.detach().numpy().transpose(1, 0, 2), 1e-12, 1e-10)
        assert close(dq[s:e], tq.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
        assert close(dk[s:e], tk.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
        assert close(dv[s:e], tv.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)


def test_gqa_group_mapping_against_sdpa():
    """q head h reads kv head h // (Hq/Hkv); dk/dv sum over the group."""
    T, Hq, Hkv, d = 9, 6, 2, 8
    cu = [0, 9]
    q, k, v, do = rand((T, Hq, d), 1), rand((T, Hkv, d), 2), rand((T, Hkv, d), 3), rand((T, Hq, d), 4)
    o, lse = oa.varlen_forward(q, k, v, cu, 0.3)
    dq, dk, dv = oa.varlen_backward(q, k, v, o, lse, do, cu, 0.3)
    tq = torch.tensor(q.transpose(1, 0, 2).copy(), requires_grad=True)
    tk = torch.tensor(k.transpose(1, 0, 2).copy(), requires_grad=True)
    tv = torch.tensor(v.transpose(1, 0, 2).copy(), requires_grad=True)
    kk = tk.repeat_interleave(3, dim=0)
    vv = tv.repeat_interleave(3, dim=0)
    to = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, is_causal=True, scale=0.3)
    (to * torch.tensor(do.transpose(1, 0, 2).copy())).sum().backward()
    assert close(o, to.detach().numpy().transpose(1, 0, 2), 1e-12, 1e-10)
    assert close(dk, tk.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
    assert close(dv, tv.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)


def test_finite_differences_of_backward():
    """Central differences (h=1e-6) of L = sum(O * dO) match the analytic gradient."""
    cu, pos, seg, q, k, v, do = random_pack(5, T_max=14, Hq=2, Hkv=1, d=4)
    scale = 0.6
    o, lse = oa.varlen_forward(q, k, v, cu, scale)
    grads = oa.varlen_backward(q, k, v, o, lse, do, cu, scale)
    h = 1e-6
    rng = np.random.default_rng(0)
    for which, g in zip(range(3), grads):
        for _ in range(12):
            arrs = [q.copy(), k.copy(), v.copy()]
            idx = tuple(rng.integers(0, n) for n in arrs[which].shape)
            arrs[which][idx] += h
            lp = (oa.varlen_forward(*arrs, cu, scale)[0] * do).sum()
            arrs[which][idx] -= 2 * h
            lm = (oa.varlen_forward(*arrs, cu, scale)[0] * do).sum()
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-7 + 1e-6 * abs(fd)


def test_page_layout_three_independent_attentions(golden_dir):
    """Blog section 1: [0,5,8,12] is three independent attentions."""
    fx = json.load(open(os.path.join(golden_dir, "three_samples_layout.json")))
    cu = fx["cu_seqlens"]
    T, H, d = 12, 2, 64
    q, k, v, do = rand((T, H, d), 1), rand((T, H, d), 2), rand((T, H, d), 3), rand((T, H, d), 4)
    scale = 1 / 8.0
    o, lse = oa.varlen_forward(q, k, v, cu, scale)
    for b in range(3):
        s, e = cu[b], cu[b + 1]
        ob, lb = oa.varlen_forward(q[s:e], k[s:e], v[s:e], [0, e - s], scale)
        assert np.array_equal(o[s:e], ob) and np.array_equal(lse[:, s:e], lb)


def test_merge_changes_only_b_c(golden_dir):
    """Blog section 1: merging to [0,5,12] makes A/(B+C).

    A's rows are bit-identical.  Causally, B's queries still see only B's keys,
    so B's O, LSE and dQ agree (to rounding); C's rows change, and B's dK/dV
    change because C's queries now read B's keys.
    """
    fx = json.load(open(os.path.join(golden_dir, "three_samples_layout.json")))
    T, H, d = 12, 2, 64
    q, k, v, do = rand((T, H, d), 1), rand((T, H, d), 2), rand((T, H, d), 3), rand((T, H, d), 4)
    scale = 1 / 8.0
    res = {}
    for name in ("cu_seqlens", "merged_cu_seqlens"):
        cu = fx[name]
        o, lse = oa.varlen_forward(q, k, v, cu, scale)
        res[name] = (o, lse) + oa.varlen_backward(q, k, v, o, lse, do, cu, scale)
    a, m = res["cu_seqlens"], res["merged_cu_seqlens"]
    for x, y in zip(a, m):
        sl = (slice(None), slice(0, 5)) if x.ndim == 2 else (slice(0, 5),)
        assert np.array_equal(x[sl], y[sl])                 # A untouched
    o, lse, dq, dk, dv = a
    o2, lse2, dq2, dk2, dv2 = m
    assert close(o[5:8], o2[5:8], 1e-13, 1e-12)            # B's O unchanged (causal)
    assert close(lse[:, 5:8], lse2[:, 5:8], 1e-13, 1e-12)
    assert close(dq[5:8], dq2[5:8], 1e-13, 1e-12)
    assert not close(o[8:], o2[8:])                          # C changes
    assert not close(dk[5:8], dk2[5:8])                      # B's keys now read by C
    # non-causal: both B's and C's outputs change
    on, _ = oa.varlen_forward(q, k, v, fx["cu_seqlens"], scale, causal=False)
    on2, _ = oa.varlen_forward(q, k, v, fx["merged_cu_seqlens"], scale, causal=False)
    assert np.array_equal(on[:5], on2[:5])
    assert not close(on[5:8], on2[5:8]) and not close(on[8:], on2[8:])


def test_closed_forms():
    """First query: O = v_0, LSE = scale q.k; length-1 segments: dQ = dK = 0 (to rounding) and dV = sum of the
    group's dO; Q = 0: prefix mean of V and LSE = ln(i+1); constant V rows: O constant."""
    T, Hq, Hkv, d = 15, 4, 2, 8
    cu = [0, 1, 5, 6, 12, 13, 15]
    q, k, v, do = rand((T, Hq, d), 1), rand((T, Hkv, d), 2), rand((T, Hkv, d), 3), rand((T, Hq, d), 4)
    scale = 0.4
    o, lse = oa.varlen_forward(q, k, v, cu, scale)
    dq, dk, dv = oa.varlen_backward(q, k, v, o, lse, do, cu, scale)
    g = Hq // Hkv
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        for h in range(Hq):
            assert np.array_equal(o[s, h], v[s, h // g])
            assert abs(lse[h, s] - scale * q[s, h] @ k[s, h // g]) < 1e-13
        if e - s == 1:
            # dS = P (dP - D) with P = 1 and dP = D up to summation order
            assert np.abs(dq[s]).max() < 1e-13 and np.abs(dk[s]).max() < 1e-13
            for hk in range(Hkv):
                assert close(dv[s, hk], do[s, hk * g:(hk + 1) * g].sum(0), 1e-14, 1e-13)
    z = np.zeros_like(q)
    o0, l0 = oa.varlen_forward(z, k, v, cu, scale)
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        for i in range(e - s):
            for h in range(Hq):
                assert close(o0[s + i, h], v[s:s + i + 1, h // g].mean(0), 1e-14, 1e-12)
                assert abs(l0[h, s + i] - np.log(i + 1)) < 1e-14
    c = rand((d,), 9)
    vc = np.broadcast_to(c, v.shape).copy()
    oc, _ = oa.varlen_forward(q, k, vc, cu, scale)
    assert close(oc, np.broadcast_to(c, oc.shape), 1e-14, 1e-13)


def test_segment_permutation_permutes_outputs():
    """Moving whole segments moves their outputs unchanged (bit-exact)."""
    lengths = [4, 7, 1, 5]
    perm = [2, 0, 3, 1]
    cu, _, _, _ = op.build_metadata(lengths)
    T, Hq, Hkv, d = int(cu[-1]), 4, 2, 8
    q, k, v, do = rand((T, Hq, d), 1), rand((T, Hkv, d), 2), rand((T, Hkv, d), 3), rand((T, Hq, d), 4)
    o, lse = oa.varlen_forward(q, k, v, cu, 0.5)
    g = oa.varlen_backward(q, k, v, o, lse, do, cu, 0.5)
    idx = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in perm])
    cu2, _, _, _ = op.build_metadata([lengths[b] for b in perm])
    o2, lse2 = oa.varlen_forward(q[idx], k[idx], v[idx], cu2, 0.5)
    g2 = oa.varlen_backward(q[idx], k[idx], v[idx], o2, lse2, do[idx], cu2, 0.5)
    assert np.array_equal(o[idx], o2) and np.array_equal(lse[:, idx], lse2)
    for a, b in zip(g, g2):
        assert np.array_equal(a[idx], b)


def test_perturbing_one_segment_leaves_others_bit_identical():
    """Course 'Optional practice': changing A leaves B's results unchanged, and with dO only on B,
    every other segment's gradients are exactly zero."""
    lengths = [6, 5, 3]
    cu, _, _, _ = op.build_metadata(lengths)
    T, Hq, Hkv, d = int(cu[-1]), 2, 2, 8
    q, k, v, do = rand((T, Hq, d), 1), rand((T, Hkv, d), 2), rand((T, Hkv, d), 3), rand((T, Hq, d), 4)
    o, lse = oa.varlen_forward(q, k, v, cu, 0.5)
    g = oa.varlen_backward(q, k, v, o, lse, do, cu, 0.5)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[:6] += 3.0
    k2[:6] -= 1.0
    v2[:6] *= 2.0
    o2, lse2 = oa.varlen_forward(q2, k2, v2, cu, 0.5)
    g2 = oa.varlen_backward(q2, k2, v2, o2, lse2, do, cu, 0.5)
    assert np.array_equal(o[6:], o2[6:]) and np.array_equal(lse[:, 6:], lse2[:, 6:])
    for a, b in zip(g, g2):
        assert np.array_equal(a[6:], b[6:])
    dob = np.zeros_like(do)
    dob[6:11] = do[6:11]
    gb = oa.varlen_backward(q, k, v, o, lse, dob, cu, 0.5)
    for a in gb:
        assert np.all(a[:6] == 0) and np.all(a[11:] == 0)
    # B's first query reads no future key: its dQ ignores every later k
    kf = k.copy()
    kf[7:] += 5.0
    of, lf = oa.varlen_forward(q, kf, v, cu, 0.5)
    assert np.array_equal(of[6], o[6])


def test_rows_sampler_matches_full_oracle():
    """The one-row-at-a-time checker agrees with the full oracle (O, LSE, dQ)."""
    cu, pos, seg, q, k, v, do = random_pack(3, T_max=50, Hq=4, Hkv=2, d=8)
    o, lse = oa.varlen_forward(q, k, v, cu, 0.3)
    dq, _, _ = oa.varlen_backward(q, k, v, o, lse, do, cu, 0.3)
    rng = np.random.default_rng(1)
    toks = rng.integers(0, q.shape[0], 20)
    heads = rng.integers(0, 4, 20)
    ro, rl, rdq = oa.rows_forward_backward(q, k, v, do, cu, toks, heads, 0.3)
    assert close(ro, o[toks, heads], 1e-13, 1e-11)
    assert close(rl, lse[heads, toks], 1e-13, 1e-11)
    assert close(rdq, dq[toks, heads], 1e-12, 1e-10)


def test_kv_head_subset_equals_full():
    cu, pos, seg, q, k, v, do = random_pack(4, T_max=30, Hq=4, Hkv=2, d=8)
    o, lse = oa.varlen_forward(q, k, v, cu, 0.3)
    g = oa.varlen_backward(q, k, v, o, lse, do, cu, 0.3)
    o1, l1 = oa.varlen_forward(q, k, v, cu, 0.3, kv_heads=[1])
    g1 = oa.varlen_backward(q, k, v, o1, l1, do, cu, 0.3, kv_heads=[1])
    assert np.array_equal(o1[:, 2:], o[:, 2:]) and np.all(np.isnan(o1[:, :2]))
    assert np.array_equal(g1[1][:, 1], g[1][:, 1]) and np.array_equal(g1[0][:, 2:], g[0][:, 2:])


def test_long_segment_row_blocking_is_exact():
    """Row blocks (used only to bound memory) do not change the result."""
    T, H, d = 300, 2, 8
    q, k, v, do = rand((T, H, d), 1), rand((T, H, d), 2), rand((T, H, d), 3), rand((T, H, d), 4)
    o, lse = oa.segment_forward(q, k, v, 0.3)
    old = oa._BLOCK_BYTES
    try:
        oa._BLOCK_BYTES = 8 * H * T * 7      # 7-row blocks
        ob, lb = oa.segment_forward(q, k, v, 0.3)
        gb = oa.segment_backward(q, k, v, ob, lb, do, 0.3)
    finally:
        oa._BLOCK_BYTES = old
    g = oa.segment_backward(q, k, v, o, lse, do, 0.3)
    assert close(o, ob, 1e-13, 1e-12) and close(lse, lb, 1e-13, 1e-12)
    for a, b in zip(g, gb):
        assert close(a, b, 1e-12, 1e-10)


def test_rejects_bad_boundaries():
    q = np.zeros((5, 1, 4))
    for cu in ([0, 3, 3, 5], [1, 5], [0, 4], [0, 6], [0, 3, 2, 5]):
        with pytest.raises(ValueError):
            oa.varlen_forward(q, q, q, cu)


@pytest.mark.parametrize("causal", [True, False])
def test_key_rows_sampler_matches_full_oracle(causal):
    """The one-key-at-a-time dK/dV checker agrees with the full oracle."""
    cu, pos, seg, q, k, v, do = random_pack(8, T_max=40, Hq=4, Hkv=2, d=8)
    o, lse = oa.varlen_forward(q, k, v, cu, 0.3, causal)
    _, dk, dv = oa.varlen_backward(q, k, v, o, lse, do, cu, 0.3, causal)
    toks = np.array([0, 3, 17, q.shape[0] - 1, 22])
    for hk in range(2):
        rk, rv = oa.key_rows_backward(q, k, v, do, cu, toks, hk, 0.3, causal)
        assert close(rk, dk[toks, hk], 1e-12, 1e-10)
        assert close(rv, dv[toks, hk], 1e-12, 1e-10)


@pytest.mark.parametrize("w", [0, 1, 3, 7])
def test_local_window_against_banded_sdpa(w):
    """Local window w: each segment equals torch's float64 SDPA under a band mask built from
    two triangles (tril(0) minus tril(-(w+1))), forward and autograd backward."""
    cu, pos, seg, q, k, v, do = random_pack(50 + w, T_max=60)
    scale = 0.29
    o, lse = oa.varlen_forward(q, k, v, cu, scale, window=w)
    dq, dk, dv = oa.varlen_backward(q, k, v, o, lse, do, cu, scale, window=w)
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        l = e - s
        ones = torch.ones(l, l, dtype=torch.bool)
        band = torch.tril(ones) & ~torch.tril(ones, diagonal=-(w + 1))
        tq, tk, tv = (torch.tensor(x[s:e].transpose(1, 0, 2), requires_grad=True) for x in (q, k, v))
        g = tq.shape[0] // tk.shape[0]
        to = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(g, 0), tv.repeat_interleave(g, 0), attn_mask=band, scale=scale)
        (to * torch.tensor(do[s:e].transpose(1, 0, 2))).sum().backward()
        assert close(o[s:e], to.detach().numpy().transpose(1, 0, 2), 1e-12, 1e-10)
        assert close(dq[s:e], tq.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
        assert close(dk[s:e], tk.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
        assert close(dv[s:e], tv.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)


def test_local_window_closed_forms():
    """w = 0: a query sees only itself (O = v, LSE = scale q.k); w >= the longest segment: no
    window; w = 1 by hand: query 2 of a segment mixes v_1 and v_2 with weights
    softmax(scale q_2.k_1, scale q_2.k_2)."""
    cu, pos, seg, q, k, v, do = random_pack(77, T_max=50, Hq=2, Hkv=2)
    scale = 0.5
    o0, l0 = oa.varlen_forward(q, k, v, cu, scale, window=0)
    assert close(o0, v, 1e-12, 1e-12)
    assert close(l0, scale * np.einsum("thc,thc->ht", q, k), 1e-12, 1e-12)
    big = int(np.diff(cu).max())
    ow, lw = oa.varlen_forward(q, k, v, cu, scale, window=big)
    on, ln = oa.varlen_forward(q, k, v, cu, scale)
    assert np.array_equal(ow, on) and np.array_equal(lw, ln)
    o1, _ = oa.varlen_forward(q, k, v, cu, scale, window=1)
    b = int(np.argmax(np.diff(cu) >= 3))
    t = int(cu[b]) + 2
    for h in range(2):
        a1, a2 = scale * q[t, h] @ k[t - 1, h], scale * q[t, h] @ k[t, h]
        w1, w2 = np.exp(a1) / (np.exp(a1) + np.exp(a2)), np.exp(a2) / (np.exp(a1) + np.exp(a2))
        assert close(o1[t, h], w1 * v[t - 1, h] + w2 * v[t, h], 1e-12, 1e-12)
    with pytest.raises(ValueError):
        oa.varlen_forward(q, k, v, cu, scale, causal=False, window=2)


@pytest.mark.parametrize("causal", [True, False])
def test_cross_attention_against_sdpa(causal):
    """cu_q != cu_k: each segment equals torch's float64 SDPA on its own Q slice and K/V slice,
    causal with the bottom-right mask built as a shifted triangle (tril with diagonal lk - lq),
    forward and autograd backward; lq = lk reduces to self-attention."""
    rng = np.random.default_rng(3)
    lq = [1, 5, 17, 3, 40]
    lk = [1, 9, 17, 30, 41]
    cuq, cuk = np.cumsum([0] + lq), np.cumsum([0] + lk)
    Tq, Tk, Hq, Hkv, d = cuq[-1], cuk[-1], 4, 2, 8
    q, do = rng.standard_normal((Tq, Hq, d)), rng.standard_normal((Tq, Hq, d))
    k, v = rng.standard_normal((Tk, Hkv, d)), rng.standard_normal((Tk, Hkv, d))
    scale = 0.41
    o, lse = oa.varlen_forward(q, k, v, cuq, scale, causal, cu_seqlens_k=cuk)
    dq, dk, dv = oa.varlen_backward(q, k, v, o, lse, do, cuq, scale, causal, cu_seqlens_k=cuk)
    for b in range(len(lq)):
        s, e, sk, ek = cuq[b], cuq[b + 1], cuk[b], cuk[b + 1]
        mask = torch.tril(torch.ones(lq[b], lk[b], dtype=torch.bool), diagonal=lk[b] - lq[b]) if causal else None
        tq = torch.tensor(q[s:e].transpose(1, 0, 2), requires_grad=True)
        tk, tv = (torch.tensor(x[sk:ek].transpose(1, 0, 2), requires_grad=True) for x in (k, v))
        to = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(2, 0), tv.repeat_interleave(2, 0), attn_mask=mask, scale=scale)
        (to * torch.tensor(do[s:e].transpose(1, 0, 2))).sum().backward()
        assert close(o[s:e], to.detach().numpy().transpose(1, 0, 2), 1e-12, 1e-10)
        assert close(dq[s:e], tq.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
        assert close(dk[sk:ek], tk.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
        assert close(dv[sk:ek], tv.grad.numpy().transpose(1, 0, 2), 1e-12, 1e-9)
    # a single query (lq = 1) under causality sees every key of its segment
    o1, _ = oa.varlen_forward(q[:1], k[:9], v[:9], [0, 1], scale, True, cu_seqlens_k=[0, 9])
    on, _ = oa.varlen_forward(q[:1], k[:9], v[:9], [0, 1], scale, False, cu_seqlens_k=[0, 9])
    assert np.array_equal(o1, on)
    with pytest.raises(ValueError):  # causal needs lq <= lk
        oa.varlen_forward(q[:5], k[:3], v[:3], [0, 5], scale, True, cu_seqlens_k=[0, 3])
