"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Bit-exact for integer work (cu_seqlens, position_ids, segment_ids, tile maps);
bf16 O within max-abs 2e-2, LSE within 1e-3 and dQ/dK/dV within relative-L2
1e-2 for floating point.  All inputs are seeded and identical on both sides.
"""
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


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    import packed_sequence_varlen_gb300 as pkg
    pkg._lib.load()
    return pkg


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def gpu_metadata(va, lengths, pad_to=0):
    lens = torch.tensor(lengths, dtype=torch.int32, device=DEV)
    T = max(sum(lengths), pad_to)
    cu, pos, seg, mx, st = va.build_metadata(lens, pad_to=pad_to, T_capacity=T)
    assert int(st.item()) == 0
    B = len(lengths) + (1 if pad_to > sum(lengths) else 0)
    return cu[:B + 1], pos, seg, int(mx.item())


def run_gpu(va, q, k, v, do, cu, max_seqlen, causal=True, scale=None):
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    out, lse = va.varlen_attn_fwd(qd, kd, vd, cu, max_seqlen, scale, causal, check_status=True)
    dq, dk, dv = va.varlen_attn_bwd(qd, kd, vd, out, lse, dod, cu, max_seqlen, scale, causal,
                                    check_status=True)
    torch.cuda.synchronize()
    return f64(out), lse.cpu().double().numpy(), (f64(dq), f64(dk), f64(dv))


def run_oracle(q, k, v, do, cu, causal=True, scale=None, kv_heads=None):
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    o, lse = oa.varlen_forward(qq, kk, vv, cu, scale, causal, kv_heads)
    g = oa.varlen_backward(qq, kk, vv, o, lse, dd, cu, scale, causal, kv_heads)
    return o, lse, g


# ------------------------------------------------------------------ integer work

@pytest.mark.parametrize("name", ["tiny", "sft8k", "gqa16k", "long64k", "tiny4k"])
def test_metadata_bit_exact(va, name):
    for real, pad_to in wl.real_packs(name)[:4]:
        cu, pos, seg, mx = gpu_metadata(va, real, pad_to)
        rcu, rpos, rseg, rmx = op.build_metadata(real, pad_to)
        assert np.array_equal(cu.cpu().numpy(), rcu)
        assert np.array_equal(pos.cpu().numpy(), rpos)
        assert np.array_equal(seg.cpu().numpy(), rseg)
        assert mx == rmx


# Streams of at most 16384 tokens cut into at most 2046 lengths get positions and segment ids
# from the scan's own block; longer ones from a separate fill launch.  Both sides of each limit.
@pytest.mark.parametrize("n,length,pad_to", [(2046, 8, 16384), (2047, 8, 16384), (2046, 8, 0),
                                             (100, 163, 16385), (100, 163, 16384), (1, 16384, 0),
                                             (0, 1, 16384), (0, 1, 16385)])
def test_metadata_fill_limits_bit_exact(va, n, length, pad_to):
    rng = np.random.default_rng(n + length + pad_to)
    lengths = [int(x) for x in rng.integers(1, 2 * length, n)] if length > 1 else [1] * n
    if pad_to and sum(lengths) > pad_to:
        lengths = [max(1, x // 2) for x in lengths]
    cu, pos, seg, mx = gpu_metadata(va, lengths, pad_to)
    rcu, rpos, rseg, rmx = op.build_metadata(lengths, pad_to)
    assert np.array_equal(cu.cpu().numpy(), rcu)
    assert np.array_equal(pos.cpu().numpy(), rpos)
    assert np.array_equal(seg.cpu().numpy(), rseg)
    assert mx == rmx


def test_metadata_page_layout_and_errors(va):
    cu, pos, seg, mx = gpu_metadata(va, [5, 3, 4])
    assert cu.cpu().tolist() == [0, 5, 8, 12]
    assert pos.cpu().tolist() == [0, 1, 2, 3, 4, 0, 1, 2, 0, 1, 2, 3] and mx == 5
    for lengths, pad in (([3, 0, 2], 0), ([4, 4], 6), ([2, -1], 0)):
        lens = torch.tensor(lengths, dtype=torch.int32, device=DEV)
        *_, st = va.build_metadata(lens, pad_to=pad, T_capacity=16)
        assert int(st.item()) == 5


# Causal calls whose mean segment length T / B is below TOKEN_MEAN put segments of at most
# TOKEN_SHORT tokens in token tiles (every map); the results do not depend on the choice.
TOKEN_SHORT = 64
TOKEN_MEAN = 256


def token_short(cu, causal):
    return TOKEN_SHORT if causal and int(cu[-1]) < TOKEN_MEAN * (len(cu) - 1) else 0


def oracle_map(va, kind, cu, Hq, Hkv, d, causal):
    BM, BN = va.tile_sizes(kind, d)
    if kind == 1:
        return ot.bwd_tile_map(cu, Hkv, BM, BN, causal, token_short(cu, causal))
    return ot.fwd_tile_map(cu, Hq, BM, BN, causal, token_short(cu, causal))


@pytest.mark.parametrize("name", ["tiny", "sft8k", "gqa16k", "long64k", "tiny4k"])
@pytest.mark.parametrize("causal", [True, False])
def test_tile_maps_bit_exact(va, name, causal):
    w = si.WORKLOADS[name]
    for lengths in wl.packs(name)[:3]:
        cu, _, _, mx = op.build_metadata(lengths)
        cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
        T = int(cu[-1])
        for kind in (0, 1, 2):
            tm, n = va.plan(cud, T, w.Hq, w.Hkv, w.d, mx, kind, causal)
            ref = oracle_map(va, kind, cu, w.Hq, w.Hkv, w.d, causal)
            assert n == len(ref)
            assert np.array_equal(tm.cpu().numpy(), ref)


def _align256(x):
    return (x + 255) // 256 * 256


def call_maps(va, cu, Hq, Hkv, d, mx, causal):
    """The maps the attention calls build for themselves (the forward's check + map launch,
    the backward preparation's planning CTAs), read back from the calls' workspaces.  Layout:
    a 256-byte header (int32 status, n_items[4], ...); a forward workspace then holds the
    map; a backward one D [Hq, T] fp32, then the kv-block and the q-block maps, each at a
    256-byte boundary and (rows / tile + B) * heads records long."""
    T, B = int(cu[-1]), len(cu) - 1
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    q = torch.zeros((T, Hq, d), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((T, Hkv, d), dtype=torch.bfloat16, device=DEV)
    ws_f = torch.empty(va.workspace_size(T, B, Hq, Hkv, d, mx, False), dtype=torch.uint8, device=DEV)
    ws_b = torch.empty(va.workspace_size(T, B, Hq, Hkv, d, mx, True), dtype=torch.uint8, device=DEV)
    o, lse = va.varlen_attn_fwd(q, k, k, cud, mx, causal=causal, workspace=ws_f, check_status=True)
    va.varlen_attn_bwd(q, k, k, o, lse, q, cud, mx, causal=causal, workspace=ws_b, check_status=True)
    torch.cuda.synchronize()

    def records(ws, n_slot, at):
        n = int(ws[4 * (1 + n_slot):4 * (2 + n_slot)].view(torch.int32).item())
        return ws[at:at + 16 * n].view(torch.int32).reshape(n, 4).cpu().numpy()

    _, BN_kv = va.tile_sizes(1, d)
    kvmap = _align256(256 + Hq * T * 4)
    qmap = _align256(kvmap + (T // BN_kv + B) * Hkv * 16)
    return {0: records(ws_f, 0, 256), 1: records(ws_b, 1, kvmap), 2: records(ws_b, 2, qmap)}


@pytest.mark.parametrize("name", ["tiny", "sft8k", "gqa16k", "long64k", "tiny4k"])
@pytest.mark.parametrize("causal", [True, False])
def test_call_maps_bit_exact(va, name, causal):
    """Packs of at most 32 segments take the planner's short path, the rest the general one;
    both must build the maps the oracle lists, record for record."""
    w = si.WORKLOADS[name]
    for lengths in wl.packs(name)[:2]:
        cu, _, _, mx = op.build_metadata(lengths)
        got = call_maps(va, cu, w.Hq, w.Hkv, w.d, mx, causal)
        for kind in (0, 1, 2):
            assert np.array_equal(got[kind], oracle_map(va, kind, cu, w.Hq, w.Hkv, w.d, causal)), kind


@pytest.mark.parametrize("B", [1, 2, 31, 32, 33, -20])
def test_call_maps_around_the_short_path_limit(va, B):
    """B < 0: -B segments of at most 64 tokens (token tiles, so the general path even for
    few segments)."""
    rng = np.random.default_rng(100 + abs(B))
    lengths = (rng.integers(1, 700, size=B) if B > 0 else rng.integers(1, 65, size=-B)).tolist()
    cu, _, _, mx = op.build_metadata(lengths)
    for causal in (True, False):
        got = call_maps(va, cu, 4, 2, 64, mx, causal)
        for kind in (0, 1, 2):
            assert np.array_equal(got[kind], oracle_map(va, kind, cu, 4, 2, 64, causal)), (kind, causal)


# ------------------------------------------------------------------ small cases

def test_tiny_page_layout_and_merge(va):
    """Blog section 1: [0,5,8,12] and the merged [0,5,12]; fp32 N(0,1) inputs rounded to bf16."""
    q, k, v, do = si.tensors(12, 2, 2, 64, dtype=torch.float32)
    q, k, v, do = (x.to(torch.bfloat16) for x in (q, k, v, do))
    res = {}
    for cu_list in ([0, 5, 8, 12], [0, 5, 12]):
        cu = torch.tensor(cu_list, dtype=torch.int32, device=DEV)
        o, lse, g = run_gpu(va, q, k, v, do, cu, max(np.diff(cu_list)))
        ro, rl, rg = run_oracle(q, k, v, do, cu_list)
        wl.assert_close_outputs(o, lse, ro, rl)
        wl.assert_close_grads(g, rg)
        res[len(cu_list)] = (o, lse) + g
    a, m = res[4], res[3]
    for x, y in zip(a, m):
        sl = (slice(None), slice(0, 5)) if x.ndim == 2 else (slice(0, 5),)
        assert np.array_equal(x[sl], y[sl])          # A's rows bit-identical
    assert np.array_equal(a[0][5:8], m[0][5:8])      # B's O: same tiles, same keys
    assert not np.array_equal(a[0][8:], m[0][8:])    # C changes


EDGE = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 1, 383, 384, 385]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("g", [1, 2])
def test_ragged_edge_lengths(va, d, causal, g):
    lengths = EDGE
    cu, _, _, mx = op.build_metadata(lengths)
    T = int(cu[-1])
    Hkv = 2
    q, k, v, do = si.tensors(T, Hkv * g, Hkv, d, seed_offset=10 * d + g)
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    o, lse, gr = run_gpu(va, q, k, v, do, cud, mx, causal)
    ro, rl, rg = run_oracle(q, k, v, do, cu, causal)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(gr, rg)
    if causal:  # a segment's first query sees only itself: O is exactly its V row
        for s in cu[:-1]:
            for h in range(Hkv * g):
                assert np.array_equal(o[s, h], si.to_f64(v[s, h // g]))


# ------------------------------------------------------------------ workloads

def check_rows_every_head(q, k, v, do, cu, o, lse, grads, seed, rows_per_head=16, keys_per_head=4):
    """Sampled rows of every q head (O, LSE, dQ) and key rows of every kv head (dK, dV), each
    computed by the oracle from its own row, so that an indexing error confined to heads the
    full-slice checks leave out is still caught.  Rows include segment starts and ends; key rows
    sit near segment ends (cheap in the oracle)."""
    dq, dk, dv = grads
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    T, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    rng = np.random.default_rng(seed)
    starts, ends = np.asarray(cu[:-1]), np.asarray(cu[1:]) - 1
    toks, heads = [], []
    for h in range(Hq):
        pick = rng.integers(0, T, rows_per_head - 2).tolist()
        pick += [int(rng.choice(starts)), int(rng.choice(ends))]
        toks += pick
        heads += [h] * len(pick)
    toks, heads = np.asarray(toks), np.asarray(heads)
    so, sl, sdq = oa.rows_forward_backward(qq, kk, vv, dd, cu, toks, heads)
    assert np.abs(o[toks, heads] - so).max() <= wl.O_MAX_ABS
    assert np.abs(lse[heads, toks] - sl).max() <= wl.LSE_MAX_ABS
    assert wl.rel_l2(dq[toks, heads], sdq) <= wl.GRAD_REL_L2
    lens = np.diff(cu)
    for hk in range(Hkv):
        segs = rng.choice(len(lens), keys_per_head, replace=False)
        ktoks = np.array([int(cu[b + 1]) - 1 - int(rng.integers(0, min(48, lens[b]))) for b in segs])
        rk, rv = oa.key_rows_backward(qq, kk, vv, dd, cu, ktoks, hk)
        assert wl.rel_l2(dk[ktoks, hk], rk) <= wl.GRAD_REL_L2
        assert wl.rel_l2(dv[ktoks, hk], rv) <= wl.GRAD_REL_L2


@pytest.mark.parametrize("index,kv_heads", [(0, [0, 17]), (1, [31]), (5, [8])])
def test_sft8k_packs(va, index, kv_heads):
    """Full-slice checks on a few kv heads, plus sampled rows of every head."""
    w = si.WORKLOADS["sft8k"]
    lengths = wl.pack("sft8k", index)
    cu, _, _, mx = op.build_metadata(lengths)
    q, k, v, do = si.tensors(int(cu[-1]), w.Hq, w.Hkv, w.d, seed_offset=100 * index)
    o, lse, g = run_gpu(va, q, k, v, do, torch.tensor(cu, device=DEV), mx)
    ro, rl, rg = run_oracle(q, k, v, do, cu, kv_heads=kv_heads)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(g, rg)
    check_rows_every_head(q, k, v, do, cu, o, lse, g, seed=index)


@pytest.mark.parametrize("which", ["first", "most_segments"])
def test_gqa16k_bins(va, which):
    """Full-slice checks on one kv head (its four q heads), plus sampled rows of every head."""
    w = si.WORKLOADS["gqa16k"]
    index = 0 if which == "first" else wl.most_segments_pack("gqa16k")
    lengths = wl.pack("gqa16k", index)
    cu, _, _, mx = op.build_metadata(lengths)
    q, k, v, do = si.tensors(int(cu[-1]), w.Hq, w.Hkv, w.d, seed_offset=index)
    o, lse, g = run_gpu(va, q, k, v, do, torch.tensor(cu, device=DEV), mx)
    ro, rl, rg = run_oracle(q, k, v, do, cu, kv_heads=[index % w.Hkv])
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(g, rg)
    check_rows_every_head(q, k, v, do, cu, o, lse, g, seed=100 + index)


def test_long64k(va):
    """Whole pack on the GPU; the oracle checks the six shorter segments in full for one kv
    head, sampled rows (O, LSE, dQ) of the 32768 and 16384 segments for every head, and the
    last key rows (dK, dV) of those two segments."""
    w = si.WORKLOADS["long64k"]
    lengths = wl.pack("long64k")
    cu, _, _, mx = op.build_metadata(lengths)
    T = int(cu[-1])
    q, k, v, do = si.tensors(T, w.Hq, w.Hkv, w.d)
    o, lse, (dq, dk, dv) = run_gpu(va, q, k, v, do, torch.tensor(cu, device=DEV), mx)
    qq, kk, vv, dd = (si.to_f64(x) for x in (q, k, v, do))
    s0 = int(cu[2])
    sub = [c - s0 for c in cu[2:]]
    hk = 5
    ro, rl = oa.varlen_forward(qq[s0:], kk[s0:], vv[s0:], sub, kv_heads=[hk])
    rg = oa.varlen_backward(qq[s0:], kk[s0:], vv[s0:], ro, rl, dd[s0:], sub, kv_heads=[hk])
    wl.assert_close_outputs(o[s0:], lse[:, s0:], ro, rl)
    wl.assert_close_grads((dq[s0:], dk[s0:], dv[s0:]), rg)
    rng = np.random.default_rng(0)
    toks = np.concatenate([rng.integers(0, int(cu[2]), 48), [0, 1, 32767, 32768, 49151]])
    heads = rng.integers(0, w.Hq, toks.size)
    so, sl, sdq = oa.rows_forward_backward(qq, kk, vv, dd, cu, toks, heads)
    assert np.abs(o[toks, heads] - so).max() <= wl.O_MAX_ABS
    assert np.abs(lse[heads, toks] - sl).max() <= wl.LSE_MAX_ABS
    assert wl.rel_l2(dq[toks, heads], sdq) <= wl.GRAD_REL_L2
    ktoks = np.array([32767 - 40, 32767 - 3, 32767, 49151 - 17, 49151])
    rk, rv = oa.key_rows_backward(qq, kk, vv, dd, cu, ktoks, 2)
    assert wl.rel_l2(dk[ktoks, 2], rk) <= wl.GRAD_REL_L2
    assert wl.rel_l2(dv[ktoks, 2], rv) <= wl.GRAD_REL_L2


def test_tiny4k_full(va):
    w = si.WORKLOADS["tiny4k"]
    lengths = wl.pack("tiny4k")
    assert 3800 < len(lengths) < 4300
    cu, _, _, mx = op.build_metadata(lengths)
    q, k, v, do = si.tensors(int(cu[-1]), w.Hq, w.Hkv, w.d)
    o, lse, g = run_gpu(va, q, k, v, do, torch.tensor(cu, device=DEV), mx)
    ro, rl, rg = run_oracle(q, k, v, do, cu)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(g, rg)
    wl.assert_close_grads_chunked(g, rg)


# Runs of short segments: one of 300 single-token segments (more than 32 segment starts in
# one token tile), runs cut at 128 and 256 rows inside a segment, a short segment alone
# between long ones, 64 (the longest token-tiled length) next to 65, and a run that ends the
# stream.
TOKEN_RUNS = [1] * 300 + [200] + [64] * 5 + [65, 3, 64, 1, 17, 700] + [33] * 20 + [2]


@pytest.mark.parametrize("d,g", [(64, 1), (128, 2)])
def test_token_tiles_mixed_runs(va, d, g):
    cu, _, _, mx = op.build_metadata(TOKEN_RUNS)
    T = int(cu[-1])
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    for kind in (0, 1, 2):  # forward, dK/dV and dQ maps: token records after segment ones
        tm, n = va.plan(cud, T, 2 * g, 2, d, mx, kind, True)
        ref = oracle_map(va, kind, cu, 2 * g, 2, d, True)
        assert (ref[:, 0] < 0).sum() > 0 and n == len(ref)
        assert np.array_equal(tm.cpu().numpy(), ref)
    q, k, v, do = si.tensors(T, 2 * g, 2, d, seed_offset=7 * d + g)
    o, lse, gr = run_gpu(va, q, k, v, do, cud, mx)
    ro, rl, rg = run_oracle(q, k, v, do, cu)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(gr, rg)
    # the rows of token-tiled segments alone (whole-tensor norms could hide them)
    short = np.repeat(np.diff(cu) <= TOKEN_SHORT, np.diff(cu))
    wl.assert_close_grads(tuple(x[short] for x in gr), tuple(x[short] for x in rg))
    wl.assert_close_grads_chunked(tuple(x[short] for x in gr), tuple(x[short] for x in rg))
    for s in cu[:-1]:  # a segment's first query sees only itself
        for h in range(2 * g):
            assert np.array_equal(o[s, h], si.to_f64(v[s, h // g]))


def test_short_segments_among_long_ones(va):
    """Mean segment length above the token-tile threshold: the short segments (1, 3, 64 tokens)
    are covered by segment records, every map and gradient as the oracle gives them."""
    lengths = [2000, 3, 1500, 64, 1, 1000]
    cu, _, _, mx = op.build_metadata(lengths)
    assert token_short(cu, True) == 0
    T = int(cu[-1])
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    for kind in (0, 1, 2):
        tm, n = va.plan(cud, T, 4, 2, 128, mx, kind, True)
        ref = oracle_map(va, kind, cu, 4, 2, 128, True)
        assert (ref[:, 0] >= 0).all() and n == len(ref)
        assert np.array_equal(tm.cpu().numpy(), ref)
    q, k, v, do = si.tensors(T, 4, 2, 128, seed_offset=77)
    o, lse, gr = run_gpu(va, q, k, v, do, cud, mx)
    ro, rl, rg = run_oracle(q, k, v, do, cu)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(gr, rg)
    short = np.repeat(np.diff(cu) <= TOKEN_SHORT, np.diff(cu))
    wl.assert_close_grads(tuple(x[short] for x in gr), tuple(x[short] for x in rg))


def test_more_segments_than_shared_offsets(va):
    """4400 segments: more than the planner keeps in shared memory (4095 boundaries), so the
    per-segment record offsets go to the workspace and one planning block builds both backward
    maps in turn.  Every tenth segment is 65..200 tokens (segment records), the rest 1..40
    (token tiles under causality); maps bit-exact, causal results as the oracle gives them."""
    rng = np.random.default_rng(11)
    lengths = [int(x) for x in rng.integers(1, 41, 4400)]
    for i in range(0, 4400, 10):
        lengths[i] = int(rng.integers(65, 201))
    cu, _, _, mx = op.build_metadata(lengths)
    T = int(cu[-1])
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    for causal in (True, False):
        for kind in (0, 1, 2):
            tm, n = va.plan(cud, T, 2, 1, 64, mx, kind, causal)
            ref = oracle_map(va, kind, cu, 2, 1, 64, causal)
            assert n == len(ref)
            assert np.array_equal(tm.cpu().numpy(), ref)
    q, k, v, do = si.tensors(T, 2, 1, 64, seed_offset=41)
    o, lse, gr = run_gpu(va, q, k, v, do, cud, mx)
    ro, rl, rg = run_oracle(q, k, v, do, cu)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(gr, rg)
    wl.assert_close_grads_chunked(gr, rg)


# ------------------------------------------------------------------ properties

def test_first_query_sees_only_itself(va):
    """Closed form: the first query of a segment has P = 1, so O is exactly its V row."""
    lengths = [37, 200, 1, 129, 64]
    cu, _, _, mx = op.build_metadata(lengths)
    q, k, v, do = si.tensors(int(cu[-1]), 4, 2, 128, seed_offset=3)
    o, lse, _ = run_gpu(va, q, k, v, do, torch.tensor(cu, device=DEV), mx)
    qq, kk = si.to_f64(q), si.to_f64(k)
    for s in cu[:-1]:
        for h in range(4):
            assert np.array_equal(o[s, h], si.to_f64(v[s, h // 2]))
            assert abs(lse[h, s] - qq[s, h] @ kk[s, h // 2] / np.sqrt(128)) < 1e-4


def test_segment_isolation_and_determinism(va):
    """Changing one segment's inputs leaves every other segment's results bit-identical;
    with dO only on one segment the others' gradients are exactly zero; runs repeat bit-exactly."""
    lengths = [300, 77, 129, 1000, 5]
    cu, _, _, mx = op.build_metadata(lengths)
    T = int(cu[-1])
    q, k, v, do = si.tensors(T, 4, 4, 64, seed_offset=9)
    cud = torch.tensor(cu, device=DEV)
    base = run_gpu(va, q, k, v, do, cud, mx)
    again = run_gpu(va, q, k, v, do, cud, mx)
    for a, b in zip(base[:2] + base[2], again[:2] + again[2]):
        assert np.array_equal(a, b)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    s, e = int(cu[1]), int(cu[2])
    q2[s:e] *= 2
    k2[s:e] += 1
    v2[s:e] -= 1
    pert = run_gpu(va, q2, k2, v2, do, cud, mx)
    keep = np.r_[0:s, e:T]
    for a, b in zip(base[:1] + base[2], pert[:1] + pert[2]):
        assert np.array_equal(a[keep], b[keep])
    assert np.array_equal(base[1][:, keep], pert[1][:, keep])
    do_b = torch.zeros_like(do)
    do_b[s:e] = do[s:e]
    _, _, gb = run_gpu(va, q, k, v, do_b, cud, mx)
    for a in gb:
        assert np.all(a[keep] == 0)


def test_strided_views_from_fused_projection(va):
    """q, k, v as views of one [T, 3, H, d] buffer (row stride 3*H*d), as a fused projection gives."""
    lengths = [100, 260, 31]
    cu, _, _, mx = op.build_metadata(lengths)
    T, H, d = int(cu[-1]), 4, 128
    g = torch.Generator().manual_seed(5)
    qkv = torch.randn((T, 3, H, d), generator=g).to(torch.bfloat16)
    do = torch.randn((T, H, d), generator=g).to(torch.bfloat16)
    qkv_d = qkv.to(DEV)
    q, k, v = qkv_d[:, 0], qkv_d[:, 1], qkv_d[:, 2]
    cud = torch.tensor(cu, device=DEV)
    out, lse = va.varlen_attn_fwd(q, k, v, cud, mx, check_status=True)
    dq, dk, dv = va.varlen_attn_bwd(q, k, v, out, lse, do.to(DEV), cud, mx, check_status=True)
    ro, rl, rg = run_oracle(qkv[:, 0], qkv[:, 1], qkv[:, 2], do, cu)
    wl.assert_close_outputs(f64(out), lse.cpu().double().numpy(), ro, rl)
    wl.assert_close_grads((f64(dq), f64(dk), f64(dv)), rg)


def test_autograd_function(va):
    lengths = [70, 190]
    cu, _, _, mx = op.build_metadata(lengths)
    q, k, v, do = si.tensors(int(cu[-1]), 4, 2, 64, seed_offset=4)
    qd, kd, vd = (x.to(DEV).requires_grad_() for x in (q, k, v))
    out = va.varlen_attn(qd, kd, vd, torch.tensor(cu, device=DEV), mx)
    out.backward(do.to(DEV))
    ro, rl, rg = run_oracle(q, k, v, do, cu)
    wl.assert_close_grads((f64(qd.grad), f64(kd.grad), f64(vd.grad)), rg)


def test_device_detected_bad_boundaries(va):
    """A cu_seqlens that breaks the contract (or a too-small max_seqlen) is reported in the
    status word and no output is written."""
    T, H, d = 64, 2, 64
    q, k, v, do = (x.to(DEV) for x in si.tensors(T, H, H, d))
    for cu_list, mx in (([0, 30, 20, 64], 40), ([0, 10, 64], 20), ([0, 32, 60], 32), ([1, 32, 64], 32)):
        cu = torch.tensor(cu_list, dtype=torch.int32, device=DEV)
        out = torch.full_like(q, 7.0)
        with pytest.raises(va.VarlenError) as e:
            va.varlen_attn_fwd(q, k, v, cu, mx, out=out, check_status=True)
        assert e.value.status == 5
        torch.cuda.synchronize()
        assert bool((out == 7.0).all())
        dq = torch.full_like(q, 3.0)
        with pytest.raises(va.VarlenError):
            va.varlen_attn_bwd(q, k, v, q, torch.zeros(H, T, device=DEV), do, cu, mx, dq=dq,
                               check_status=True)
        assert bool((dq == 3.0).all())


@pytest.mark.parametrize("d", [64, 128])
def test_running_max_rescale_path(va, d):
    """Keys whose magnitude grows along each segment make the row max jump by far more than
    2^8 between key tiles, which forces the forward to rescale O in TMEM; neighbouring
    segments sit in the same tiles, so a wrong rescale would also break isolation."""
    lengths = [700, 90, 1100, 33]
    cu, _, _, mx = op.build_metadata(lengths)
    T, H = int(cu[-1]), 4
    q, k, v, do = si.tensors(T, H, H, d, seed_offset=77)
    ramp = torch.ones(T)
    for b in range(len(lengths)):
        s, e = int(cu[b]), int(cu[b + 1])
        ramp[s:e] = 1.0 + torch.arange(e - s, dtype=torch.float32) / 48.0
    k = (k.float() * ramp[:, None, None]).to(torch.bfloat16)
    o, lse, g = run_gpu(va, q, k, v, do, torch.tensor(cu, device=DEV), mx)
    ro, rl, rg = run_oracle(q, k, v, do, cu)
    wl.assert_close_outputs(o, lse, ro, rl)
    wl.assert_close_grads(g, rg)
