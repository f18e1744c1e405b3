"""Pins for the planner, boundary metadata, tile maps and loss probe oracles (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import loss as ol
from oracle import packing as op
from oracle import tiles as ot

try:  # only the planner property test uses hypothesis; without it, seeded random cases
    from hypothesis import given, settings, strategies as st
except ImportError:
    given = None


def test_three_sample_metadata(golden_dir):
    fx = json.load(open(os.path.join(golden_dir, "three_samples_layout.json")))
    cu, pos, seg, mx = op.build_metadata(fx["lengths"])
    assert cu.tolist() == fx["cu_seqlens"]
    assert pos.tolist() == fx["position_ids"]
    assert seg.tolist() == [0] * 5 + [1] * 3 + [2] * 4
    assert mx == fx["max_seqlen"]
    # boundary compilation (blog section 3) inverts the positions, both readings
    for at_min in (False, True):
        cu2, mx2 = op.cu_seqlens_from_position_ids(pos, reset_at_min=at_min)
        assert cu2.tolist() == fx["cu_seqlens"] and mx2 == fx["max_seqlen"]
    # positions that start at 1 need the minimum-based reading
    cu3, _ = op.cu_seqlens_from_position_ids(pos + 1, reset_at_min=True)
    assert cu3.tolist() == fx["cu_seqlens"]


def test_boundary_plane_check():
    """Blog section 3: the compiled array must start at 0; the strict reading rejects a
    plane whose positions repeat inside a sample (mRoPE's visual coordinates)."""
    page = [0, 1, 2, 3, 4, 0, 1, 2, 0, 1, 2, 3]
    assert op.boundary_plane_ok(page) and op.boundary_plane_ok(page, strict=True)
    assert op.boundary_plane_ok(page, reset_at_min=True, strict=True)
    shifted = [p + 1 for p in page]
    assert not op.boundary_plane_ok(shifted)                     # no position 0 at index 0
    assert op.boundary_plane_ok(shifted, reset_at_min=True, strict=True)
    assert not op.boundary_plane_ok([1, 0, 1, 2])                # first token not a reset
    repeated = [0, 0, 0, 1, 1, 1, 2, 2, 0, 1]                    # a plane with repeated values
    assert op.boundary_plane_ok(repeated) and not op.boundary_plane_ok(repeated, strict=True)
    assert not op.boundary_plane_ok([0, 1, 3], strict=True)      # a gap inside a sample
    assert not op.boundary_plane_ok([])
    # one-token samples are valid in the strict reading
    assert op.boundary_plane_ok([0, 0, 0], strict=True)
    cu, mx = op.cu_seqlens_from_position_ids([0, 0, 0])
    assert cu.tolist() == [0, 1, 2, 3] and mx == 1


def test_tail_pad_segment():
    cu, pos, seg, mx = op.build_metadata([3, 2], pad_to=8)
    assert cu.tolist() == [0, 3, 5, 8]
    assert pos.tolist() == [0, 1, 2, 0, 1, 0, 1, 2]
    assert seg.tolist() == [0, 0, 0, 1, 1, 2, 2, 2] and mx == 3
    cu, _, _, _ = op.build_metadata([3, 5], pad_to=8)      # exact fill: no pad segment
    assert cu.tolist() == [0, 3, 8]
    with pytest.raises(ValueError):
        op.build_metadata([5, 5], pad_to=8)


def test_nine_target_rows(golden_dir):
    """Course 'Fill only the current row': next-fit at capacity 6 gives rows 3+2 and 4."""
    fx = json.load(open(os.path.join(golden_dir, "nine_target_fixture.json")))
    lengths = [len(x) for x in fx["pair_inputs"]]
    assert lengths == [3, 2, 4]
    assert op.next_fit(lengths, fx["capacity"]) == [[0, 1], [2]]
    rows = op.packed_storage_rows(fx["pair_inputs"], fx["pair_targets"], fx["capacity"])
    assert rows["inputs"] == fx["rows_inputs"]
    assert rows["targets"] == fx["rows_targets"]
    assert rows["segments"] == fx["rows_segments"]
    assert rows["positions"] == fx["rows_positions"]
    assert rows["input_valid"] == fx["rows_valid"]
    assert sum(map(len, rows["inputs"])) == fx["stored_cells"]
    assert sum(map(sum, rows["target_valid"])) == fx["real_targets"]
    # each real row is one segment list of the metadata oracle; pad cells sit outside
    for r, pack in enumerate(op.next_fit(lengths, fx["capacity"])):
        cu, pos, seg, _ = op.build_metadata([lengths[i] for i in pack])
        n = int(cu[-1])
        assert pos.tolist() == fx["rows_positions"][r][:n]


def test_nine_target_permissions(golden_dir):
    """B's first query (column 3) may use only column 3; its second uses columns 3 and 4."""
    fx = json.load(open(os.path.join(golden_dir, "nine_target_fixture.json")))
    seg, pos, val = fx["rows_segments"][0], fx["rows_positions"][0], fx["rows_valid"][0]

    def allowed(i, j):
        return val[i] and val[j] and seg[i] == seg[j] and pos[j] <= pos[i]
    c = fx["b_first_query_column"]
    assert [j for j in range(6) if allowed(c, j)] == fx["b_first_query_allowed_keys"]
    assert [j for j in range(6) if allowed(c + 1, j)] == fx["b_second_query_allowed_keys"]


def test_stream_targets_pairs_inside_documents(golden_dir):
    """The three fixture documents as one packed stream: the targets are exactly the page's
    nine (input, target) pairs, no pair crosses a document boundary, and they equal the
    ms-swift layout (labels = ids with -100 at each sample's first label, shifted by one)."""
    fx = json.load(open(os.path.join(golden_dir, "nine_target_fixture.json")))
    docs = [i + t[-1:] for i, t in zip(fx["pair_inputs"], fx["pair_targets"])]
    assert [len(d) for d in docs] == [4, 3, 5]
    ids = sum(docs, [])
    cu = np.cumsum([0] + [len(d) for d in docs])
    tg = ol.stream_targets(ids, cu)
    pairs = [(ids[t], int(tg[t])) for t in range(len(ids)) if tg[t] != ol.IGNORE_INDEX]
    want = [(a, b) for i, t in zip(fx["pair_inputs"], fx["pair_targets"]) for a, b in zip(i, t)]
    assert pairs == want and len(pairs) == fx["real_targets"]
    assert [t for t in range(len(ids)) if tg[t] == ol.IGNORE_INDEX] == [3, 6, 11]  # each last token
    labels = np.array(ids)
    labels[cu[:-1]] = ol.IGNORE_INDEX                                          # sample-local -100
    shifted = np.append(labels[1:], ol.IGNORE_INDEX)
    assert np.array_equal(tg, shifted)
    # a global shift of the concatenation would add the EOS -> BOS pairs at each join
    assert {(1, 0)} & set(zip(ids[:-1], ids[1:])) and (1, 0) not in pairs


def test_nine_target_loss_probe(golden_dir):
    """Token-weighted loss = 11 ln2 / 9 = 0.847180 (sum 7.624619); the row-mean and the
    document-mean weightings give 0.831777 and 0.924196 and must not be what we compute."""
    fx = json.load(open(os.path.join(golden_dir, "nine_target_fixture.json")))
    V = fx["vocab"]
    tg = np.asarray(fx["rows_targets"]).reshape(-1)
    seg = np.asarray(fx["rows_segments"]).reshape(-1)
    elig = np.asarray(fx["rows_valid"]).reshape(-1)
    qmap = {int(k): v for k, v in fx["gold_probability_by_segment"].items()}
    qcell = [qmap.get(int(s), 0.5) for s in seg]
    z = ol.constructed_logits(tg, elig, qcell, V)
    s, mean, grad = ol.token_weighted_loss(z, tg, elig)
    p = 10 ** -fx["printed_decimals"]
    assert abs(s - fx["loss_sum_printed"]) < p and abs(s - 11 * math.log(2)) < 1e-12
    assert abs(mean - fx["loss_mean_printed"]) < p
    assert abs(mean - 11 * math.log(2) / 9) < 1e-12
    assert abs(mean - fx["row_mean_printed"]) > 1e-3
    assert abs(mean - fx["document_mean_printed"]) > 1e-3
    # the two wrong weightings reproduce the page's other printed numbers
    nll = -np.log(np.asarray(qcell))[elig]
    rows = np.asarray(fx["rows_valid"])
    row_means = [nll[:rows[0].sum()].mean(), nll[rows[0].sum():].mean()]
    assert abs(np.mean(row_means) - fx["row_mean_printed"]) < p
    segs = seg[elig]
    doc_means = [nll[segs == d].mean() for d in (0, 1, 2)]
    assert abs(np.mean(doc_means) - fx["document_mean_printed"]) < p
    # gradient against torch autograd of the same objective
    import torch
    tz = torch.tensor(z, requires_grad=True)
    idx = torch.tensor(np.nonzero(elig)[0])
    lm = torch.nn.functional.cross_entropy(tz[idx], torch.tensor(tg)[idx], reduction="mean")
    lm.backward()
    assert np.allclose(grad, tz.grad.numpy(), atol=1e-15, rtol=1e-12)
    assert np.all(grad[~elig] == 0)
    with pytest.raises(ValueError):
        ol.token_weighted_loss(z, tg, np.zeros_like(elig))


def test_next_fit_rules():
    assert op.next_fit([3, 3, 6, 1], 6) == [[0, 1], [2], [3]]   # exact fill opens no extra row
    assert op.next_fit([], 6) == []
    with pytest.raises(ValueError):
        op.next_fit([7], 6)                                      # never split
    with pytest.raises(ValueError):
        op.next_fit([0], 6)


def test_best_fit_decreasing_small():
    # sorted: 5(i1) 4(i0) 3(i3) 2(i2) 2(i4) 1(i5)
    assert op.best_fit_decreasing([4, 5, 2, 3, 2, 1], 6) == [[1, 5], [0, 2], [3, 4]]
    assert op.best_fit_decreasing([2, 2, 2], 6) == [[0, 1, 2]]
    # two bins with equal room: the earlier one wins
    assert op.best_fit_decreasing([3, 3, 1], 4) == [[0, 2], [1]]


def _bfd_brute(lengths, cap):
    """Independent restatement: one pass per item over explicit bin contents."""
    order = sorted(range(len(lengths)), key=lambda i: (-lengths[i], i))
    bins = []
    for i in order:
        cands = [(cap - sum(lengths[j] for j in b), n) for n, b in enumerate(bins)]
        cands = [c for c in cands if c[0] >= lengths[i]]
        if cands:
            bins[min(cands)[1]].append(i)
        else:
            bins.append([i])
    return bins


def _planner_properties(lengths, cap):
    for packs in (op.next_fit(lengths, cap), op.best_fit_decreasing(lengths, cap)):
        flat = sorted(i for p in packs for i in p)
        assert flat == list(range(len(lengths)))                 # multiset preserved
        assert all(sum(lengths[i] for i in p) <= cap for p in packs)
        assert all(p for p in packs)
    nf = op.next_fit(lengths, cap)
    assert [i for p in nf for i in p] == list(range(len(lengths)))   # order kept
    for a, b in zip(nf, nf[1:]):                                 # b's first did not fit a
        assert sum(lengths[i] for i in a) + lengths[b[0]] > cap
    assert op.best_fit_decreasing(lengths, cap) == _bfd_brute(lengths, cap)


if given is not None:
    @settings(max_examples=150, deadline=None)
    @given(st.lists(st.integers(1, 50), max_size=60), st.integers(50, 120))
    def test_planner_properties(lengths, cap):
        _planner_properties(lengths, cap)
else:
    def test_planner_properties():
        rng = np.random.default_rng(2024)
        for _ in range(150):
            n = int(rng.integers(0, 61))
            _planner_properties([int(x) for x in rng.integers(1, 51, n)], int(rng.integers(50, 121)))


# ----------------------------------------------------------------- tile maps

def _allowed_edges(cu):
    e = set()
    for b in range(len(cu) - 1):
        for i in range(cu[b], cu[b + 1]):
            for j in range(cu[b], i + 1):
                e.add((i, j))
    return e


@pytest.mark.parametrize("BM,BN", [(2, 2), (4, 2), (2, 4), (128, 128), (256, 128)])
@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("short_div", [0, 2, 1])
def test_fwd_tile_map_covers_each_allowed_edge_once(BM, BN, seed, short_div):
    """Course 'History': tile traversal visits the same permitted edges as query order.

    short_div > 0 turns on token tiles for segments of at most BN / short_div tokens."""
    rng = np.random.default_rng(seed)
    short = BN // short_div if short_div else 0
    lengths = rng.integers(1, 3 * max(BM, BN) // 2 + 2, size=5).tolist()
    if short:  # a run of short segments in the middle and one at the end
        lengths = lengths[:2] + rng.integers(1, short + 1, size=7).tolist() + lengths[2:] + [short, 1]
    cu, _, _, _ = op.build_metadata(lengths)
    H = 2
    tm = ot.fwd_tile_map(cu, H, BM, BN, True, short)
    allowed = _allowed_edges(cu.tolist())
    for h in range(H):
        seen = []
        for it in tm[tm[:, 2] == h]:
            cover = ot.fwd_item_edges(cu, it, BM, BN)
            hit = [e for e in cover if e in allowed]
            assert hit, "a listed tile has no permitted edge"
            seen.extend(hit)
            b, m, _, nb = (int(x) for x in it)
            if b < 0:      # token tile: rows [t0, t0 + rows) of short segments
                t0, rows = m, nb
                assert 1 <= rows <= BM
                assert all(cu[x + 1] - cu[x] <= short for x in range(len(cu) - 1)
                           if cu[x] < t0 + rows and cu[x + 1] > t0)
                assert cu[-1 - b] <= t0 < cu[-b]          # f holds row t0
                continue
            s, l = cu[b], cu[b + 1] - cu[b]
            assert l > short
            last_row = s + min(l, (m + 1) * BM) - 1
            assert (last_row, s + (nb - 1) * BN) in allowed      # last kv tile is needed
        assert sorted(seen) == sorted(allowed)                  # each edge exactly once
    seg = tm[tm[:, 0] >= 0]
    tok = tm[tm[:, 0] < 0]
    assert np.array_equal(tm, np.concatenate([seg, tok]))     # token records come last
    # order: segments by cost class (floor log2 of their total key tiles), then head,
    # then most key tiles first
    cost = {}
    for b, m, h, nb in seg:
        if h == 0:
            cost[int(b)] = cost.get(int(b), 0) + int(nb)
    keys = [(-(cost[int(r[0])].bit_length() - 1), r[0], r[2], -r[3], r[1]) for r in seg]
    assert keys == sorted(keys)
    # records of one (segment, head) are contiguous
    groups = [(r[0], r[2]) for r in seg]
    assert len(set(groups)) == len([g for i, g in enumerate(groups) if i == 0 or g != groups[i - 1]])
    # token records by (first row, head), every head of a tile
    tkeys = [(r[1], r[2]) for r in tok]
    assert tkeys == sorted(tkeys) and len(tok) % H == 0


def test_token_tile_map_hand_example():
    """Lengths 3, 2, 1, 300, 4, 60 with BM=256, BN=128, short=64, one head, worked by hand.

    Segments 0-2 form the run [0, 6) (one tile of 6 rows, first segment 0); segment 3
    (300 tokens) keeps its q blocks m=1 (3 key blocks) and m=0 (2 key blocks); segments
    4-5 form the run [306, 370) (one tile of 64 rows starting in segment 4)."""
    cu, _, _, _ = op.build_metadata([3, 2, 1, 300, 4, 60])
    tm = ot.fwd_tile_map(cu, 1, 256, 128, True, 64)
    assert tm.tolist() == [[3, 1, 0, 3], [3, 0, 0, 2], [-1, 0, 0, 6], [-5, 306, 0, 64]]
    assert ot.token_item_key_blocks(cu, tm[2], 128) == 1
    assert ot.token_item_key_blocks(cu, tm[3], 128) == 1
    # a run longer than one tile, cut at 256 rows; the second tile starts inside a segment
    lengths = [40] * 10
    cu, _, _, _ = op.build_metadata(lengths)
    tm = ot.fwd_tile_map(cu, 2, 256, 128, True, 64)
    assert tm.tolist() == [[-1, 0, 0, 256], [-1, 0, 1, 256], [-7, 256, 0, 144], [-7, 256, 1, 144]]
    assert ot.token_item_key_blocks(cu, tm[2], 128) == 2   # keys [240, 400)
    # non-causal calls and short = 0 keep segment records only
    assert (ot.fwd_tile_map(cu, 1, 256, 128, False, 64)[:, 0] >= 0).all()
    assert (ot.fwd_tile_map(cu, 1, 256, 128, True, 0)[:, 0] >= 0).all()


@pytest.mark.parametrize("BM,BN", [(2, 2), (2, 4), (4, 2), (128, 128), (64, 128)])
@pytest.mark.parametrize("short", [0, 1, 2, 64])
def test_bwd_tile_map_covers_each_allowed_edge_once(BM, BN, short):
    lengths = [5, 1, 9, 3, 260, 130, 2, 1, 1, 64, 3]
    cu, _, _, _ = op.build_metadata(lengths)
    tm = ot.bwd_tile_map(cu, 1, BM, BN, True, short)
    allowed = _allowed_edges(cu.tolist())
    seen = []
    for it in tm:
        b, n, _h, nq = (int(x) for x in it)
        hit = [e for e in ot.bwd_item_edges(cu, it, BM, BN) if e in allowed]
        assert hit
        seen.extend(hit)
        if b < 0:   # token tile: BN-row tiles of a run of short segments
            assert 1 <= nq <= BN and cu[-1 - b] <= n < cu[-b]
            assert all(cu[x + 1] - cu[x] <= short for x in range(len(cu) - 1)
                       if cu[x] < n + nq and cu[x + 1] > n)
            continue
        s, l = cu[b], cu[b + 1] - cu[b]
        assert l > short
        m0 = -(-l // BM) - nq
        cols = range(s + n * BN, s + min(l, (n + 1) * BN))
        # rows before m0 * BM see none of these keys
        assert all((i, j) not in allowed for i in range(s, s + m0 * BM) for j in cols)
    assert sorted(seen) == sorted(allowed)
    tok = tm[tm[:, 0] < 0]
    assert np.array_equal(tm[len(tm) - len(tok):], tok)      # token records come last
    assert [(r[1], r[2]) for r in tok] == sorted((r[1], r[2]) for r in tok)


def test_bwd_token_map_hand_example():
    """Lengths 3, 2, 1, 300, 4, 60 with BM=64, BN=128, short=64: segment 3's kv blocks
    n = 0, 1, 2 see 5, 3, 1 q blocks (m_start = 2n); the runs [0, 6) and [306, 370) are one
    key tile each."""
    cu, _, _, _ = op.build_metadata([3, 2, 1, 300, 4, 60])
    tm = ot.bwd_tile_map(cu, 1, 64, 128, True, 64)
    assert tm.tolist() == [[3, 0, 0, 5], [3, 1, 0, 3], [3, 2, 0, 1], [-1, 0, 0, 6], [-5, 306, 0, 64]]
    # key 305 (last of segment 3) is not in a token tile; key 309 (last of segment 4) is seen
    # by queries 309 only; key 306 by 306..309
    edges = ot.bwd_item_edges(cu, tm[4], 64, 128)
    assert (309, 306) in edges and (310, 306) in edges     # covered; (310, 306) not permitted
    allowed = _allowed_edges(cu.tolist())
    assert (310, 306) not in allowed and (309, 306) in allowed


def test_tile_map_noncausal_counts():
    cu = [0, 300, 301]
    tm = ot.fwd_tile_map(cu, 1, 128, 128, causal=False)
    assert tm.tolist() == [[0, 0, 0, 3], [0, 1, 0, 3], [0, 2, 0, 3], [1, 0, 0, 1]]


def test_tile_map_order_small_example():
    """Segments 300 and 1000 at BM=256, BN=128, causal, 2 heads: the long segment (cost
    2+4+6+8 = 20, class 4) precedes the short one (2+3 = 5, class 2); within a (segment, head)
    the block with the most key tiles comes first."""
    tm = ot.fwd_tile_map([0, 300, 1300], 2, 256, 128)
    assert tm.tolist() == [[1, 3, 0, 8], [1, 2, 0, 6], [1, 1, 0, 4], [1, 0, 0, 2],
                           [1, 3, 1, 8], [1, 2, 1, 6], [1, 1, 1, 4], [1, 0, 1, 2],
                           [0, 1, 0, 3], [0, 0, 0, 2], [0, 1, 1, 3], [0, 0, 1, 2]]
    tb = ot.bwd_tile_map([0, 300, 1300], 1, 64, 128)
    # segment 1 (l=1000): Mq=16, kv blocks 0..7 with n_q = 16,14,...,2 (sum 72, class 6);
    # segment 0 (l=300): Mq=5, kv blocks 0..2 with n_q = 5,3,1 (sum 9, class 3)
    assert tb[:, 0].tolist() == [1] * 8 + [0] * 3
    assert tb[:8, 3].tolist() == [16, 14, 12, 10, 8, 6, 4, 2]
    assert tb[8:, 3].tolist() == [5, 3, 1]


@pytest.mark.parametrize("layout", ["right", "left", "holes"])
def test_unpad_pad_bridge(layout):
    """Blog section 4's padded-batch path: per row the real tokens, in order, form one segment;
    pad(unpad(x)) keeps the real tokens and zeroes the padding; and varlen attention over the
    unpadded stream equals each row's attention over its own real tokens, whatever the padding
    side (brute force per row)."""
    from oracle import attention as oa
    rng = np.random.default_rng({"right": 1, "left": 2, "holes": 3}[layout])
    Bp, S, H, d = 4, 9, 2, 8
    lens = [9, 3, 6, 1]
    mask = np.zeros((Bp, S), dtype=np.int32)
    for r, L in enumerate(lens):
        if layout == "right":
            mask[r, :L] = 1
        elif layout == "left":
            mask[r, S - L:] = 1
        else:
            mask[r, rng.choice(S, L, replace=False)] = 1
    idx, inv, cu, T, mx = op.unpad_index(mask)
    assert T == sum(lens) and list(cu) == [0, 9, 12, 18, 19] and mx == 9
    assert (idx[T:] == -1).all() and sorted(idx[:T]) == list(idx[:T])
    assert all(inv[f] == i for i, f in enumerate(idx[:T])) and (inv >= 0).sum() == T
    x = rng.standard_normal((Bp * S, H, d))
    packed = op.gather_rows(x, idx[:T])
    back = op.gather_rows(packed, inv)
    assert np.array_equal(back, x * mask.reshape(-1, 1, 1))
    q, k, v = (rng.standard_normal((Bp, S, H, d)) for _ in range(3))
    pq, pk, pv = (op.gather_rows(t.reshape(Bp * S, H, d), idx[:T]) for t in (q, k, v))
    o, _ = oa.varlen_forward(pq, pk, pv, cu)
    out = op.gather_rows(o, inv).reshape(Bp, S, H, d)
    for r in range(Bp):
        sel = mask[r].astype(bool)
        ro, _ = oa.segment_forward(q[r, sel], k[r, sel], v[r, sel], 1 / np.sqrt(d))
        assert np.allclose(out[r, sel], ro, atol=1e-12) and (out[r, ~sel] == 0).all()
    with pytest.raises(ValueError):
        op.unpad_index(np.array([[1, 0], [0, 0]]))


@pytest.mark.parametrize("BM,BN", [(2, 2), (4, 2), (2, 4), (256, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("w", [0, 1, 5, 100, 300])
def test_window_tile_maps_cover_each_allowed_edge_once(BM, BN, w):
    """Local window w (a query sees itself and the w keys before it): the forward (q-block)
    and backward (kv-block) maps cover every permitted edge exactly once, every listed tile
    holds a permitted edge, and a segment's blocks keep block order."""
    lengths = [5, 1, 9, 3, 260, 130, 2, 700, 64, 3]
    cu, _, _, _ = op.build_metadata(lengths)
    cu = [int(x) for x in cu]
    allowed = {(i, j) for (i, j) in _allowed_edges(cu)
               if j >= i - w}
    fm = ot.fwd_tile_map(cu, 1, BM, BN, True, 64, window=w)   # token tiles stay off
    bm = ot.bwd_tile_map(cu, 1, BM, BN, True, 64, window=w)
    assert (fm[:, 0] >= 0).all() and (bm[:, 0] >= 0).all()
    for tm, edges in ((fm, ot.fwd_item_edges), (bm, ot.bwd_item_edges)):
        seen = []
        for it in tm:
            hit = [e for e in edges(cu, it, BM, BN, window=w) if e in allowed]
            assert hit, "a listed tile has no permitted edge"
            seen.extend(hit)
        assert sorted(seen) == sorted(allowed)
        for b in set(int(x) for x in tm[:, 0]):
            blk = [int(r[1]) for r in tm if r[0] == b]
            assert blk == (sorted(blk, reverse=True) if tm is fm else sorted(blk))


@pytest.mark.parametrize("BM,BN", [(2, 2), (4, 2), (2, 4), (256, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("causal", [True, False])
def test_cross_tile_maps_cover_each_allowed_edge_once(BM, BN, causal):
    """cu_q != cu_k with bottom-right causal alignment (query i of a segment sees keys
    j <= i + lk - lq): the q-block and kv-block maps cover every permitted (query, key) pair
    exactly once, every listed tile holds one, and lq = lk gives the self-attention maps."""
    lq = [1, 5, 17, 3, 40, 300, 129, 2]
    lk = [1, 9, 17, 30, 41, 700, 129, 260]
    cuq, cuk = [int(x) for x in np.cumsum([0] + lq)], [int(x) for x in np.cumsum([0] + lk)]
    allowed = {(cuq[b] + i, cuk[b] + j) for b in range(len(lq)) for i in range(lq[b]) for j in range(lk[b])
               if not causal or j <= i + lk[b] - lq[b]}
    fm = ot.fwd_tile_map(cuq, 1, BM, BN, causal, 64, cu_k=cuk)
    bm = ot.bwd_tile_map(cuq, 1, BM, BN, causal, 64, cu_k=cuk)
    assert (fm[:, 0] >= 0).all() and (bm[:, 0] >= 0).all()   # no token records
    for tm, edges in ((fm, ot.fwd_item_edges), (bm, ot.bwd_item_edges)):
        seen = []
        for it in tm:
            hit = [e for e in edges(cuq, it, BM, BN, cu_k=cuk) if e in allowed]
            assert hit, "a listed tile has no permitted edge"
            seen.extend(hit)
        assert sorted(seen) == sorted(allowed)
    # lq = lk gives the self-attention maps; with BM >= BN (every map the library builds) q-block
    # counts strictly grow with the block, so last-first is also the self maps' count order
    if BM >= BN:
        assert np.array_equal(ot.fwd_tile_map(cuq, 2, BM, BN, causal, cu_k=cuq), ot.fwd_tile_map(cuq, 2, BM, BN, causal))
    assert np.array_equal(ot.bwd_tile_map(cuq, 2, BM, BN, causal, cu_k=cuq), ot.bwd_tile_map(cuq, 2, BM, BN, causal))
