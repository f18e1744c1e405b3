"""GPU parity of the packed loss layout against the float64 oracle (oracle/loss.py).

Targets formed inside each segment are bit-exact; the token-weighted loss and its logit
gradient are compared with the oracle on identical inputs, and the pages' nine-target probe
must give its printed 7.624619 / 0.847180 (11 ln2 and 11 ln2 / 9).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import loss as ol
from oracle import packing as op
import _workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
VA_ERR_BAD_TARGETS = 8


@pytest.fixture(scope="module")
def va():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from packed_sequence_varlen_gb300 import build as b
    b.build()
    import packed_sequence_varlen_gb300 as pkg
    pkg._lib.load()
    return pkg


def nine_target_stream(golden_dir):
    fx = json.load(open(os.path.join(golden_dir, "nine_target_fixture.json")))
    docs = [i + t[-1:] for i, t in zip(fx["pair_inputs"], fx["pair_targets"])]
    ids = sum(docs, [])
    cu = np.cumsum([0] + [len(d) for d in docs])
    return fx, ids, cu


def test_nine_target_probe(va, golden_dir):
    """The pages' three documents as one packed stream: the device forms the nine targets,
    and the constructed logits (gold probability 1/2, 1/4, 1/2 per document) give the
    printed token-weighted loss, not the row-mean or document-mean ones."""
    fx, ids, cu = nine_target_stream(golden_dir)
    idd = torch.tensor(ids, dtype=torch.int32, device=DEV)
    cud = torch.tensor(cu, dtype=torch.int32, device=DEV)
    tg = va.loss_targets(idd, cud).cpu().numpy()
    ref = ol.stream_targets(ids, cu)
    assert np.array_equal(tg, ref)
    elig = ref != ol.IGNORE_INDEX
    seg = np.repeat(np.arange(3), np.diff(cu))
    qmap = {int(k): v for k, v in fx["gold_probability_by_segment"].items()}
    z = ol.constructed_logits(ref, elig, [qmap[int(s)] for s in seg], fx["vocab"])
    rs, rmean, rgrad = ol.token_weighted_loss(z, ref, elig)
    logits = torch.tensor(z, dtype=torch.float32, device=DEV)
    loss, count, grad = va.token_ce(logits, torch.tensor(tg, device=DEV), check_status=True)
    s, mean = loss.cpu().tolist()
    # fp32 per row: nine base-2 log-sum-exps of magnitude ~ log2(266), each rounded at 2^-24
    # relative, keep the sum within 1e-5 of 11 ln2 (the printed values are 11 ln2 and 11 ln2 / 9
    # to six decimals)
    assert int(count.item()) == fx["real_targets"] == 9
    assert abs(s - 11 * math.log(2)) < 1e-5 and abs(s - fx["loss_sum_printed"]) < 1e-5
    assert abs(mean - 11 * math.log(2) / 9) < 2e-6 and abs(mean - fx["loss_mean_printed"]) < 2e-6
    assert abs(mean - fx["row_mean_printed"]) > 1e-3 and abs(mean - fx["document_mean_printed"]) > 1e-3
    g = grad.cpu().double().numpy()
    assert np.abs(g - rgrad).max() < 1e-6
    assert np.all(g[~elig] == 0)


def test_targets_bit_exact_on_workload_boundaries(va):
    """Targets of random token ids over every workload's first pack boundaries."""
    gen = torch.Generator().manual_seed(5)
    for name in ("sft8k", "gqa16k", "long64k", "tiny4k"):
        lengths = wl.pack(name)
        cu, *_ = op.build_metadata(lengths)
        T = int(cu[-1])
        ids = torch.randint(0, 50000, (T,), generator=gen, dtype=torch.int32)
        tg = va.loss_targets(ids.to(DEV), torch.tensor(cu, dtype=torch.int32, device=DEV))
        assert np.array_equal(tg.cpu().numpy(), ol.stream_targets(ids.numpy(), cu))


# 16-byte row accesses (bf16, V = 32000); element-wise rows (fp32, V = 5003: rows not 16-byte
# multiples); 16-byte accesses with an element-wise tail (bf16, V = 1001 in rows of 1008)
@pytest.mark.parametrize("dtype,V,stride", [(torch.bfloat16, 32000, 32000), (torch.float32, 5003, 5003),
                                            (torch.bfloat16, 1001, 1008)])
def test_token_ce_random(va, dtype, V, stride):
    """Logits N(0, 3^2) rounded to the dtype, targets from packed segments (about a fifth of
    the rows ignored), one ignored row full of NaN: loss sum relative 1e-5, mean, count exact,
    gradient relative-L2 1e-2 (bf16 output) or 1e-5 (fp32), ignored rows exactly zero."""
    gen = torch.Generator().manual_seed(V)
    lengths = [int(x) for x in torch.randint(1, 40, (100,), generator=gen)]
    cu, *_ = op.build_metadata(lengths)
    T = int(cu[-1])
    ids = torch.randint(0, V, (T,), generator=gen, dtype=torch.int32)
    ref_t = ol.stream_targets(ids.numpy(), cu)
    z = (3 * torch.randn(T, V, generator=gen)).to(dtype)
    elig = ref_t != ol.IGNORE_INDEX
    bad_row = int(np.nonzero(~elig)[0][3])
    z[bad_row] = float("nan")           # never read: the row has no target
    tg = va.loss_targets(ids.to(DEV), torch.tensor(cu, dtype=torch.int32, device=DEV))
    zd = torch.zeros(T, stride, dtype=dtype, device=DEV)[:, :V]
    zd.copy_(z)
    gd = torch.full((T, stride), 7.0, dtype=dtype, device=DEV)[:, :V]
    loss, count, grad = va.token_ce(zd, tg, grad=gd, check_status=True)
    zz = z.double().numpy()
    zz[bad_row] = 0.0                   # the oracle skips it too; any finite value
    rs, rmean, rgrad = ol.token_weighted_loss(zz, ref_t, elig)
    s, mean = loss.cpu().tolist()
    assert int(count.item()) == int(elig.sum())
    assert abs(s - rs) <= 1e-5 * abs(rs) and abs(mean - rmean) <= 1e-5 * abs(rmean)
    g = grad.cpu().double().numpy()
    assert np.all(g[~elig] == 0) and np.isfinite(g).all()
    tol = 1e-2 if dtype == torch.bfloat16 else 1e-5
    assert wl.rel_l2(g[elig], rgrad[elig]) <= tol
    # no gradient requested: the same loss
    loss2, _, none = va.token_ce(zd, tg, grad=False)
    assert none is None and loss2.cpu().tolist() == [s, mean]


def test_token_ce_device_errors(va):
    """An eligible target outside [0, V), or no eligible target, sets VA_ERR_BAD_TARGETS in the
    status word and the loss to NaN."""
    z = torch.randn(6, 50, device=DEV)
    ws = torch.empty(va._lib.load().varlen_token_ce_workspace_size(6), dtype=torch.uint8, device=DEV)
    for t in ([1, 2, 50, -100, 3, 4], [1, -5, 2, 3, 4, 5], [-100] * 6):
        loss, _, _ = va.token_ce(z, torch.tensor(t, dtype=torch.int32, device=DEV), workspace=ws)
        assert va.read_status(ws) == VA_ERR_BAD_TARGETS
        assert all(math.isnan(x) for x in loss.cpu().tolist())
    loss, _, _ = va.token_ce(z, torch.tensor([1, 2, 49, -100, 0, 4], dtype=torch.int32, device=DEV), workspace=ws)
    assert va.read_status(ws) == 0 and all(math.isfinite(x) for x in loss.cpu().tolist())
