"""The multi-process path of bench.py on CPU: world size 2 over gloo (no GPU).

Replicas only: each rank takes its own packs (no data-path collective); the only collectives
are the whole-job timing reductions -- the elapsed time is the maximum over ranks and the
work the sum over ranks."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        idx = bench.rank_pack_indices(rank, 16, 40)
        # rank r ran 10 + r ms and did (r + 1) * 100 units per step over 3 steps
        mx, tot = bench.aggregate(10.0 + rank, 100.0 * (rank + 1), 3, dist, "cpu")
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{mx} {tot} {' '.join(map(str, idx))}\n")
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for r in rows:
        assert float(r[0]) == 11.0               # the slowest rank's time
        assert float(r[1]) == 3 * (100 + 200)    # every rank's work
    idx0, idx1 = (list(map(int, r[2:])) for r in rows)
    assert idx0 == list(range(16)) and idx1 == list(range(16, 32))
    assert not set(idx0) & set(idx1)             # disjoint packs: no exchange needed


def test_single_process_aggregate_and_wraparound():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(5.0, 7.0, 4) == (5.0, 28.0)
    assert bench.rank_pack_indices(2, 16, 40) == [(32 + i) % 40 for i in range(16)]


@pytest.mark.parametrize("name", ["sft8k", "gqa16k", "long64k", "tiny4k"])
def test_bench_packs_are_the_workload_packs(name):
    """Every pack a rank times is one of the workload's own packs (the ones the parity tests
    check): tiny4k, for one, is its first next-fit row, not the partial row its leftover
    draws would form."""
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    import _workloads as wl
    from oracle import packing as op
    old = bench.WORKLOAD, bench.PACKS_PER_STEP
    try:
        bench.WORKLOAD, bench.PACKS_PER_STEP = name, 16
        own = [list(p) for p, _ in wl.real_packs(name)]
        for rank in (0, 1):
            packs, idx, w = bench.batch_packs(rank, (op.next_fit, op.best_fit_decreasing))
            assert len(packs) == 16 and all(0 <= i < len(own) for i in idx)
            assert all(list(p) == own[i] for p, i in zip(packs, idx))
    finally:
        bench.WORKLOAD, bench.PACKS_PER_STEP = old
