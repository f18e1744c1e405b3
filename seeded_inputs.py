"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA path.

This module only draws random numbers and names workload sizes. It holds none
of the method's arithmetic: no packing decision, no boundary array, no
attention.  Both sides (the CPU oracle in ``oracle/`` and the GPU library in
``packed_sequence_varlen_gb300/``) receive the same raw draws from here and
each runs its own planner, metadata and attention code on them.

Workloads (the shapes of the pages' packing examples, scaled to training sizes;
the pages measure on no public dataset, so these stand alone):

* ``tiny``      -- T=12 as segments 5/3/4 (and 5/7 merged), H=2, d=64, fp32
                   N(0,1) tensors, the three-sample layout of "Packing与
                   FlashAttention Varlen", section 1.
* ``sft8k``     -- segment lengths uniform in [32, 2048], next-fit into a
                   packing length of 8192, tail padded to 8192; Hq=Hkv=32, d=128.
* ``gqa16k``    -- 400 lengths rint(lognormal(ln 512, 1.0)) clipped to
                   [16, 8192], best-fit-decreasing into 16384, tail padded;
                   Hq=32, Hkv=8, d=128.
* ``long64k``   -- fixed segments [32768,16384,8192,4096,2048,1024,512,512],
                   T=65536, Hq=Hkv=16, d=128.
* ``tiny4k``    -- lengths uniform in [1, 64], next-fit into 131072, first row
                   (about 4000 segments), tail padded; Hq=Hkv=8, d=64.

Tensor draws: ``torch.Generator().manual_seed(s)`` then ``randn`` in fp32 on
the CPU, rounded to bf16 (s = 1, 2, 3, 4 for q, k, v, dO, plus an optional
offset for several packs).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    Hq: int
    Hkv: int
    d: int
    capacity: int          # packing length (tokens per pack)
    strategy: str          # "next_fit" | "best_fit_decreasing" | "fixed"
    pad_to: int            # pack is tail padded to this many tokens (0: no pad)
    causal: bool = True
    description: str = ""
    fixed_lengths: tuple = field(default_factory=tuple)
    packs_used: int = 0    # the workload is its first this many packs (0: all of them)


WORKLOADS = {
    "tiny": Workload("tiny", 2, 2, 64, 12, "fixed", 0,
                     description="T=12, segments 5/3/4, H=2, d=64, fp32 N(0,1)",
                     fixed_lengths=(5, 3, 4)),
    "sft8k": Workload("sft8k", 32, 32, 128, 8192, "next_fit", 8192,
                      description="lengths U[32,2048], next-fit into 8192, "
                                  "tail padded, Hq=Hkv=32, d=128, bf16"),
    "gqa16k": Workload("gqa16k", 32, 8, 128, 16384, "best_fit_decreasing", 16384,
                       description="400 lengths lognormal(median 512, sigma 1) "
                                   "clipped [16,8192], BFD into 16384, tail padded, "
                                   "Hq=32, Hkv=8, d=128, bf16"),
    "long64k": Workload("long64k", 16, 16, 128, 65536, "fixed", 0,
                        description="segments 32768..512, T=65536, Hq=Hkv=16, "
                                    "d=128, bf16",
                        fixed_lengths=(32768, 16384, 8192, 4096, 2048, 1024, 512, 512)),
    "tiny4k": Workload("tiny4k", 8, 8, 64, 131072, "next_fit", 131072,
                       description="lengths U[1,64], next-fit into 131072, first "
                                   "row (~4000 segments), tail padded, Hq=Hkv=8, "
                                   "d=64, bf16",
                       packs_used=1),
}


def raw_lengths(name: str, seed: int = 0) -> np.ndarray:
    """The raw document-length stream a workload packs (int64, in draw order).

    Only random draws: the planner (next-fit / best-fit-decreasing) that turns
    this stream into packs is applied separately by each side.
    """
    w = WORKLOADS[name]
    if w.strategy == "fixed":
        return np.asarray(w.fixed_lengths, dtype=np.int64)
    rng = np.random.default_rng(seed)
    if name == "sft8k":
        # enough documents for well over 16 packs of 8192 tokens
        return rng.integers(32, 2049, size=400).astype(np.int64)
    if name == "gqa16k":
        x = rng.lognormal(mean=np.log(512.0), sigma=1.0, size=400)
        return np.clip(np.rint(x), 16, 8192).astype(np.int64)
    if name == "tiny4k":
        # the first next-fit row of 131072 tokens needs about 4000 draws
        return rng.integers(1, 65, size=6000).astype(np.int64)
    raise KeyError(name)


def random_lengths(rng: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    """Uniform integer lengths in [lo, hi] for property tests."""
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def tensors(T: int, Hq: int, Hkv: int, d: int, seed_offset: int = 0,
            dtype: torch.dtype = torch.bfloat16, with_dout: bool = True):
    """q, k, v (and dO) as CPU tensors [T, H, d]: N(0,1) fp32 draws, then cast.

    Seeds are 1, 2, 3, 4 (+ ``seed_offset``) for q, k, v, dO.
    """
    def draw(seed, H):
        g = torch.Generator().manual_seed(seed + seed_offset)
        x = torch.randn((T, H, d), generator=g, dtype=torch.float32)
        return x.to(dtype)

    q = draw(1, Hq)
    k = draw(2, Hkv)
    v = draw(3, Hkv)
    if not with_dout:
        return q, k, v
    return q, k, v, draw(4, Hq)


def to_f64(x: torch.Tensor) -> np.ndarray:
    """Exact upcast of a CPU tensor (bf16 / fp32) to a float64 numpy array."""
    return x.detach().to(torch.float64).cpu().numpy()
