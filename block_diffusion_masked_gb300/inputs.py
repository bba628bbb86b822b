"""Seeded synthetic inputs for block-diffusion attention.

Shared by the tests, the benchmark and the smoke check.  It holds none of the
method's arithmetic: it only draws i.i.d. normal numbers from a seeded CPU
generator, scales them and rounds them to bf16 (round to nearest even), so
that the CUDA path and the oracle read the very same low-precision values.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; draw q, k, v, dout in
that order as float32 N(0, 1) of shape (batch, 2n, heads, headdim); multiply
by ``std``; cast to bfloat16.
"""

from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One benchmark/parity workload: shapes, block size, input scale, seed."""

    name: str
    batch: int
    n: int
    heads: int
    headdim: int
    block_size: int
    std: float = 1.0
    seed: int = 0

    @property
    def seqlen(self) -> int:
        return 2 * self.n


# The five workloads the performance claims and parity tests are stated on.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 64, 2, 64, 4, 1.0, 0),
    "small": Workload("small", 8, 1024, 16, 128, 16, 1.0, 1),
    "mid": Workload("mid", 4, 2048, 32, 128, 4, 1.0, 2),
    "long": Workload("long", 1, 8192, 16, 64, 32, 0.5, 3),
    "hd256_bs1": Workload("hd256_bs1", 2, 4096, 8, 256, 1, 1.0, 4),
    "hd256_bs64": Workload("hd256_bs64", 2, 4096, 8, 256, 64, 1.0, 4),
    "hd256_bs128": Workload("hd256_bs128", 2, 4096, 8, 256, 128, 1.0, 4),
}


def make_inputs(batch, n, heads, headdim, seed=0, std=1.0, with_dout=True):
    """Return bf16 CPU tensors q, k, v (and dout) of shape (batch, 2n, heads, headdim)."""
    g = torch.Generator("cpu").manual_seed(seed)
    shape = (batch, 2 * n, heads, headdim)
    names = ("q", "k", "v", "dout") if with_dout else ("q", "k", "v")
    out = []
    for _ in names:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x = x * std
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def make_workload_inputs(w: Workload, with_dout=True):
    return make_inputs(w.batch, w.n, w.heads, w.headdim, seed=w.seed, std=w.std,
                       with_dout=with_dout)
