"""Seeded synthetic inputs for the five benchmark / parity workloads.

This module draws random inputs only; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.
No dataset or trained weight is involved: every tensor is drawn on the CPU
with ``torch.Generator().manual_seed(1000 + number)`` in the order X, W, b,
fitness (fp32 draws, then cast where a workload says bf16). Fitness is either
N(0, 1) or "centered ranks": a seeded random permutation r of 0..pop-1 mapped
to r / (pop - 1) - 0.5, a value in [-0.5, 0.5]. Distributions are written
N(mean, variance), so W ~ N(0, 1/in) has standard deviation 1/sqrt(in) and
b ~ N(0, 0.01) has standard deviation 0.1.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch


@dataclasses.dataclass
class Layer:
    in_f: int
    out_f: int
    weight: torch.Tensor               # (out, in)
    bias: Optional[torch.Tensor]       # (out,) or None
    offset: int                        # weight block offset; bias block at offset + out*in


@dataclasses.dataclass
class Workload:
    number: int
    name: str
    description: str
    pop: int
    batch: int
    sigma: float
    seeds: torch.Tensor                # (pop,) int64
    x: torch.Tensor                    # (pop, batch, in) of the first layer
    layers: List[Layer]
    fitness: torch.Tensor              # (pop,) fp32
    activation: Optional[str] = None   # between layers
    forward: bool = True               # the workload runs the forward
    grads: bool = True                 # the workload runs the gradient estimates
    # Raw returns (pop,) fp32 for the workloads whose fitness is centered ranks: the
    # full ES generation shapes them into ranks on the device. Drawn from a separate
    # generator (seed 2000 + number), so the other tensors do not depend on them.
    returns: Optional[torch.Tensor] = None

    def to(self, device) -> "Workload":
        d = dataclasses.replace(self)
        d.seeds = self.seeds.to(device)
        d.x = self.x.to(device)
        d.fitness = self.fitness.to(device)
        d.returns = None if self.returns is None else self.returns.to(device)
        d.layers = [dataclasses.replace(l, weight=l.weight.to(device),
                                        bias=None if l.bias is None else l.bias.to(device))
                    for l in self.layers]
        return d

    def first(self, pop: int) -> "Workload":
        """The same workload restricted to its first ``pop`` individuals (smaller
        cases of the same shapes, e.g. for profiling)."""
        if not 1 <= pop <= self.pop:
            raise ValueError(f"pop must be in [1, {self.pop}]")
        d = dataclasses.replace(self)
        d.pop = pop
        d.seeds = self.seeds[:pop]
        d.fitness = self.fitness[:pop]
        d.returns = None if self.returns is None else self.returns[:pop]
        if self.x.dim() == 3:
            d.x = self.x[:pop]
        return d

    @property
    def noise_elements(self) -> int:
        """pop * (parameters of every block): noise elements per full regeneration."""
        return self.pop * sum(l.out_f * l.in_f + (l.out_f if l.bias is not None else 0)
                              for l in self.layers)


def centered_ranks(pop: int, gen: torch.Generator) -> torch.Tensor:
    r = torch.randperm(pop, generator=gen).to(torch.float64)
    return (r / max(pop - 1, 1) - 0.5).to(torch.float32)


def _returns(number: int, pop: int) -> torch.Tensor:
    """Synthetic raw returns N(0, 1), rounded to multiples of 1/64 so that ties occur."""
    g = torch.Generator().manual_seed(2000 + number)
    return torch.round(torch.randn(pop, generator=g, dtype=torch.float32) * 64) / 64


def _normal(shape, var: float, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32) * math.sqrt(var)


NAMES = {1: "tiny", 2: "es_mlp", 3: "mid", 4: "grad_only", 5: "large_tc"}
DESCRIPTIONS = {
    1: "tiny ES linear: pop 8 (seeds 0..7), batch 4, 32->16, fp32, sigma 0.01",
    2: "ES MLP policy: pop 1024, batch 1, 64->256->256->8 with tanh, fp32, sigma 0.02, centered ranks",
    3: "mid perturbed linear: pop 4096, batch 32, 1024->1024, X bf16, W fp32, sigma 0.01",
    4: "gradient-only: out=in=4096, pop 16384 (seeds 1..16384), sigma 0.005, offset 123456789",
    5: "large tensor-core forward: pop 256, batch 256, 4096->4096, X/W/Y bf16, sigma 0.01",
}


def make(number: int) -> Workload:
    """Build workload ``number`` (1..5) on the CPU."""
    g = torch.Generator().manual_seed(1000 + number)
    if number == 1:
        pop, batch, in_f, out_f = 8, 4, 32, 16
        x = _normal((pop, batch, in_f), 1.0, g)
        w = _normal((out_f, in_f), 1.0 / in_f, g)
        b = torch.zeros(out_f)
        f = _normal((pop,), 1.0, g)
        return Workload(1, NAMES[1], DESCRIPTIONS[1], pop, batch, 0.01, torch.arange(pop, dtype=torch.int64),
                        x, [Layer(in_f, out_f, w, b, 0)], f)
    if number == 2:
        pop, batch, dims = 1024, 1, [64, 256, 256, 8]
        x = _normal((pop, batch, dims[0]), 1.0, g)
        shapes = []
        for a, c in zip(dims[:-1], dims[1:]):
            shapes += [(c, a), (c,)]
        offs, total = [], 0
        for s in shapes:
            offs.append(total)
            total += math.prod(s)
        layers = []
        for li, (a, c) in enumerate(zip(dims[:-1], dims[1:])):
            w = _normal((c, a), 1.0 / a, g)
            layers.append(Layer(a, c, w, torch.zeros(c), offs[2 * li]))
        f = centered_ranks(pop, g)
        return Workload(2, NAMES[2], DESCRIPTIONS[2], pop, batch, 0.02,
                        torch.arange(pop, dtype=torch.int64), x, layers, f, activation="tanh",
                        returns=_returns(2, pop))
    if number == 3:
        pop, batch, in_f, out_f = 4096, 32, 1024, 1024
        x = _normal((pop, batch, in_f), 1.0, g).to(torch.bfloat16)
        w = _normal((out_f, in_f), 1.0 / in_f, g)
        b = _normal((out_f,), 0.01, g)
        f = _normal((pop,), 1.0, g)
        return Workload(3, NAMES[3], DESCRIPTIONS[3], pop, batch, 0.01,
                        torch.arange(pop, dtype=torch.int64), x, [Layer(in_f, out_f, w, b, 0)], f)
    if number == 4:
        pop, in_f, out_f = 16384, 4096, 4096
        f = centered_ranks(pop, g)
        layer = Layer(in_f, out_f, torch.empty(0), torch.empty(0), 123456789)
        return Workload(4, NAMES[4], DESCRIPTIONS[4], pop, 0, 0.005,
                        torch.arange(1, pop + 1, dtype=torch.int64), torch.empty(0), [layer], f,
                        forward=False, returns=_returns(4, pop))
    if number == 5:
        pop, batch, in_f, out_f = 256, 256, 4096, 4096
        x = _normal((pop, batch, in_f), 1.0, g).to(torch.bfloat16)
        w = _normal((out_f, in_f), 1.0 / in_f, g).to(torch.bfloat16)
        b = _normal((out_f,), 0.01, g).to(torch.bfloat16)
        f = _normal((pop,), 1.0, g)
        return Workload(5, NAMES[5], DESCRIPTIONS[5], pop, batch, 0.01,
                        torch.arange(pop, dtype=torch.int64), x, [Layer(in_f, out_f, w, b, 0)], f,
                        grads=False)
    raise ValueError(f"no workload {number}")
