"""One ES generation of a population split over the ranks of a process group.

EvoX API page "evox.triton_kernels.kernels.virtual_noise", section "Noise
indexing scheme": element k of block b of individual i has the noise of index
``offsets[b] + k``, so a contiguous range ``[e0, e1)`` of the flat parameter
vector (every block laid out by ``compute_offsets``, weights then bias, layer by
layer) is, for the gradient, the same as a block of ``e1 - e0`` elements starting
at ``offset + e0``; within one weight block a row block ``[r0, r1)`` is the range
``[r0*in, r1*in)``. The module description's estimate sums over the whole
population, and individuals are independent in the forward. So one generation
over ``world`` ranks is:

  1. forward of the rank's individuals ``[p0, p1)`` with the replicated
     parameters (``virtual_perturbed_mlp``: every layer in one launch);
  2. the rank's returns (the caller's objective on its outputs) all-gathered
     into the population's returns -- ``pop`` floats, the one exchange before
     the gradient (seeds are known everywhere);
  3. the centered ranks of all returns (every rank computes the same vector);
  4. the gradient estimate and the step ``theta += lr * grad`` over the rank's
     range ``[e0, e1)`` of the flat parameter vector, for the whole population:
     one ``gradient_update`` call at ``offset + e0``;
  5. the updated ranges all-gathered into the parameter vector, which is then
     replicated again (``n_params`` floats).

Ranges are contiguous and balanced: rank r of w owns ``[ceil(n/w)*r, ...)``; the
gathers move equal-sized, zero-padded chunks. No kernel of one rank waits on
another rank's: the exchanges are collectives between launches. The compute
steps are the library's by default; ``ops`` replaces them (tests run the
orchestration on CPU processes with stand-ins).
"""

from __future__ import annotations

from typing import Callable, Optional, Sequence

import torch


def split(n: int, world: int, rank: int):
    """Rank ``rank``'s contiguous range ``(lo, hi)`` of ``n`` items in chunks of
    ``ceil(n / world)`` (the last ranks' chunks may be short or empty)."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError(f"bad split: n={n}, world={world}, rank={rank}")
    chunk = -(-n // world)
    lo = min(n, rank * chunk)
    return lo, min(n, lo + chunk)


class LibraryOps:
    """The generation's compute steps as the library's calls (the product path)."""

    def forward(self, x, weights, biases, seeds, sigma, offsets, activation):
        from .api import virtual_perturbed_mlp
        return virtual_perturbed_mlp(x, weights, biases, seeds, sigma, offsets, activation=activation)

    def centered_ranks(self, returns):
        from .api import centered_ranks
        return centered_ranks(returns)

    def gradient_update(self, fitness, seeds, theta_range, sigma, pop, lr, offset):
        from .api import gradient_update
        return gradient_update(fitness, seeds, theta_range, sigma, pop, lr, offset)


def world_and_rank(group=None):
    """(world size, rank) of ``group``; (1, 0) when no process group is initialised."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def all_gather_padded(local: torch.Tensor, chunk: int, n: int, group=None) -> torch.Tensor:
    """Concatenate every rank's ``local`` (at most ``chunk`` elements, 1-D) in rank
    order and return the first ``n`` elements. Chunks are zero-padded to ``chunk``
    so that every rank sends the same size. CUDA tensors go through the host when
    the group's backend is gloo. With one rank (or no process group) this is
    ``local`` itself."""
    import torch.distributed as dist

    world, _ = world_and_rank(group)
    if world == 1:
        return local[:n]
    backend = dist.get_backend(group)
    dev = local.device
    via_host = dev.type == "cuda" and backend == "gloo"
    buf = torch.zeros(chunk, dtype=local.dtype, device="cpu" if via_host else dev)
    buf[:local.numel()] = local.to(buf.device)
    if backend == "nccl":
        out = torch.empty(world * chunk, dtype=local.dtype, device=dev)
        dist.all_gather_into_tensor(out, buf, group=group)
    else:
        parts = [torch.empty_like(buf) for _ in range(world)]
        dist.all_gather(parts, buf, group=group)
        out = torch.cat(parts)
    return out[:n].to(dev)


def es_generation(theta: torch.Tensor, dims: Sequence[int], x_local: torch.Tensor,
                  seeds: torch.Tensor, returns_fn: Callable[[torch.Tensor], torch.Tensor],
                  sigma: float, lr: float, *, offset: int = 0, activation: Optional[str] = "tanh",
                  group=None, ops=None) -> dict:
    """One ES generation of the policy ``dims[0] -> dims[1] -> ... -> dims[-1]`` whose
    parameters ``theta`` (fp32, flat: W_0, b_0, W_1, b_1, ... as compute_offsets lays
    them out, starting at element index ``offset``) are replicated on every rank.

    seeds       the whole population's seeds (pop,), the same on every rank;
    x_local     this rank's individuals' inputs (p1 - p0, batch, dims[0]), where
                ``(p0, p1) = split(pop, world, rank)``;
    returns_fn  the objective: this rank's outputs (p1 - p0, batch, dims[-1]) -> its
                returns (p1 - p0,) fp32.
    theta is updated in place (the same values on every rank afterwards). Returns the
    population's returns and fitness, this rank's gradient range and its bounds.
    Without an initialised process group the generation runs on one rank."""
    ops = ops or LibraryOps()
    world, rank = world_and_rank(group)
    pop = int(seeds.numel())
    n = int(theta.numel())
    shapes = []
    for a, c in zip(dims[:-1], dims[1:]):
        shapes += [(c, a), (c,)]
    from .api import compute_offsets
    offs = compute_offsets(shapes)
    if offs[-1] + shapes[-1][0] != n:
        raise ValueError(f"theta has {n} elements, the layers {offs[-1] + shapes[-1][0]}")
    views = []
    for o, sh in zip(offs, shapes):
        size = 1
        for d in sh:
            size *= d
        views.append(theta[o:o + size].view(*sh))

    # 1. forward of this rank's individuals
    p0, p1 = split(pop, world, rank)
    if x_local.shape[0] != p1 - p0:
        raise ValueError(f"rank {rank} holds individuals [{p0}, {p1}) but x_local has {x_local.shape[0]}")
    if p1 > p0:
        y = ops.forward(x_local, views[0::2], views[1::2], seeds[p0:p1], sigma,
                        [offset + o for o in offs[0::2]], activation)
        ret_local = returns_fn(y).reshape(-1).to(torch.float32)
    else:
        ret_local = torch.zeros(0, dtype=torch.float32, device=theta.device)
    # 2. the population's returns
    returns = all_gather_padded(ret_local, -(-pop // world), pop, group)
    # 3. fitness shaping (identical on every rank)
    fitness = ops.centered_ranks(returns)
    # 4. this rank's range of the flat gradient and its update, over the whole population
    e0, e1 = split(n, world, rank)
    grad = ops.gradient_update(fitness, seeds, theta[e0:e1], sigma, pop, lr, offset + e0) \
        if e1 > e0 else torch.zeros(0, dtype=torch.float32, device=theta.device)
    # 5. the updated parameters, replicated again
    theta.copy_(all_gather_padded(theta[e0:e1], -(-n // world), n, group))
    return {"returns": returns, "fitness": fitness, "grad_range": grad, "range": (e0, e1),
            "individuals": (p0, p1)}
