"""The population-sharded ES generation (virtual_noise_perturbed_gb300.sharded) on CPU
processes: gloo ranks on 127.0.0.1.

The generation's orchestration -- which individuals a rank runs forward, the
all-gather of the returns, which range of the flat parameter vector a rank's
gradient covers and at which noise offset, the all-gather of the updated
parameters -- is run with the compute steps replaced:
  * by recording stand-ins whose outputs encode their arguments, so that every
    element of the result shows which call produced it (exact checks of the
    partition, the offsets and the gather order at 2 and 3 ranks, uneven sizes);
  * by the oracle's functions, so that the reassembled generation (returns,
    fitness and updated parameters) can be compared with the oracle's own
    unsharded generation (the method's row-slice identity at the level of a
    whole generation).
On a GPU the same function runs the library's kernels (tests/test_gpu_sharded.py)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from virtual_noise_perturbed_gb300.sharded import split


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(world, target, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res, key=lambda r: r[0])


def test_split_covers_the_range_in_equal_chunks():
    for n in (0, 1, 2, 7, 8, 9, 84488, 100003):
        for world in (1, 2, 3, 4, 8):
            parts = [split(n, world, r) for r in range(world)]
            chunk = -(-n // world)
            assert parts[0][0] == 0 and parts[-1][1] == n
            for (a, b), (c, d) in zip(parts, parts[1:]):
                assert b == c                                # contiguous, in rank order
            assert all(0 <= hi - lo <= chunk for lo, hi in parts)
            assert all(lo == min(n, r * chunk) for r, (lo, _) in enumerate(parts))
    with pytest.raises(ValueError):
        split(4, 2, 2)


class RecordingOps:
    """Stand-ins whose results encode their arguments (exact in float32)."""

    def __init__(self):
        self.calls = []

    def forward(self, x, weights, biases, seeds, sigma, offsets, activation):
        self.calls.append(("forward", seeds.tolist(), list(offsets)))
        out = weights[-1].shape[0]
        # output (k, batch, out): the individual's seed, so the returns name who made them
        return seeds.to(torch.float32)[:, None, None].expand(-1, x.shape[1], out).clone()

    def centered_ranks(self, returns):
        self.calls.append(("ranks", returns.tolist()))
        return returns * 2

    def gradient_update(self, fitness, seeds, theta_range, sigma, pop, lr, offset):
        self.calls.append(("grad", int(offset), int(theta_range.numel()), int(pop), int(seeds.numel())))
        g = (offset + torch.arange(theta_range.numel(), dtype=torch.float64)).to(torch.float32) \
            + float(fitness.sum())
        theta_range.add_(g * lr)
        return g


def _recording_worker(rank, world, port, q, pop, dims, offset):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from virtual_noise_perturbed_gb300.sharded import es_generation
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n = sum(a * c + c for a, c in zip(dims[:-1], dims[1:]))
        theta = torch.arange(n, dtype=torch.float32) * 0.5
        seeds = torch.arange(pop, dtype=torch.int64) * 3 + 100
        p0, p1 = split(pop, world, rank)
        x = torch.zeros(p1 - p0, 2, dims[0])
        ops = RecordingOps()
        r = es_generation(theta, dims, x, seeds, lambda y: y[:, 0, 0], 0.1, 1.0, offset=offset,
                          activation=None, ops=ops)
        q.put((rank, theta.tolist(), r["returns"].tolist(), r["range"], r["individuals"], ops.calls))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,pop,dims", [(2, 7, [3, 5, 2]), (3, 8, [4, 6, 6, 1]), (2, 1, [2, 3])])
def test_partition_offsets_and_gathers_are_exact(world, pop, dims):
    offset = 1000
    res = _run(world, _recording_worker, pop, dims, offset)
    n = sum(a * c + c for a, c in zip(dims[:-1], dims[1:]))
    seeds = [s * 3 + 100 for s in range(pop)]
    fit_sum = 2.0 * sum(seeds)
    want = [0.5 * e + (offset + e) + fit_sum for e in range(n)]   # theta + lr*grad, lr = 1
    # the layers' weight offsets: compute_offsets over (W_0, b_0, ...) shifted by `offset`
    w_offs, pos = [], 0
    for a, c in zip(dims[:-1], dims[1:]):
        w_offs.append(offset + pos)
        pos += a * c + c
    for rank, theta, returns, rng, inds, calls in res:
        assert theta == want                                   # every element from its own range
        assert returns == [float(s) for s in seeds]            # gathered in population order
        assert rng == split(n, world, rank) and inds == split(pop, world, rank)
        fwd = [c for c in calls if c[0] == "forward"]
        p0, p1 = inds
        if p1 > p0:
            assert fwd == [("forward", seeds[p0:p1], w_offs)]
        else:
            assert fwd == []
        grad = [c for c in calls if c[0] == "grad"]
        e0, e1 = rng
        assert grad == ([("grad", offset + e0, e1 - e0, pop, pop)] if e1 > e0 else [])


class OracleOps:
    """The compute steps as the oracle's functions (float64), for checking the
    orchestration against the oracle's unsharded generation."""

    def forward(self, x, weights, biases, seeds, sigma, offsets, activation):
        from oracle import es
        h = x.double().numpy()
        for l, (w, b) in enumerate(zip(weights, biases)):
            h = es.perturbed_linear(h, w.double().numpy(), b.double().numpy(), seeds.numpy(), sigma, offsets[l])
            if activation == "tanh" and l < len(weights) - 1:
                h = np.tanh(h)
        return torch.from_numpy(h)

    def centered_ranks(self, returns):
        from oracle import es
        return torch.from_numpy(es.centered_ranks(returns.numpy()))

    def gradient_update(self, fitness, seeds, theta_range, sigma, pop, lr, offset):
        from oracle import es
        g = es.bias_gradient(fitness.numpy(), seeds.numpy(), (theta_range.numel(),), sigma, pop, offset)
        theta_range.copy_(torch.from_numpy(es.es_update(theta_range.numpy(), g, lr)))
        return torch.from_numpy(g)


def _policy(pop, dims, seed):
    g = torch.Generator().manual_seed(seed)
    n = sum(a * c + c for a, c in zip(dims[:-1], dims[1:]))
    theta = (torch.randn(n, generator=g) * 0.3).to(torch.float32)
    x = torch.randn(pop, 2, dims[0], generator=g)
    seeds = torch.arange(pop, dtype=torch.int64) * 7 + 1
    return theta, x, seeds


def _oracle_worker(rank, world, port, q, pop, dims, offset):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from virtual_noise_perturbed_gb300.sharded import es_generation
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        theta, x, seeds = _policy(pop, dims, 3)
        p0, p1 = split(pop, world, rank)
        r = es_generation(theta, dims, x[p0:p1], seeds, lambda y: y[:, :, 0].sum(-1), 0.05, 0.1,
                          offset=offset, ops=OracleOps())
        q.put((rank, theta.double().numpy(), r["returns"].double().numpy(), r["fitness"].double().numpy()))
    finally:
        dist.destroy_process_group()


def test_sharded_generation_equals_the_oracles_unsharded_generation():
    from oracle import es
    pop, dims, offset, sigma, lr = 7, [5, 9, 3], 77, 0.05, 0.1
    res = _run(2, _oracle_worker, pop, dims, offset)
    theta, x, seeds = _policy(pop, dims, 3)
    shapes = []
    for a, c in zip(dims[:-1], dims[1:]):
        shapes += [(c, a), (c,)]
    offs = es.compute_offsets(shapes)
    th = theta.double().numpy()
    h = x.double().numpy()
    for l in range(len(dims) - 1):
        o = offs[2 * l]
        c, a = shapes[2 * l]
        w = th[o:o + a * c].reshape(c, a)
        b = th[o + a * c:o + a * c + c]
        h = es.perturbed_linear(h, w, b, seeds.numpy(), sigma, offset + o)
        if l < len(dims) - 2:
            h = np.tanh(h)
    returns = h[:, :, 0].sum(-1)
    fit = es.centered_ranks(returns.astype(np.float32))
    grad = es.bias_gradient(fit, seeds.numpy(), (th.size,), sigma, pop, offset)
    want = es.es_update(theta.numpy(), grad, lr)
    for rank, th_r, ret_r, fit_r in res:
        assert np.allclose(ret_r, returns.astype(np.float32), rtol=0, atol=1e-6)
        assert np.array_equal(fit_r, fit)
        # the ranks' parameter ranges were updated in float64 and gathered as float32
        assert np.allclose(th_r, want.astype(np.float32), rtol=0, atol=1e-6)


def test_without_a_process_group_the_generation_runs_on_one_rank():
    from virtual_noise_perturbed_gb300.sharded import es_generation
    assert not dist.is_initialized()
    ops = RecordingOps()
    theta = torch.arange(12, dtype=torch.float32)
    r = es_generation(theta, [3, 3], torch.zeros(4, 1, 3), torch.arange(4), lambda y: y[:, 0, 0], 0.1, 1.0,
                      activation=None, ops=ops)
    assert r["range"] == (0, 12) and r["individuals"] == (0, 4)
    assert theta.tolist() == [2.0 * e + 12.0 for e in range(12)]    # e + (0 + e) + sum(2 * seeds)
    assert [c[0] for c in ops.calls] == ["forward", "ranks", "grad"]
