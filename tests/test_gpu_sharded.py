"""The population-sharded ES generation with the library's kernels: two processes
on the one GPU, the exchanges as gloo collectives between launches (no kernel
of one process waits on the other's).

Rank r runs the forward of its individuals, the returns are all-gathered, every
rank ranks them, rank r computes the gradient and update of its range of the
flat parameter vector at offset + e0, and the ranges are all-gathered. Checked:
both ranks end with the same parameters; the update equals the oracle's
gradient of the whole population (fitness = the oracle's centered ranks of the
gathered returns) within the fp32 tolerance; the returns equal the oracle's
forward of the policy."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tests.parity import TOL_FP32, assert_close

pytestmark = pytest.mark.gpu

POP, DIMS, SIGMA, LR, OFFSET = 96, [64, 256, 256, 8], 0.02, 0.5, 4321


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _policy():
    g = torch.Generator().manual_seed(9)
    n = sum(a * c + c for a, c in zip(DIMS[:-1], DIMS[1:]))
    theta = torch.randn(n, generator=g) * 0.1
    x = torch.randn(POP, 1, DIMS[0], generator=g)
    seeds = torch.arange(POP, dtype=torch.int64) * 11 + 5
    return theta, x, seeds


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from virtual_noise_perturbed_gb300 import device_status
    from virtual_noise_perturbed_gb300.sharded import es_generation, split
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        theta, x, seeds = _policy()
        p0, p1 = split(POP, world, rank)
        th = theta.cuda()
        r = es_generation(th, DIMS, x[p0:p1].cuda(), seeds.cuda(), lambda y: y[:, 0, :].sum(-1),
                          SIGMA, LR, offset=OFFSET)
        device_status()
        q.put((rank, th.cpu().numpy(), r["returns"].cpu().numpy(), r["fitness"].cpu().numpy()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_on_one_gpu_match_the_oracle():
    from oracle import es
    from virtual_noise_perturbed_gb300.build import build
    build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=300) for _ in procs], key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, th0, ret0, fit0), (_, th1, ret1, fit1) = res
    assert np.array_equal(th0, th1) and np.array_equal(ret0, ret1) and np.array_equal(fit0, fit1)

    theta, x, seeds = _policy()
    shapes = []
    for a, c in zip(DIMS[:-1], DIMS[1:]):
        shapes += [(c, a), (c,)]
    offs = es.compute_offsets(shapes)
    th = theta.double().numpy()
    h = x.double().numpy()
    for l in range(len(DIMS) - 1):
        o = offs[2 * l]
        c, a = shapes[2 * l]
        h = es.perturbed_linear(h, th[o:o + a * c].reshape(c, a), th[o + a * c:o + a * c + c],
                                seeds.numpy(), SIGMA, OFFSET + o)
        if l < len(DIMS) - 2:
            h = np.tanh(h)
    assert_close(ret0, h[:, 0, :].sum(-1), TOL_FP32, "returns")
    fit = es.centered_ranks(ret0)
    assert np.array_equal(fit0, fit)
    grad = es.bias_gradient(fit, seeds.numpy(), (th.size,), SIGMA, POP, OFFSET)
    got = (th0.astype(np.float64) - theta.numpy().astype(np.float64)) / float(np.float32(LR))
    # theta + lr*grad is rounded to float32: allow that rounding beside the tolerance
    slack = np.max(np.abs(theta.numpy())) * 2.0 ** -23 / float(np.float32(LR))
    rms = np.sqrt(np.mean(grad ** 2))
    assert np.max(np.abs(got - grad)) <= TOL_FP32 * rms + slack
