"""GPU parity of the noise dump, the gradient estimates and the reduction metric
against the CPU oracle (bit-exact noise; gradients within 1e-4 of the RMS)."""

import numpy as np
import pytest
import torch

from oracle import es
from tests.parity import TOL_FP32, assert_close, to_np
from virtual_noise_perturbed_gb300 import (VNError, compute_offsets, gradient_update, noise_dump,
                                           virtual_bias_gradient, virtual_flat_gradient,
                                           virtual_reduce_metric, virtual_weight_gradient, workloads)
from virtual_noise_perturbed_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
M64 = (1 << 64) - 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


SEEDS = np.array([0, 1, -1, 7, -(2 ** 63), 2 ** 63 - 1, 123456789012345, -987654321], dtype=np.int64)


@pytest.mark.parametrize("n", [1, 3, 4, 1023, 4096, 4099, 12345])
@pytest.mark.parametrize("offset", [0, 123456789, (1 << 32) - 5, M64 - 100])
def test_dump_bit_exact(n, offset):
    got = noise_dump(torch.from_numpy(SEEDS).to(DEV), n, offset).cpu().numpy()
    want = es.noise_dump(SEEDS, n, offset)
    assert got.dtype == np.float32 and np.array_equal(got, want)


def test_dump_int32_seeds_and_unaligned_output():
    s32 = torch.tensor([-3, 5, 2 ** 31 - 1], dtype=torch.int32, device=DEV)
    got = noise_dump(s32, 77, 9).cpu().numpy()
    assert np.array_equal(got, es.noise_dump(np.array([-3, 5, 2 ** 31 - 1]), 77, 9))
    # a row length that is not a multiple of 4 takes the scalar-store path
    buf = torch.empty(3 * 77 + 1, dtype=torch.float32, device=DEV)
    from virtual_noise_perturbed_gb300 import _lib
    import ctypes
    lib = _lib.load()
    seeds = torch.tensor([-3, 5, 2 ** 31 - 1], dtype=torch.int64, device=DEV)
    st = lib.vn_noise_dump(ctypes.c_void_p(seeds.data_ptr()), 3, 77, 9,
                           ctypes.c_void_p(buf.data_ptr() + 4), ctypes.c_void_p(0))
    assert st == 0
    torch.cuda.synchronize()
    assert np.array_equal(buf[1:].cpu().numpy().reshape(3, 77), got)


def test_dump_large_windows_and_identity():
    """A 64 x 2^20 dump (256 MB, many CTA chunks): windows anchored at both ends
    match the oracle; the window identity holds at full size."""
    seeds = torch.arange(64, dtype=torch.int64, device=DEV) * 7919 - 3
    n, off = (1 << 20) + 3, (1 << 32) - 1000
    d = noise_dump(seeds, n, off)
    s_np = seeds.cpu().numpy()
    for rows, t0, t1 in [([0, 1], 0, 5000), ([31, 63], n - 5000, n), ([63], 1 << 19, (1 << 19) + 4097)]:
        want = es.noise_dump(s_np[rows], t1 - t0, off + t0)
        assert np.array_equal(d[rows, t0:t1].cpu().numpy(), want)
    t0, t1 = 100001, 600003
    assert torch.equal(d[:, t0:t1], noise_dump(seeds, t1 - t0, off + t0))


def test_dump_workload_index_ranges():
    """The element ranges the five workloads regenerate, windowed at their ends."""
    for number in (1, 2, 3, 4, 5):
        w = workloads.make(number)
        total = sum(l.out_f * l.in_f + l.out_f for l in w.layers)
        first = w.layers[0].offset
        seeds = w.seeds[[0, w.pop // 2, w.pop - 1]]
        for t0 in (0, max(0, total - 4096)):
            got = noise_dump(seeds.to(DEV), min(4096, total), first + t0).cpu().numpy()
            assert np.array_equal(got, es.noise_dump(seeds.numpy(), min(4096, total), first + t0))


def _grad_case(pop, out_f, in_f, sigma, offset, seed_base=0, rows=None):
    g = torch.Generator().manual_seed(pop * 31 + out_f)
    f = torch.randn(pop, generator=g)
    seeds = torch.arange(pop, dtype=torch.int64) * 3 + seed_base
    got = virtual_weight_gradient(f.to(DEV), seeds.to(DEV), (out_f, in_f), sigma, pop, offset)
    want = es.weight_gradient(f.numpy(), seeds.numpy(), (out_f, in_f), sigma, pop, offset, rows=rows)
    got = to_np(got) if rows is None else to_np(got)[rows]
    return assert_close(got, want, TOL_FP32, f"grad pop={pop} {out_f}x{in_f}")


@pytest.mark.parametrize("pop,out_f,in_f", [(1, 1, 1), (8, 16, 32), (37, 5, 301), (300, 64, 65),
                                            (1024, 8, 256), (2000, 33, 100), (4096, 17, 1024)])
def test_weight_gradient_matches_oracle(pop, out_f, in_f):
    _grad_case(pop, out_f, in_f, 0.02, 987654, seed_base=-5)


def test_weight_gradient_one_hot_recovers_noise_exactly():
    pop, sigma, out_f, in_f, off = 8, 2.0 ** -7, 13, 77, (1 << 32) - 20
    seeds = torch.arange(1, pop + 1, dtype=torch.int64, device=DEV)
    dump = es.noise_dump(np.arange(1, pop + 1), out_f * in_f, off)
    for m in range(pop):
        f = torch.zeros(pop, device=DEV)
        f[m] = pop * sigma
        g = virtual_weight_gradient(f, seeds, (out_f, in_f), sigma, pop, off).cpu().numpy()
        assert np.array_equal(g, dump[m].reshape(out_f, in_f))


def test_gradient_cluster_split_is_deterministic_and_matches():
    # 2048 elements, pop 1024: the population is split over an 8-CTA cluster.
    d = _grad_case(1024, 8, 256, 0.02, 82432)
    assert d <= TOL_FP32
    f = torch.randn(1024, device=DEV)
    s = torch.arange(1024, device=DEV)
    a = virtual_weight_gradient(f, s, (8, 256), 0.02, 1024, 5)
    b = virtual_weight_gradient(f, s, (8, 256), 0.02, 1024, 5)
    assert torch.equal(a, b)


def test_bias_gradient_matches_oracle_and_forward_offset():
    pop, out_f, in_f, sigma, off = 512, 300, 7, 0.05, 1000
    g = torch.Generator().manual_seed(5)
    f = torch.randn(pop, generator=g)
    seeds = torch.arange(pop, dtype=torch.int64) - 100
    got = virtual_bias_gradient(f.to(DEV), seeds.to(DEV), (out_f,), sigma, pop, off + out_f * in_f)
    want = es.bias_gradient(f.numpy(), seeds.numpy(), (out_f,), sigma, pop, off + out_f * in_f)
    assert_close(to_np(got), want, TOL_FP32, "bias grad")


def test_workload1_gradients():
    w = workloads.make(1)
    l = w.layers[0]
    gw = virtual_weight_gradient(w.fitness.to(DEV), w.seeds.to(DEV), (l.out_f, l.in_f), w.sigma, w.pop, l.offset)
    gb = virtual_bias_gradient(w.fitness.to(DEV), w.seeds.to(DEV), (l.out_f,), w.sigma, w.pop,
                               l.offset + l.out_f * l.in_f)
    assert_close(to_np(gw), es.weight_gradient(w.fitness.numpy(), w.seeds.numpy(), (l.out_f, l.in_f),
                                               w.sigma, w.pop, l.offset), TOL_FP32, "w1 grad_W")
    assert_close(to_np(gb), es.bias_gradient(w.fitness.numpy(), w.seeds.numpy(), (l.out_f,), w.sigma,
                                             w.pop, l.offset + l.out_f * l.in_f), TOL_FP32, "w1 grad_b")


def test_workload2_all_gradients():
    w = workloads.make(2)
    f, s = w.fitness.numpy(), w.seeds.numpy()
    for l in w.layers:
        gw = virtual_weight_gradient(w.fitness.to(DEV), w.seeds.to(DEV), (l.out_f, l.in_f), w.sigma,
                                     w.pop, l.offset)
        gb = virtual_bias_gradient(w.fitness.to(DEV), w.seeds.to(DEV), (l.out_f,), w.sigma, w.pop,
                                   l.offset + l.out_f * l.in_f)
        assert_close(to_np(gw), es.weight_gradient(f, s, (l.out_f, l.in_f), w.sigma, w.pop, l.offset),
                     TOL_FP32, "w2 grad_W")
        assert_close(to_np(gb), es.bias_gradient(f, s, (l.out_f,), w.sigma, w.pop,
                                                 l.offset + l.out_f * l.in_f), TOL_FP32, "w2 grad_b")


def test_flat_gradient_covers_every_block():
    """One flat reduction over the ES MLP's parameter vector equals the per-block
    oracle gradients, block by block (the layout of compute_offsets)."""
    w = workloads.make(2)
    shapes = []
    for l in w.layers:
        shapes += [(l.out_f, l.in_f), (l.out_f,)]
    offs = es.compute_offsets(shapes)
    assert compute_offsets(shapes) == offs
    n = offs[-1] + shapes[-1][0]
    flat = to_np(virtual_flat_gradient(w.fitness.to(DEV), w.seeds.to(DEV), n, w.sigma, w.pop, 0))
    f, s = w.fitness.numpy(), w.seeds.numpy()
    for (shape, off) in zip(shapes, offs):
        size = int(np.prod(shape))
        if len(shape) == 2:
            want = es.weight_gradient(f, s, shape, w.sigma, w.pop, off).ravel()
        else:
            want = es.bias_gradient(f, s, shape, w.sigma, w.pop, off)
        assert_close(flat[off:off + size], want, TOL_FP32, f"flat block at {off}")


def test_workload3_gradient_windows():
    w = workloads.make(3)
    l = w.layers[0]
    gw = virtual_weight_gradient(w.fitness.to(DEV), w.seeds.to(DEV), (l.out_f, l.in_f), w.sigma, w.pop, l.offset)
    rows = [0, 1, 511, 1023]
    want = es.weight_gradient(w.fitness.numpy(), w.seeds.numpy(), (l.out_f, l.in_f), w.sigma, w.pop,
                              l.offset, rows=rows)
    assert_close(to_np(gw)[rows], want, TOL_FP32, "w3 grad_W rows")


def test_workload4_full_size_windows():
    """4096 x 4096 over pop 16384, in the launch configuration the bench times:
    rows anchored at both ends against the oracle, the bias gradient in full,
    and the row-slice identity grad_W[r0:r1] == grad_W(offset + r0*in, r1 - r0 rows)."""
    w = workloads.make(4)
    l = w.layers[0]
    fit, seeds = w.fitness.to(DEV), w.seeds.to(DEV)
    gw = virtual_weight_gradient(fit, seeds, (l.out_f, l.in_f), w.sigma, w.pop, l.offset)
    rows = [0, l.out_f - 1]
    want = es.weight_gradient(w.fitness.numpy(), w.seeds.numpy(), (l.out_f, l.in_f), w.sigma, w.pop,
                              l.offset, rows=rows)
    assert_close(to_np(gw)[rows], want, TOL_FP32, "w4 grad_W rows")
    boff = l.offset + l.out_f * l.in_f
    assert boff == 140234005
    gb = virtual_bias_gradient(fit, seeds, (l.out_f,), w.sigma, w.pop, boff)
    assert_close(to_np(gb), es.bias_gradient(w.fitness.numpy(), w.seeds.numpy(), (l.out_f,), w.sigma,
                                             w.pop, boff), TOL_FP32, "w4 grad_b")
    r0, r1 = 2000, 2100
    part = virtual_weight_gradient(fit, seeds, (r1 - r0, l.in_f), w.sigma, w.pop, l.offset + r0 * l.in_f)
    assert torch.allclose(part, gw[r0:r1], rtol=0, atol=1e-5 * float(gw.abs().max()))


@pytest.mark.parametrize("pop,n", [(1, 1), (5, 1000), (300, 4099), (16, 1 << 16), (2, 300001),
                                   (8, 1 << 20), (1500, 1 << 16)])
def test_reduce_metric_matches_oracle(pop, n):
    """Sizes on every launch shape: one CTA per individual, an individual split
    over a cluster of 2 to 8 CTAs when the population is small, and (1500
    individuals) halves of individuals when whole ones would leave the last
    round of CTAs mostly idle."""
    g = torch.Generator().manual_seed(n)
    c = torch.randn(n, generator=g)
    seeds = torch.arange(pop, dtype=torch.int64) * 11 - 4
    got = virtual_reduce_metric(c.to(DEV), seeds.to(DEV), 0.3, n, 77)
    want = es.reduce_metric(c.numpy(), seeds.numpy(), 0.3, n, 77)
    assert_close(to_np(got), want, TOL_FP32, "reduce metric")


def test_invalid_calls_raise():
    s = torch.arange(4, device=DEV)
    with pytest.raises(VNError):
        virtual_weight_gradient(torch.ones(4, device=DEV), s, (2, 2), 0.0, 4, 0)
    with pytest.raises(ValueError):
        virtual_weight_gradient(torch.ones(3, device=DEV), s, (2, 2), 0.1, 4, 0)
    with pytest.raises(ValueError):
        noise_dump(torch.arange(4), 3, 0)  # CPU tensor: no CPU path exists


def test_output_buffers_are_written_in_place():
    """``out=``: the result lands in the caller's buffer (NaN-filled first), which is
    returned, with the bits a fresh call gives; a buffer of the wrong shape is refused."""
    g = torch.Generator().manual_seed(21)
    pop, n, sigma, off = 37, 1003, 0.03, 12345
    seeds = (torch.arange(pop, dtype=torch.int64) * 7 - 3).to(DEV)
    fit = torch.randn(pop, generator=g).to(DEV)
    center = torch.randn(n, generator=g).to(DEV)

    def into(fn, shape, *args, **kw):
        want = fn(*args, **kw)
        buf = torch.full(shape, float("nan"), device=DEV)
        got = fn(*args, out=buf, **kw)
        assert got is buf and torch.equal(got, want), fn.__name__

    into(noise_dump, (pop, n), seeds, n, off)
    into(noise_dump, (pop, n), seeds, n, off, noise="gaussian")
    into(virtual_weight_gradient, (17, 59), fit, seeds, (17, 59), sigma, pop, off)
    into(virtual_bias_gradient, (17,), fit, seeds, (17,), sigma, pop, off)
    into(virtual_flat_gradient, (n,), fit, seeds, n, sigma, pop, off)
    into(virtual_reduce_metric, (pop,), center, seeds, sigma, n, off)

    theta0 = torch.randn(n, generator=g).to(DEV)
    theta_a, theta_b = theta0.clone(), theta0.clone()
    grad_a = gradient_update(fit, seeds, theta_a, sigma, pop, 0.1, off)
    buf = torch.full((n,), float("nan"), device=DEV)
    grad_b = gradient_update(fit, seeds, theta_b, sigma, pop, 0.1, off, out=buf)
    assert grad_b is buf and torch.equal(grad_a, grad_b) and torch.equal(theta_a, theta_b)

    with pytest.raises(ValueError):
        noise_dump(seeds, n, off, out=torch.empty(pop, n + 1, device=DEV))
    with pytest.raises(ValueError):
        virtual_flat_gradient(fit, seeds, n, sigma, pop, off, out=torch.empty(n, dtype=torch.float64, device=DEV))
