"""GPU parity of the Gaussian-noise variant (Box-Muller on the finalizer's two halves).

The GPU evaluates log2, cos and sqrt with the hardware approximations; their error
bounds (absolute 2^-22 for log2 on [1/2, 2], 2^-21.4 for cos on [-pi, pi]) give
|G_gpu - G| <= sqrt(2 ln 2 * 2^-22) ~ 6e-4 where u1 is within ~2^-12 of 1 (G near 0)
and ~1e-6 elsewhere; the tests use 1e-3 for the maximum and 2e-6 for the mean. The
gradient keeps the usual 1e-4 of the oracle's RMS. The uniform kind through the same
entry points is bit-identical to the plain entry points."""

import numpy as np
import pytest
import torch

from oracle import es
from tests.parity import TOL_FP32, assert_close, to_np
from virtual_noise_perturbed_gb300 import (VNError, noise_dump,
                                           virtual_bias_gradient, virtual_flat_gradient,
                                           virtual_perturbed_mlp)
from virtual_noise_perturbed_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("pop,n,offset", [(1, 3, 0), (4, 4099, 2 ** 32 - 5), (64, 12345, 2 ** 64 - 101),
                                          (3, 8192 * 2 + 1, 7)])
def test_gaussian_dump_within_the_error_bound(pop, n, offset):
    seeds = torch.arange(pop, dtype=torch.int64) * 7 - 3
    got = noise_dump(seeds.to(DEV), n, offset, noise="gaussian").cpu().numpy().astype(np.float64)
    want = es.gaussian_dump(seeds.numpy(), n, offset)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got))
    assert err.max() <= 1e-3, err.max()
    assert err.mean() <= 2e-6, err.mean()


def test_uniform_kind_is_the_plain_dump():
    seeds = torch.arange(5, dtype=torch.int64, device=DEV)
    a = noise_dump(seeds, 9999, 11)
    b = noise_dump(seeds, 9999, 11, noise="uniform")
    assert torch.equal(a, b)
    with pytest.raises(ValueError):
        noise_dump(seeds, 10, 0, noise="cauchy")


@pytest.mark.parametrize("pop,n", [(8, 1000), (1024, 3000), (4096, 256), (3, 70001)])
def test_gaussian_gradient_matches_oracle(pop, n):
    g = torch.Generator().manual_seed(pop + n)
    f = torch.randn(pop, generator=g)
    seeds = torch.arange(pop, dtype=torch.int64) + 100
    got = virtual_flat_gradient(f.to(DEV), seeds.to(DEV), n, 0.02, pop, 555, noise="gaussian")
    want = es.gaussian_flat_gradient(f.numpy(), seeds.numpy(), n, 0.02, pop, 555)
    assert_close(to_np(got), want, TOL_FP32, f"gaussian gradient pop {pop} n {n}")


def test_gaussian_gradient_one_hot_recovers_the_dump():
    pop, n, sigma = 8, 777, 2.0 ** -7
    seeds = torch.arange(pop, dtype=torch.int64, device=DEV) * 3
    d = noise_dump(seeds, n, 99, noise="gaussian")
    for m in (0, 5):
        f = torch.zeros(pop, device=DEV)
        f[m] = pop * sigma
        got = virtual_flat_gradient(f, seeds, n, sigma, pop, 99, noise="gaussian")
        assert torch.equal(got, d[m])


def test_uniform_kind_is_the_plain_gradient():
    g = torch.Generator().manual_seed(3)
    f = torch.randn(300, generator=g).to(DEV)
    seeds = torch.arange(300, dtype=torch.int64, device=DEV)
    a = virtual_bias_gradient(f, seeds, (5000,), 0.01, 300, 42)
    b = virtual_flat_gradient(f, seeds, 5000, 0.01, 300, 42, noise="uniform")
    assert torch.equal(a, b)


def test_unknown_kind_is_refused_by_the_library():
    from virtual_noise_perturbed_gb300 import _lib
    lib = _lib.load()
    P = __import__("ctypes").c_void_p
    assert lib.vn_noise_dump_ex(P(0x1000), 1, 4, 0, 7, P(0x1000), P(0)) == 4
    assert lib.vn_gradient_ex(P(0x1000), P(0x1000), 1, 4, 0.1, 0, 2, P(0x1000), P(0)) == 4
    with pytest.raises(VNError):
        virtual_flat_gradient(torch.ones(2, device=DEV), torch.arange(2, device=DEV), 4, 0.0, 2)


def _chain_case(dims, pop, batch, seed):
    g = torch.Generator().manual_seed(seed)
    ws = [torch.randn((c, a), generator=g) / a ** 0.5 for a, c in zip(dims[:-1], dims[1:])]
    bs = [torch.randn(c, generator=g) * 0.1 for c in dims[1:]]
    x = torch.randn((pop, batch, dims[0]), generator=g)
    seeds = torch.arange(pop, dtype=torch.int64) * 3 + 1
    shapes = []
    for a, c in zip(dims[:-1], dims[1:]):
        shapes += [(c, a), (c,)]
    return x, ws, bs, seeds, es.compute_offsets(shapes)[0::2]


@pytest.mark.parametrize("dims,pop,batch", [([64, 256, 256, 8], 5, 1), ([13, 37, 5], 11, 3),
                                            ([32, 64, 16], 7, 8), ([40, 24], 300, 2)])
def test_gaussian_forward_chain_matches_oracle(dims, pop, batch):
    """The policy forward with Gaussian-variant noise (vn_perturbed_mlp_ex) against the
    oracle's layer-by-layer chain with the same noise: within 1e-4 of the output RMS
    (the approximations' error, at most 6e-4 on a rare element, is scaled by sigma)."""
    x, ws, bs, seeds, offs = _chain_case(dims, pop, batch, len(dims) + pop)
    sigma = 0.05
    y = virtual_perturbed_mlp(x.to(DEV), [w.to(DEV) for w in ws], [b.to(DEV) for b in bs],
                              seeds.to(DEV), sigma, offs, activation="tanh", noise="gaussian")
    h = x.numpy().astype(np.float64)
    for l, (w, b) in enumerate(zip(ws, bs)):
        h = es.perturbed_linear(h, w.numpy(), b.numpy(), seeds.numpy(), sigma, offs[l], noise="gaussian")
        if l + 1 < len(ws):
            h = np.tanh(h)
    assert_close(to_np(y), h, TOL_FP32, f"gaussian chain {dims}")


def test_gaussian_forward_one_hot_reads_the_dump_bit_for_bit():
    """X rows e_k, W = 0, sigma = 1, no bias: Y[i, k, j] is the GPU's own Gaussian dump
    at offset + j*in + k, bit for bit (same noise, same scaling, no other arithmetic)."""
    pop, in_f, out_f, off = 6, 8, 40, 2 ** 40 + 3
    x = torch.eye(in_f).repeat(pop, 1, 1)
    seeds = torch.arange(pop, dtype=torch.int64) - 2
    y = virtual_perturbed_mlp(x.to(DEV), [torch.zeros(out_f, in_f, device=DEV)], None, seeds.to(DEV),
                              1.0, [off], activation=None, noise="gaussian").cpu()
    d = noise_dump(seeds.to(DEV), out_f * in_f, off, noise="gaussian").cpu().view(pop, out_f, in_f)
    assert torch.equal(y, d.transpose(1, 2))


def test_gaussian_forward_uniform_kind_is_the_plain_chain():
    x, ws, bs, seeds, offs = _chain_case([24, 48, 6], 9, 2, 5)
    args = (x.to(DEV), [w.to(DEV) for w in ws], [b.to(DEV) for b in bs], seeds.to(DEV), 0.1, offs)
    a = virtual_perturbed_mlp(*args, noise="uniform")
    g = virtual_perturbed_mlp(*args, noise="gaussian")
    assert not torch.equal(a, g)
    with pytest.raises(ValueError):
        virtual_perturbed_mlp(*args, noise="cauchy")


def test_gaussian_policy_workload_full_size_sampled():
    """The ES policy workload at full size (pop 1024) in its one-launch Gaussian forward,
    against the oracle's Gaussian chain on individuals anchored at both ends plus a
    seeded sample."""
    from virtual_noise_perturbed_gb300 import workloads
    w = workloads.make(2)
    ws = [l.weight for l in w.layers]
    bs = [l.bias for l in w.layers]
    offs = [l.offset for l in w.layers]
    y = virtual_perturbed_mlp(w.x.to(DEV), [t.to(DEV) for t in ws], [t.to(DEV) for t in bs],
                              w.seeds.to(DEV), w.sigma, offs, activation="tanh", noise="gaussian")
    rng = np.random.default_rng(2)
    inds = sorted({0, 1, w.pop - 2, w.pop - 1} | set(rng.choice(w.pop, 8, replace=False).tolist()))
    h = w.x.numpy()[inds].astype(np.float64)
    seeds = w.seeds.numpy()[inds]
    for l, (wt, bt) in enumerate(zip(ws, bs)):
        h = es.perturbed_linear(h, wt.numpy(), bt.numpy(), seeds, w.sigma, offs[l], noise="gaussian")
        if l + 1 < len(ws):
            h = np.tanh(h)
    assert_close(to_np(y)[inds], h, TOL_FP32, "gaussian policy workload")


def _linear_case(pop, batch, in_f, out_f, xdt, wdt, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((pop, batch, in_f), generator=g).to(xdt)
    w = (torch.randn((out_f, in_f), generator=g) / in_f ** 0.5).to(wdt)
    b = (torch.randn(out_f, generator=g) * 0.1).to(wdt)
    seeds = torch.arange(pop, dtype=torch.int64) * 5 + 2
    return x, w, b, seeds


@pytest.mark.parametrize("pop,batch,in_f,out_f,wdt", [(3, 40, 128, 200, torch.bfloat16),
                                                      (2, 256, 512, 130, torch.bfloat16),
                                                      (5, 32, 64, 128, torch.float32)])
def test_gaussian_tensor_core_forward_matches_oracle(pop, batch, in_f, out_f, wdt):
    """The tensor-core forward with the Gaussian kind against the oracle's float64
    forward with the same noise, within the bf16 path's 2e-2 of the output RMS."""
    from virtual_noise_perturbed_gb300 import virtual_perturbed_linear
    from tests.parity import TOL_BF16
    x, w, b, seeds = _linear_case(pop, batch, in_f, out_f, torch.bfloat16, wdt, in_f + pop)
    y = virtual_perturbed_linear(x.to(DEV), w.to(DEV), b.to(DEV), seeds.to(DEV), 0.05, 321, path="tc",
                                 noise="gaussian")
    want = es.perturbed_linear(x.float().numpy(), w.float().numpy(), b.float().numpy(), seeds.numpy(),
                               0.05, 321, noise="gaussian")
    assert_close(to_np(y), want, TOL_BF16, "gaussian tc forward")


def test_gaussian_tensor_core_one_hot_reads_the_bf16_dump():
    """X rows e_k (bf16), W = 0, sigma = 1, no bias: Y[i, k, j] = bf16 of the GPU's Gaussian
    dump at offset + j*in + k, bit for bit (pins the Gaussian unit inside the swizzled tile)."""
    from virtual_noise_perturbed_gb300 import virtual_perturbed_linear
    pop, in_f, out_f, off = 2, 32, 136, 77
    x = torch.eye(in_f, dtype=torch.bfloat16).repeat(pop, 1, 1)
    seeds = torch.tensor([9, -9], dtype=torch.int64)
    y = virtual_perturbed_linear(x.to(DEV), torch.zeros(out_f, in_f, dtype=torch.bfloat16, device=DEV),
                                 None, seeds.to(DEV), 1.0, off, path="tc", noise="gaussian").cpu()
    d = noise_dump(seeds.to(DEV), out_f * in_f, off, noise="gaussian").cpu().view(pop, out_f, in_f)
    assert torch.equal(y, d.transpose(1, 2).to(torch.bfloat16))


def test_gaussian_single_layer_cuda_core_forward():
    """fp32 W, batch <= 8: the Gaussian single layer runs on the chain kernel whatever
    the population (here 6 individuals, forced "ffma" and automatic), against the
    oracle; a Gaussian call only the single-layer kernel could run is refused."""
    from virtual_noise_perturbed_gb300 import virtual_perturbed_linear
    x, w, b, seeds = _linear_case(6, 3, 70, 33, torch.float32, torch.float32, 4)
    want = es.perturbed_linear(x.numpy(), w.numpy(), b.numpy(), seeds.numpy(), 0.1, 55, noise="gaussian")
    for path in ("auto", "ffma"):
        y = virtual_perturbed_linear(x.to(DEV), w.to(DEV), b.to(DEV), seeds.to(DEV), 0.1, 55, path=path,
                                     noise="gaussian")
        assert_close(to_np(y), want, TOL_FP32, f"gaussian single layer {path}")
    with pytest.raises(VNError):
        virtual_perturbed_linear(x.to(DEV), w.to(DEV).to(torch.bfloat16), b.to(DEV), seeds.to(DEV), 0.1, 55,
                                 noise="gaussian")
