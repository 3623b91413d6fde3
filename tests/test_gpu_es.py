"""GPU parity of the ES bookkeeping steps (centered ranks, parameter update) and of
one full ES generation of the policy workload, against the CPU oracle.

Ranks are integers turned into floats by one fp32 division and subtraction:
bit-exact. The update is one fp32 fma per element: within one float32 rounding
of the oracle's float64 value."""

import numpy as np
import pytest
import torch

from oracle import es
from tests.parity import TOL_FP32, assert_close, to_np
from virtual_noise_perturbed_gb300 import (VNError, centered_ranks, compute_offsets, es_update,
                                           gradient_update, virtual_flat_gradient,
                                           virtual_perturbed_mlp, workloads)
from virtual_noise_perturbed_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


@pytest.mark.parametrize("pop", [1, 2, 5, 255, 256, 257, 1024, 2047, 2048, 2049, 5000])
def test_centered_ranks_bit_exact(pop):
    rng = np.random.default_rng(pop)
    f = (rng.integers(-50, 50, size=pop) / 8).astype(np.float32)      # many ties
    got = centered_ranks(torch.from_numpy(f).to(DEV)).cpu().numpy()
    assert np.array_equal(got, es.centered_ranks(f))


def test_centered_ranks_special_values():
    f = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-45, -1e-45, 3.0, 3.0],
                 dtype=np.float32)
    got = centered_ranks(torch.from_numpy(f).to(DEV)).cpu().numpy()
    assert np.array_equal(got, es.centered_ranks(f))


@pytest.mark.parametrize("number", [2, 4])
def test_centered_ranks_of_the_workloads_returns(number):
    w = workloads.make(number)
    got = centered_ranks(w.returns.to(DEV)).cpu().numpy()
    assert np.array_equal(got, es.centered_ranks(w.returns.numpy()))


def _check_update(theta, grad, lr):
    want = es.es_update(theta.cpu().numpy(), grad.cpu().numpy(), lr)
    es_update(theta, grad, lr)
    got = theta.cpu().numpy().astype(np.float64)
    # one float32 rounding of the exact value
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -24 + 1e-45)


@pytest.mark.parametrize("n", [1, 3, 4, 1001, 84488, 1 << 20])
def test_es_update(n):
    g = torch.Generator().manual_seed(n)
    _check_update(torch.randn(n, generator=g).to(DEV), torch.randn(n, generator=g).to(DEV), 0.0173)


def test_es_update_unaligned_and_errors():
    g = torch.Generator().manual_seed(5)
    base = torch.randn(1003, generator=g).to(DEV)
    grad = torch.randn(1003, generator=g).to(DEV)
    _check_update(base[1:], grad[:-1], -0.5)          # 4-byte but not 16-byte aligned: scalar path
    with pytest.raises(VNError, match="VALUE"):
        es_update(base, grad, float("nan"))
    with pytest.raises(ValueError):
        es_update(base, grad[:10], 0.1)
    with pytest.raises(VNError, match="VALUE"):
        centered_ranks(base, out=base)                 # in place is refused (the input would change)


def test_one_es_generation_of_the_policy():
    """Forward (one launch), ranks of the returns, flat gradient of all six blocks,
    update of the flat parameter vector: the generation's new parameters against
    the oracle's (exact ranks, float64 gradient)."""
    w = workloads.make(2)
    dims = [w.layers[0].in_f] + [l.out_f for l in w.layers]
    shapes = []
    for a, c in zip(dims[:-1], dims[1:]):
        shapes += [(c, a), (c,)]
    offs = es.compute_offsets(shapes)
    assert compute_offsets(shapes) == offs
    n = offs[-1] + shapes[-1][0]
    theta0 = torch.cat([t.reshape(-1) for l in w.layers for t in (l.weight, l.bias)])
    theta = theta0.to(DEV)
    views = [theta[o:o + int(np.prod(sh))].view(sh) for o, sh in zip(offs, shapes)]
    y = virtual_perturbed_mlp(w.x.to(DEV), views[0::2], views[1::2], w.seeds.to(DEV), w.sigma,
                              offs[0::2], activation="tanh")
    assert y.shape == (w.pop, 1, 8)
    fit = centered_ranks(w.returns.to(DEV))
    grad = virtual_flat_gradient(fit, w.seeds.to(DEV), n, w.sigma, w.pop, 0)
    lr = 0.05
    es_update(theta, grad, lr)
    torch.cuda.synchronize()
    fit_ref = es.centered_ranks(w.returns.numpy())
    assert np.array_equal(fit.cpu().numpy(), fit_ref)
    grad_ref = es.bias_gradient(fit_ref, w.seeds.numpy(), (n,), w.sigma, w.pop, 0)
    assert_close(to_np(grad), grad_ref, TOL_FP32, "generation gradient")
    delta = theta.cpu().numpy().astype(np.float64) - theta0.numpy().astype(np.float64)
    assert_close(delta, float(np.float32(lr)) * grad_ref, TOL_FP32, "generation update")


@pytest.mark.parametrize("n,pop,noise", [(1, 3, "uniform"), (255, 64, "uniform"), (84488, 1024, "uniform"),
                                         (70001, 300, "uniform"), (4096 * 33 + 7, 4096, "uniform"),
                                         (5000, 257, "gaussian")])
def test_gradient_update_matches_the_two_launches(n, pop, noise):
    """The fused estimate + step gives the same bits as vn_gradient_ex followed by
    vn_es_update, for the cluster-split sizes (small n) and the plain ones (large n),
    both noise kinds; and its gradient is the oracle's within the fp32 tolerance."""
    g = torch.Generator().manual_seed(n + pop)
    f = torch.randn(pop, generator=g).to(DEV)
    seeds = (torch.arange(pop, dtype=torch.int64) * 7 - 3).to(DEV)
    theta0 = torch.randn(n, generator=g).to(DEV)
    sigma, lr, off = 0.02, 0.05, 12345
    theta_fused = theta0.clone()
    grad_fused = gradient_update(f, seeds, theta_fused, sigma, pop, lr, off, noise=noise)
    grad_two = virtual_flat_gradient(f, seeds, n, sigma, pop, off, noise=noise)
    theta_two = es_update(theta0.clone(), grad_two, lr)
    torch.cuda.synchronize()
    assert torch.equal(grad_fused, grad_two)
    assert torch.equal(theta_fused, theta_two)
    if noise == "uniform" and n * pop <= 10 ** 7:
        want = es.bias_gradient(f.cpu().numpy(), seeds.cpu().numpy(), (n,), sigma, pop, off)
        assert_close(to_np(grad_fused), want, TOL_FP32, "fused gradient")


def test_gradient_update_refusals():
    theta = torch.zeros(8, device=DEV)
    with pytest.raises(ValueError):
        gradient_update(torch.ones(4, device=DEV), torch.arange(4, device=DEV), theta.double(), 0.1, 4, 0.1)
    with pytest.raises(VNError):
        gradient_update(torch.ones(4, device=DEV), torch.arange(4, device=DEV), theta, 0.1, 4, float("inf"))


def test_adjacent_slices_of_one_buffer():
    """Fitness and theta carved from one allocation back to back (no shared byte), and
    theta and grad likewise: validation accepts them, and the results are the bits that
    separate buffers give. Slices that share bytes are refused before any launch."""
    pop, n, sigma, lr, off = 300, 4099, 0.02, 0.05, 777
    g = torch.Generator().manual_seed(11)
    fit = torch.randn(pop, generator=g)
    theta0 = torch.randn(n, generator=g)
    seeds = torch.arange(pop, dtype=torch.int64).to(DEV)

    buf = torch.cat([fit, theta0]).to(DEV)               # [fitness | theta]
    grad_a = gradient_update(buf[:pop], seeds, buf[pop:], sigma, pop, lr, off)
    theta_b = theta0.to(DEV)
    grad_b = gradient_update(fit.to(DEV), seeds, theta_b, sigma, pop, lr, off)
    assert torch.equal(grad_a, grad_b) and torch.equal(buf[pop:], theta_b)
    assert torch.equal(buf[:pop].cpu(), fit)             # the input is untouched

    buf2 = torch.cat([theta0, grad_b.cpu()]).to(DEV)     # [theta | grad]
    es_update(buf2[:n], buf2[n:], lr)
    theta_c = theta0.to(DEV)
    es_update(theta_c, grad_b, lr)
    assert torch.equal(buf2[:n], theta_c)

    with pytest.raises(VNError, match="VALUE"):
        es_update(buf2[:n], buf2[n - 4:2 * n - 4], lr)   # grad's first 4 floats are theta's last
    with pytest.raises(VNError, match="VALUE"):
        gradient_update(buf[:pop], seeds, buf[pop - 1:pop - 1 + n], sigma, pop, lr, off)
