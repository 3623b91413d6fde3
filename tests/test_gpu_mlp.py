"""GPU parity of the one-launch perturbed policy (vn_perturbed_mlp) against the CPU oracle.

The oracle side chains the oracle's perturbed linear layer by layer (float64,
noise materialised) with numpy's tanh between layers; the kernel keeps the
activations on chip. fp32 arithmetic: within 1e-4 of the oracle's RMS. A
one-layer one-hot case recovers the noise bit for bit."""

import numpy as np
import pytest
import torch

from oracle import es, splitmix
from tests.parity import TOL_FP32, assert_close, to_np
from virtual_noise_perturbed_gb300 import (VNError, compute_offsets, virtual_perturbed_linear,
                                           virtual_perturbed_mlp, workloads)
from virtual_noise_perturbed_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _layers(dims, seed, bias_mask=None):
    g = torch.Generator().manual_seed(seed)
    ws, bs = [], []
    for l, (a, c) in enumerate(zip(dims[:-1], dims[1:])):
        ws.append(torch.randn((c, a), generator=g) / max(a, 1) ** 0.5)
        has_b = True if bias_mask is None else bias_mask[l]
        bs.append(torch.randn(c, generator=g) * 0.1 if has_b else None)
    return ws, bs


def _offsets(dims):
    """The weight blocks' offsets by the oracle's compute_offsets over (W_0, b_0, W_1, ...)."""
    shapes = []
    for a, c in zip(dims[:-1], dims[1:]):
        shapes += [(c, a), (c,)]
    return es.compute_offsets(shapes)[0::2]


def _oracle_chain(x, ws, bs, seeds, sigma, offsets, act, individuals=None):
    """Layer-by-layer oracle: es.perturbed_linear then tanh (not on the last layer)."""
    s = seeds.numpy()
    h = x.float().numpy().astype(np.float64)
    if individuals is not None:
        s = s[individuals]
        if h.ndim == 3:
            h = h[individuals]
    for l, (w, b) in enumerate(zip(ws, bs)):
        h = es.perturbed_linear(h, w.numpy(), None if b is None else b.numpy(), s, sigma, offsets[l])
        if act == "tanh" and l + 1 < len(ws):
            h = np.tanh(h)
    return h


def _check(dims, pop, batch, *, shared=False, xdt=torch.float32, act="tanh", bias_mask=None,
           sigma=0.03, seed=0, base_offset=0):
    ws, bs = _layers(dims, seed, bias_mask)
    g = torch.Generator().manual_seed(seed + 1)
    x = torch.randn((batch, dims[0]) if shared else (pop, batch, dims[0]), generator=g).to(xdt)
    seeds = torch.arange(pop, dtype=torch.int64) * 3 + 11
    offs = [o + base_offset for o in _offsets(dims)]
    # With no base offset the library lays the blocks out itself (its own
    # compute_offsets, offsets=None); the oracle side uses the oracle's.
    y = virtual_perturbed_mlp(x.to(DEV), [w.to(DEV) for w in ws],
                              [None if b is None else b.to(DEV) for b in bs], seeds.to(DEV), sigma,
                              offs if base_offset else None, activation=act)
    want = _oracle_chain(x, ws, bs, seeds, sigma, offs, act)
    if shared:
        assert want.shape == (pop, batch, dims[-1])
    return assert_close(to_np(y), want, TOL_FP32, f"mlp {dims} pop {pop} batch {batch}")


@pytest.mark.parametrize("dims,pop,batch", [
    ([64, 256, 256, 8], 5, 1),        # the policy's shape, few individuals
    ([13, 37, 5], 11, 3),             # ragged: no dimension a multiple of 8
    ([4, 300, 3], 9, 2),              # one chunk per row (one lane per row), wide hidden layer
    ([16, 24, 32, 40, 48, 56, 64, 72, 8], 6, 1),   # eight layers
    ([32, 64, 16], 7, 8),             # batch 8: one individual per group
    ([40, 520, 33], 3, 4),            # rows longer than 32 chunks (several chunks per lane)
    ([64, 256, 256, 8], 400, 5),      # many groups per CTA
])
def test_mlp_matches_oracle(dims, pop, batch):
    _check(dims, pop, batch)


def test_mlp_shared_x_bf16_x_no_act_partial_biases():
    _check([24, 40, 8], 10, 2, shared=True)
    _check([24, 40, 8], 10, 2, xdt=torch.bfloat16)
    _check([24, 40, 8], 10, 2, act=None)
    _check([24, 40, 40, 8], 10, 2, bias_mask=[False, True, False])
    _check([24, 40, 8], 10, 2, base_offset=(1 << 64) - 5000)   # indices wrap mod 2^64


def test_mlp_sigma_zero_is_a_plain_tanh_network():
    """sigma = 0: the chain is tanh(tanh(x W0^T + b0) W1^T + b1) W2^T + b2, against
    float64 matmuls of the same inputs."""
    dims, pop, batch = [40, 96, 64, 5], 10, 2
    ws, bs = _layers(dims, 3, None)
    x = torch.randn((pop, batch, dims[0]), generator=torch.Generator().manual_seed(4))
    seeds = torch.arange(pop, dtype=torch.int64)
    y = virtual_perturbed_mlp(x.to(DEV), [w.to(DEV) for w in ws], [b.to(DEV) for b in bs],
                              seeds.to(DEV), 0.0, _offsets(dims), activation="tanh")
    h = x.double()
    for li, (w, b) in enumerate(zip(ws, bs)):
        h = h @ w.double().T + b.double()
        if li < len(ws) - 1:
            h = torch.tanh(h)
    assert_close(to_np(y), h.numpy(), TOL_FP32, "mlp sigma 0")


def test_mlp_zero_width_layer_gives_bias_plus_bias_noise():
    # A hidden layer of width 0: the next layer sees in = 0, so its output is
    # b + sigma*nb (the in == 0 case of the single-layer entry point).
    _check([8, 0, 6], 4, 1)


def test_mlp_one_hot_single_layer_is_bit_exact():
    """x rows e_k, W = 0, no bias, sigma = 1: y[i, r, j] = N_i[j, k_r] exactly."""
    pop, in_f, out_f, batch = 6, 40, 24, 4
    ks = [0, 7, 8, 39]
    x = torch.zeros(pop, batch, in_f)
    for r, k in enumerate(ks):
        x[:, r, k] = 1.0
    seeds = torch.tensor([0, 1, -1, 2**62, -2**63, 12345], dtype=torch.int64)
    off = 2**32 - 100
    y = virtual_perturbed_mlp(x.to(DEV), [torch.zeros(out_f, in_f, device=DEV)], None,
                              seeds.to(DEV), 1.0, [off], activation=None).cpu().numpy()
    for i in range(pop):
        n_i = es.weight_noise(int(seeds[i]), out_f, in_f, off).astype(np.float32)
        for r, k in enumerate(ks):
            assert np.array_equal(y[i, r], n_i[:, k])


def test_mlp_matches_per_layer_calls_on_the_policy_workload():
    """The ES MLP policy at full size: the one-launch chain against three
    single-layer calls (fp32 both; summation orders differ), and against the
    oracle on sampled individuals (anchored at both ends plus random ones)."""
    w = workloads.make(2)
    ws = [l.weight.to(DEV) for l in w.layers]
    bs = [l.bias.to(DEV) for l in w.layers]
    offs = [l.offset for l in w.layers]
    y = virtual_perturbed_mlp(w.x.to(DEV), ws, bs, w.seeds.to(DEV), w.sigma, offs, activation="tanh")
    h = w.x.to(DEV)
    for li, l in enumerate(w.layers):
        h = virtual_perturbed_linear(h, ws[li], bs[li], w.seeds.to(DEV), w.sigma, l.offset,
                                     activation="tanh" if li < 2 else None)
    assert_close(to_np(y), to_np(h), TOL_FP32, "mlp vs per-layer")
    rng = np.random.default_rng(2)
    inds = sorted({0, 1, 511, 1022, 1023} | set(rng.choice(np.arange(2, 1022), 11, replace=False).tolist()))
    want = _oracle_chain(w.x, [l.weight for l in w.layers], [l.bias for l in w.layers], w.seeds,
                         w.sigma, offs, "tanh", individuals=inds)
    assert_close(to_np(y)[inds], want, TOL_FP32, "mlp workload 2")


def test_mlp_is_repeatable():
    w = workloads.make(2)
    args = (w.x.to(DEV), [l.weight.to(DEV) for l in w.layers], [l.bias.to(DEV) for l in w.layers],
            w.seeds.to(DEV), w.sigma, [l.offset for l in w.layers])
    y1 = virtual_perturbed_mlp(*args)
    y2 = virtual_perturbed_mlp(*args)
    assert torch.equal(y1, y2)


def test_mlp_refuses_what_it_cannot_run():
    s = torch.arange(3, device=DEV)
    with pytest.raises(VNError, match="SHAPE"):
        virtual_perturbed_mlp(torch.randn(3, 9, 4, device=DEV), [torch.randn(5, 4, device=DEV)], None,
                              s, 0.1)                                   # batch 9 > 8
    with pytest.raises(VNError, match="SHAPE"):
        virtual_perturbed_mlp(torch.randn(3, 8, 4, device=DEV), [torch.randn(40000, 4, device=DEV)],
                              None, s, 0.1)                             # too wide for shared memory
    with pytest.raises(ValueError):
        virtual_perturbed_mlp(torch.randn(3, 1, 4, device=DEV), [torch.randn(5, 4, device=DEV).half()],
                              None, s, 0.1)                             # fp32 weights only
