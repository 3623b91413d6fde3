"""GPU parity of the perturbed linear forward against the CPU oracle.

fp32 (FFMA) path within 1e-4 of the oracle's RMS; bf16 tensor-core path within
2e-2; one-hot inputs recover the noise bit for bit."""

import numpy as np
import pytest
import torch

from oracle import es
from tests.parity import TOL_BF16, TOL_FP32, assert_close, to_np
from virtual_noise_perturbed_gb300 import (VNError, noise_dump, perturbed_linear_path,
                                           virtual_perturbed_linear, workloads)
from virtual_noise_perturbed_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _case(pop, batch, in_f, out_f, *, shared=False, bias=True, xdt=torch.float32, wdt=torch.float32,
          bdt=torch.float32, sigma=0.05, offset=12345, seed=0):
    g = torch.Generator().manual_seed(seed + 17 * pop + batch)
    x = torch.randn((batch, in_f) if shared else (pop, batch, in_f), generator=g).to(xdt)
    w = (torch.randn((out_f, in_f), generator=g) / max(in_f, 1) ** 0.5).to(wdt)
    b = (torch.randn(out_f, generator=g) * 0.1).to(bdt) if bias else None
    seeds = torch.arange(pop, dtype=torch.int64) * 5 - 7
    return x, w, b, seeds, sigma, offset


def _run_and_check(x, w, b, seeds, sigma, offset, tol, path="auto", individuals=None, act=None):
    y = virtual_perturbed_linear(x.to(DEV), w.to(DEV), None if b is None else b.to(DEV),
                                 seeds.to(DEV), sigma, offset, path=path, activation=act)
    want = es.perturbed_linear(x.float().numpy(), w.float().numpy(),
                               None if b is None else b.float().numpy(), seeds.numpy(), sigma,
                               offset, individuals=individuals)
    if act == "tanh":
        want = np.tanh(want)
    got = to_np(y) if individuals is None else to_np(y)[individuals]
    return assert_close(got, want, tol, f"forward {tuple(x.shape)}->{w.shape[0]} {path}")


@pytest.mark.parametrize("pop,batch,in_f,out_f", [
    (1, 1, 1, 1), (8, 4, 32, 16), (9, 1, 64, 256), (13, 3, 67, 33), (3, 8, 200, 5),
    (5, 11, 130, 40), (17, 2, 1, 70), (2, 17, 257, 31)])
def test_ffma_forward_matches_oracle(pop, batch, in_f, out_f):
    _run_and_check(*_case(pop, batch, in_f, out_f), TOL_FP32, path="ffma")


@pytest.mark.parametrize("shared,bias", [(True, True), (True, False), (False, False)])
def test_ffma_forward_shared_x_and_no_bias(shared, bias):
    _run_and_check(*_case(11, 3, 96, 45, shared=shared, bias=bias), TOL_FP32, path="ffma")


@pytest.mark.parametrize("xdt,wdt,bdt", [(torch.bfloat16, torch.float32, torch.float32),
                                         (torch.float32, torch.bfloat16, torch.bfloat16),
                                         (torch.bfloat16, torch.bfloat16, torch.bfloat16)])
def test_ffma_forward_bf16_inputs(xdt, wdt, bdt):
    x, w, b, s, sig, off = _case(10, 2, 80, 50, xdt=xdt, wdt=wdt, bdt=bdt)
    tol = TOL_BF16 if (xdt == torch.bfloat16 and wdt == torch.bfloat16) else TOL_FP32
    _run_and_check(x, w, b, s, sig, off, tol, path="ffma")


def test_ffma_forward_tanh_epilogue():
    _run_and_check(*_case(12, 2, 64, 48), TOL_FP32, path="ffma", act="tanh")


def test_forward_in_zero_is_bias_plus_bias_noise():
    pop, out_f, off = 6, 9, 4242
    b = torch.randn(out_f)
    seeds = torch.arange(pop, dtype=torch.int64)
    y = virtual_perturbed_linear(torch.empty((pop, 2, 0), device=DEV), torch.empty((out_f, 0), device=DEV),
                                 b.to(DEV), seeds.to(DEV), 0.5, off, path="ffma")
    nb = es.noise_dump(seeds.numpy(), out_f, off).astype(np.float64)
    want = b.numpy().astype(np.float64)[None, None, :] + 0.5 * nb[:, None, :]
    assert_close(to_np(y), np.broadcast_to(want, (pop, 2, out_f)), TOL_FP32, "in=0")


@pytest.mark.parametrize("path,pop,batch,xdt,wdt", [
    ("ffma", 9, 3, torch.float32, torch.float32), ("auto", 200, 2, torch.float32, torch.float32),
    ("tc", 5, 40, torch.bfloat16, torch.float32), ("tc", 3, 33, torch.bfloat16, torch.bfloat16)])
def test_sigma_zero_is_a_plain_linear_layer(path, pop, batch, xdt, wdt):
    """sigma = 0 removes the noise: Y[i] = X[i] W^T + b on every path, against a
    float64 matmul of the same (bf16-rounded where the path takes bf16) inputs."""
    x, w, b, seeds, _, off = _case(pop, batch, 72, 150, xdt=xdt, wdt=wdt, bdt=wdt)
    y = virtual_perturbed_linear(x.to(DEV), w.to(DEV), b.to(DEV), seeds.to(DEV), 0.0, off, path=path)
    want = (x.double() @ w.double().T + b.double()).numpy()
    tol = TOL_BF16 if path == "tc" else TOL_FP32
    assert_close(to_np(y), want, tol, f"sigma 0 {path}")


@pytest.mark.parametrize("path", ["ffma"])
def test_forward_one_hot_is_bit_exact(path):
    """X rows = e_k, W = 0, b = 0, sigma = 1: Y[i, k, :] = N_i[:, k] + nb_i exactly."""
    pop, in_f, out_f, off = 5, 64, 40, (1 << 32) - 300
    x = torch.eye(in_f).repeat(pop, 1, 1)
    seeds = torch.tensor([3, -4, 5, -6, 2 ** 62], dtype=torch.int64)
    y = virtual_perturbed_linear(x.to(DEV), torch.zeros(out_f, in_f, device=DEV),
                                 torch.zeros(out_f, device=DEV), seeds.to(DEV), 1.0, off, path=path)
    dump = es.noise_dump(seeds.numpy(), out_f * in_f + out_f, off)
    for i in range(pop):
        n_i = dump[i, : out_f * in_f].reshape(out_f, in_f)
        want = (n_i + dump[i, out_f * in_f:][:, None]).T
        assert np.array_equal(y[i].cpu().numpy(), want)
    # and the forward's noise is the dump's noise on the GPU as well
    gdump = noise_dump(seeds.to(DEV), out_f * in_f, off).cpu().numpy()
    y0 = virtual_perturbed_linear(x.to(DEV), torch.zeros(out_f, in_f, device=DEV), None,
                                  seeds.to(DEV), 1.0, off, path=path)
    for i in range(pop):
        assert np.array_equal(y0[i].cpu().numpy(), gdump[i].reshape(out_f, in_f).T)


@pytest.mark.parametrize("pop,batch,in_f,out_f,shared,bias,act", [
    (152, 1, 64, 256, False, True, "tanh"), (300, 3, 67, 33, True, False, None),
    (1000, 8, 40, 5, False, True, None), (157, 2, 0, 9, False, True, "tanh"),
    (500, 1, 1030, 3, False, True, "tanh")])
def test_auto_cuda_core_forward_of_large_populations(pop, batch, in_f, out_f, shared, bias, act):
    """fp32 W, batch <= 8 and at least one individual per SM: the automatic path
    runs the one-launch chain kernel with one layer (its activation included);
    against the oracle and against the single-layer kernel (path="ffma")."""
    x, w, b, seeds, sig, off = _case(pop, batch, in_f, out_f, shared=shared, bias=bias)
    _run_and_check(x, w, b, seeds, sig, off, TOL_FP32, act=act)
    args = (x.to(DEV), w.to(DEV), None if b is None else b.to(DEV), seeds.to(DEV), sig, off)
    auto = virtual_perturbed_linear(*args, activation=act)
    ffma = virtual_perturbed_linear(*args, activation=act, path="ffma")
    scale = float(ffma.abs().max()) if ffma.numel() else 1.0
    assert torch.allclose(auto, ffma, rtol=0, atol=1e-5 * max(scale, 1e-6))


def test_workload1_forward():
    w = workloads.make(1)
    l = w.layers[0]
    _run_and_check(w.x, l.weight, l.bias, w.seeds, w.sigma, l.offset, TOL_FP32)


def test_workload2_policy_forward():
    """Three perturbed layers with tanh between, as the ES MLP policy step runs them."""
    w = workloads.make(2)
    h = w.x.to(DEV)
    want = w.x.numpy().astype(np.float64)
    for li, l in enumerate(w.layers):
        act = "tanh" if li < len(w.layers) - 1 else None
        h = virtual_perturbed_linear(h, l.weight.to(DEV), l.bias.to(DEV), w.seeds.to(DEV), w.sigma,
                                     l.offset, activation=act)
        want = es.perturbed_linear(want, l.weight.numpy(), l.bias.numpy(), w.seeds.numpy(), w.sigma,
                                   l.offset)
        if act:
            want = np.tanh(want)
        assert_close(to_np(h), want, TOL_FP32, f"w2 layer {li}")


def test_invalid_forward_calls_raise():
    x = torch.randn(2, 3, 8, device=DEV)
    w = torch.randn(4, 8, device=DEV)
    s = torch.arange(2, device=DEV)
    with pytest.raises(ValueError):
        virtual_perturbed_linear(x, torch.randn(4, 9, device=DEV), None, s, 0.1, 0)
    with pytest.raises(ValueError):
        virtual_perturbed_linear(x, w, None, torch.arange(3, device=DEV), 0.1, 0)
    with pytest.raises(VNError):
        virtual_perturbed_linear(x, w, None, s, float("inf"), 0)
    with pytest.raises(TypeError):
        virtual_perturbed_linear(x.half(), w, None, s, 0.1, 0)
    assert perturbed_linear_path(x, w) == "ffma"  # fp32 x never takes the tensor-core path


# ---------------------------------------------------------------------------
# Tensor-core (tcgen05/TMEM) path
# ---------------------------------------------------------------------------

TC_CASES = [
    # pop, batch, in, out, w dtype, shared, bias   (what each case exercises)
    (3, 32, 128, 200, torch.bfloat16, False, True),    # two M tiles, ragged out
    (5, 16, 64, 128, torch.float32, False, True),      # fp32 W, minimum N
    (2, 40, 136, 130, torch.bfloat16, False, True),    # ragged batch (N=48) and K (136)
    (11, 32, 192, 64, torch.float32, True, False),     # shared x, no bias, G=8 with a partial group
    (2, 256, 128, 256, torch.bfloat16, False, True),   # N=256, two 128-row halves per unit
    (1, 300, 64, 160, torch.bfloat16, False, True),    # batch > 256: two N tiles
    (20, 24, 1032, 40, torch.float32, False, True),    # many k chunks, ragged last chunk
    # Stage shapes (two 64-k atoms per stage unless they do not fit beside the W ring):
    # the cases above take two atoms with two W tiles (batch <= 128) or one W tile
    # (batch 256, bf16 W); fp32 W with a batch above 128 takes one-atom stages.
    (2, 200, 96, 130, torch.float32, False, True),     # fp32 W, N=208: one-atom stages, ragged K and out
    # bf16 W with a batch above 192: two stages beside one W tile. An even number
    # of k chunks takes the instance with compile-time stage slots, an odd one the
    # general ring.
    (3, 200, 512, 200, torch.bfloat16, False, True),   # even (4 chunks), ragged batch and out
    (2, 200, 392, 130, torch.bfloat16, False, True),   # even (4 chunks), ragged last k chunk
    (3, 200, 384, 200, torch.bfloat16, False, True),   # odd (3 chunks): the general ring
    (160, 200, 256, 128, torch.bfloat16, False, True), # even, 160 units on 152 CTAs: parity across units
]


@pytest.mark.parametrize("pop,batch,in_f,out_f,wdt,shared,bias", TC_CASES)
def test_tc_forward_matches_oracle(pop, batch, in_f, out_f, wdt, shared, bias):
    x, w, b, s, sig, off = _case(pop, batch, in_f, out_f, shared=shared, bias=bias,
                                 xdt=torch.bfloat16, wdt=wdt, bdt=wdt)
    _run_and_check(x, w, b, s, sig, off, TOL_BF16, path="tc")


def _random_tc_shapes(n, seed):
    """Seeded random shapes for the tensor-core path: batches from the minimum N to two N
    tiles, in any multiple of 8 up to 632 (even and odd numbers of k chunks, ragged last
    chunks), ragged out, both W dtypes, shared X, with and without bias, any 64-bit offset.
    They land on every stage schedule: grouped individuals, one individual per unit on the
    fixed two-stage loop or the general ring, one-atom stages."""
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(n):
        shapes.append((int(rng.integers(1, 4)), int(rng.integers(16, 300)), 8 * int(rng.integers(1, 80)),
                       int(rng.integers(1, 300)),
                       torch.bfloat16 if rng.random() < 0.7 else torch.float32,
                       bool(rng.random() < 0.2), bool(rng.random() < 0.8),
                       int(rng.integers(0, 1 << 62)) * 4 + int(rng.integers(0, 4))))
    return shapes


@pytest.mark.parametrize("pop,batch,in_f,out_f,wdt,shared,bias,offset", _random_tc_shapes(16, 2026))
def test_tc_forward_random_shapes(pop, batch, in_f, out_f, wdt, shared, bias, offset):
    x, w, b, s, sig, _ = _case(pop, batch, in_f, out_f, shared=shared, bias=bias,
                               xdt=torch.bfloat16, wdt=wdt, bdt=wdt, seed=in_f + out_f)
    _run_and_check(x, w, b, s, sig, offset, TOL_BF16, path="tc")


def test_tc_forward_one_hot_reads_bf16_noise_exactly():
    """X rows = e_k, W = 0, b = 0, sigma = 1 on the tensor-core path: the perturbed
    weight is bf16(N_i[j, k]) and the fp32 accumulation of one product is exact, so
    Y[i, k, :] = bf16(N_i[:, k]) + nb_i bit for bit. Pins the swizzled operand layout,
    the descriptors and the TMEM addressing to the noise indexing."""
    pop, in_f, out_f, off = 3, 64, 160, 777
    x = torch.eye(in_f).repeat(pop, 1, 1).to(torch.bfloat16)
    seeds = torch.tensor([9, -10, 11], dtype=torch.int64)
    y = virtual_perturbed_linear(x.to(DEV), torch.zeros(out_f, in_f, dtype=torch.bfloat16, device=DEV),
                                 torch.zeros(out_f, dtype=torch.bfloat16, device=DEV), seeds.to(DEV),
                                 1.0, off, path="tc")
    dump = torch.from_numpy(es.noise_dump(seeds.numpy(), out_f * in_f + out_f, off))
    for i in range(pop):
        n_bf = dump[i, : out_f * in_f].reshape(out_f, in_f).to(torch.bfloat16).float()
        nb = dump[i, out_f * in_f:]
        want = (n_bf + nb[:, None]).T.to(torch.bfloat16)   # Y is bf16 for bf16 x and W
        assert torch.equal(y[i].cpu(), want)


@pytest.mark.parametrize("in_f", [64, 192, 320])
def test_tc_one_hot_with_zero_sigma_reads_w_exactly(in_f):
    """With sigma = 0, no bias and X rows one-hot at k, the perturbed weight is W itself
    (bf16(W + 0) = W), so Y[i, k, :] = W[:, k] bit for bit. Pins how the hashing warps
    read the staged W tile: its rows (two M tiles, the second ragged), its 64-k atoms
    and its k chunks, on each stage schedule. Sizes:
    in = 64 (batch 64: four individuals per unit, one a partial group), 192 (one
    individual per unit, two stages, an even number of k chunks: the fixed loop) and 320
    (an odd number of k chunks, and a batch above 256: two N tiles)."""
    pop, out_f = 3, 200
    gen = torch.Generator().manual_seed(in_f)
    w = (torch.randn(out_f, in_f, generator=gen) / 3).to(torch.bfloat16)
    x = torch.eye(in_f).repeat(pop, 1, 1).to(torch.bfloat16)
    seeds = torch.tensor([5, -6, 7], dtype=torch.int64)
    y = virtual_perturbed_linear(x.to(DEV), w.to(DEV), None, seeds.to(DEV), 0.0, 99, path="tc")
    want = w.T.unsqueeze(0).expand(pop, in_f, out_f)
    assert torch.equal(y.cpu(), want)


def test_tc_and_auto_path_selection():
    x = torch.randn(2, 32, 64, device=DEV).to(torch.bfloat16)
    w = torch.randn(16, 64, device=DEV)
    assert perturbed_linear_path(x, w) == "tc"
    assert perturbed_linear_path(x[:, :8], w) == "ffma"          # batch < 16
    with pytest.raises(VNError):
        virtual_perturbed_linear(torch.randn(2, 32, 60, device=DEV).to(torch.bfloat16),
                                 torch.randn(16, 60, device=DEV), None, torch.arange(2, device=DEV),
                                 0.1, 0, path="tc")                 # in % 8 != 0


def test_tc_repeated_calls_are_identical_and_status_clean():
    x, w, b, s, sig, off = _case(9, 32, 256, 256, xdt=torch.bfloat16, wdt=torch.float32)
    args = (x.to(DEV), w.to(DEV), b.to(DEV), s.to(DEV), sig, off)
    y1 = virtual_perturbed_linear(*args, path="tc")
    y2 = virtual_perturbed_linear(*args, path="tc")
    assert torch.equal(y1, y2)
    from virtual_noise_perturbed_gb300 import device_status
    device_status()


def _workload_tc(number, individuals):
    """The workload's full-size call in the bench's launch configuration, checked on the
    sampled individuals against the exact forward (within 2e-2 of its RMS) and against
    the oracle's bf16 model (W + sigma*N_i rounded to bfloat16; Y too where Y is bf16),
    which fixes what the rounding itself costs: the bf16 floor, printed beside the
    kernel's deviation."""
    w = workloads.make(number)
    l = w.layers[0]
    y = virtual_perturbed_linear(w.x.to(DEV), l.weight.to(DEV), l.bias.to(DEV), w.seeds.to(DEV),
                                 w.sigma, l.offset)
    assert perturbed_linear_path(w.x.to(DEV)[:1], l.weight.to(DEV)) == "tc"
    got = to_np(y[individuals])
    args = (w.x[individuals].float().numpy(), l.weight.float().numpy(), l.bias.float().numpy(),
            w.seeds[individuals].numpy(), w.sigma, l.offset)
    want = es.perturbed_linear(*args)
    model = es.perturbed_linear_bf16(*args)               # W' rounded, Y not yet
    y_bf16 = y.dtype == torch.bfloat16
    if y_bf16:
        model = es.round_bf16(model)
    rms = float(np.sqrt(np.mean(want ** 2)))
    floor = float(np.max(np.abs(model - want))) / rms
    dev_exact = assert_close(got, want, TOL_BF16, f"workload {number}")
    # The kernel forms W' in fp32 and rounds it (and Y) to bfloat16 round-to-nearest-even,
    # so it differs from the model only where fp32 accumulation or the fp32 step before
    # the bfloat16 rounding tips a value across a rounding boundary: rarely, by one
    # bfloat16 spacing. Its RMS distance from the model is therefore a small fraction of
    # the model's own distance from the exact result; W' truncated or rounded the wrong
    # way would put it at that distance or beyond.
    model_rms = float(np.sqrt(np.mean((model - want) ** 2)))
    kernel_rms = float(np.sqrt(np.mean((got - model) ** 2)))
    assert kernel_rms <= 0.25 * model_rms, (kernel_rms / rms, model_rms / rms)
    assert dev_exact <= 2 * floor, (dev_exact, floor)
    print(f"workload {number}: deviation {dev_exact:.3e} of the RMS (bf16 floor {floor:.3e}); "
          f"RMS distance to the bf16 model {kernel_rms / rms:.2e}, model to exact {model_rms / rms:.2e}")
    return dev_exact


def _sample(pop, anchored, extra, seed):
    """Anchored individuals plus ``extra`` drawn at random (seeded), sorted."""
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(pop), anchored)
    return sorted(set(anchored) | set(rng.choice(rest, size=extra, replace=False).tolist()))


def test_workload3_forward_full_size_windows():
    _workload_tc(3, _sample(4096, [0, 1, 7, 8, 2047, 4094, 4095], 9, 3))


def test_workload5_forward_full_size_windows():
    _workload_tc(5, _sample(256, [0, 128, 255], 9, 5))


@pytest.mark.parametrize("number", [3, 5])
def test_tc_full_size_is_repeatable_under_l2_flush(number):
    """A property at any size: the same call gives the same bits every time.

    Each call runs after a 256 MiB buffer is rewritten (cold L2), which changes
    the relative timing of the kernel's roles; a missing ordering between them
    (a shared-memory tile overwritten before every reader is done) shows up as
    outputs that change from call to call."""
    w = workloads.make(number)
    l = w.layers[0]
    args = (w.x.to(DEV), l.weight.to(DEV), l.bias.to(DEV), w.seeds.to(DEV), w.sigma, l.offset)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(4):
        flush.zero_()
        outs.append(virtual_perturbed_linear(*args, path="tc"))
    torch.cuda.synchronize()
    for y in outs[1:]:
        assert torch.equal(y, outs[0])
