"""Pins for the CPU oracle: each test ties the oracle to something other than itself.

The EvoX API page "evox.triton_kernels.kernels.virtual_noise" prints no noise
values, so the hash is pinned through mathematics: an inverse of the finalizer
derived here step by step, closed-form special states, the generator's stream
property, and the statistics the page states. The method is pinned by brute
force on tiny shapes, exact one-hot recoveries, an expectation identity of the
ES estimate, and the page's worked example for ``compute_offsets``.
"""

import json
import math
import os
import random

import numpy as np
import pytest

from oracle import es, splitmix as sm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1


# ---------------------------------------------------------------------------
# An inverse of the printed finalizer, derived independently of the oracle:
# undo "x ^= x >> r" by re-applying the shift until the top bits propagate, and
# undo "x *= G" with the multiplicative inverse of the odd constant mod 2**64.
# ---------------------------------------------------------------------------

def _unxorshift_right(y: int, r: int) -> int:
    x = y
    for _ in range(64 // r + 1):
        x = y ^ (x >> r)
    return x & M64


def _inverse_finalizer(y: int, gamma: int) -> int:
    g_inv = pow(gamma, -1, 1 << 64)
    y = _unxorshift_right(y, 31)
    y = (y * g_inv) & M64
    y = _unxorshift_right(y, 27)
    y = (y * g_inv) & M64
    y = _unxorshift_right(y, 30)
    return y


GAMMA_PAGE = int(json.load(open(os.path.join(GOLDEN, "gamma.json")))["gamma_decimal"])
EDGE = [0, 1, 2, (1 << 32) - 1, 1 << 32, (1 << 63) - 1, 1 << 63, M64, 0x9E3779B97F4A7C15]


def _rand_u64(rng, n):
    return [rng.getrandbits(64) for _ in range(n)]


def test_gamma_is_the_printed_constant():
    assert sm.GAMMA == GAMMA_PAGE
    assert GAMMA_PAGE == 0x9E3779B97F4A7C15  # the golden ratio constant of splitmix64
    assert GAMMA_PAGE % 2 == 1               # odd, so the multiply is a bijection mod 2**64


def test_finalizer_inverts_with_independent_inverse():
    rng = random.Random(1)
    for z in EDGE + _rand_u64(rng, 20000):
        y = sm.mix64(z)
        assert 0 <= y <= M64
        assert _inverse_finalizer(y, GAMMA_PAGE) == z
        assert sm.mix64(_inverse_finalizer(z, GAMMA_PAGE)) == z


def test_finalizer_numpy_matches_python_int():
    rng = random.Random(2)
    zs = EDGE + _rand_u64(rng, 100000)
    got = sm.mix64_np(np.array(zs, dtype=np.uint64))
    assert [int(v) for v in got] == [sm.mix64(z) for z in zs]


def test_noise_numpy_matches_python_int_including_wrapping():
    rng = random.Random(3)
    seeds = [0, 1, -1, -(2 ** 63), 2 ** 63 - 1] + [rng.randrange(-2 ** 63, 2 ** 63) for _ in range(40)]
    offsets = [0, 123456789, (1 << 32) - 3, (1 << 64) - 5]
    for off in offsets:
        d = es.noise_dump(np.array(seeds, dtype=np.int64), 9, off)
        for r, s in enumerate(seeds):
            for t in range(9):
                assert d[r, t] == np.float32(sm.noise(s, off + t))


def test_zero_state_gives_minus_half():
    # mix(0) == 0 by inspection of the finalizer (xor-shifts and products of 0).
    assert sm.mix64(0) == 0
    assert sm.noise(0, M64) == -0.5          # state = 0 + (2**64) * G = 0 mod 2**64
    rng = random.Random(4)
    for idx in [0, 1, 77, 1 << 40] + [rng.getrandbits(64) for _ in range(100)]:
        seed = (-(idx + 1) * GAMMA_PAGE) & M64  # makes the state exactly 0
        assert sm.noise(seed, idx) == -0.5


def test_stream_property_of_the_state():
    # Reading R1: element idx of seed s is element idx-k of seed s + k*G.
    rng = random.Random(5)
    for _ in range(2000):
        s, idx, k = rng.getrandbits(64), rng.getrandbits(64), rng.randrange(1, 1000)
        assert sm.noise(s, idx) == sm.noise((s + k * GAMMA_PAGE) & M64, (idx - k) & M64)


def test_low_32_bits_map_to_the_uniform():
    """Choose the hash output, invert it to a state, and check the value read off it.

    Pins that the low (not high) 32 bits are used, that the top 23 of them make
    the mantissa, and the -0.5 shift."""
    rng = random.Random(6)
    cases = [
        (0x00000000_00000000, -0.5),
        (0xFFFFFFFF_00000000, -0.5),               # high half ignored
        (0x00000000_000001FF, -0.5),               # bits below 9 dropped
        (0x00000000_FFFFFFFF, 0.5 - 2 ** -23),     # the largest value, < 0.5
        (0x12345678_80000000, 0.0),
        (0x00000000_00000200, -0.5 + 2 ** -23),
    ]
    for _ in range(2000):
        h = rng.getrandbits(64)
        cases.append((h, ((h & 0xFFFFFFFF) >> 9) / 2 ** 23 - 0.5))
    for h, want in cases:
        state = _inverse_finalizer(h, GAMMA_PAGE)
        idx = rng.getrandbits(64)
        seed = (state - (idx + 1) * GAMMA_PAGE) & M64
        assert sm.noise(seed, idx) == want


def test_noise_statistics_stated_on_the_page():
    n = 1_000_000
    seeds = np.array([7, -3], dtype=np.int64)
    d = es.noise_dump(seeds, n // 2, 999).astype(np.float64).ravel()
    assert np.all(np.isfinite(d))
    assert d.min() >= -0.5 and d.max() < 0.5
    m = d * 2 ** 23
    assert np.all(m == np.round(m))                     # multiples of 2**-23
    assert abs(d.mean()) < 5 * math.sqrt(1 / 12 / n)     # mean ~ 0
    assert abs(d.var() - 1 / 12) < 5 * 7.5e-5           # variance 1/12
    counts, _ = np.histogram(d, bins=64, range=(-0.5, 0.5))
    chi2 = ((counts - n / 64) ** 2 / (n / 64)).sum()
    assert chi2 < 63 + 6 * math.sqrt(2 * 63)            # uniform, 63 dof


def test_signed_and_int32_seeds():
    a = es.noise_dump(np.array([-1, 5, -7], dtype=np.int32), 33, 10)
    b = es.noise_dump(np.array([-1, 5, -7], dtype=np.int64), 33, 10)
    c = es.noise_dump(np.array([M64, 5, M64 - 6], dtype=np.uint64), 33, 10)
    assert np.array_equal(a, b) and np.array_equal(b, c)


def test_dump_window_identity():
    seeds = np.arange(5, dtype=np.int64) * 1000003 - 2
    full = es.noise_dump(seeds, 300, 77)
    for t0, t1 in [(0, 1), (17, 123), (250, 300)]:
        assert np.array_equal(full[:, t0:t1], es.noise_dump(seeds, t1 - t0, 77 + t0))


def test_compute_offsets_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "compute_offsets.json")))
    assert es.compute_offsets([tuple(s) for s in g["param_shapes"]]) == g["offsets"]
    # The ES MLP policy 64 -> 256 -> 256 -> 8, weights then bias per layer.
    shapes = [(256, 64), (256,), (256, 256), (256,), (8, 256), (8,)]
    assert es.compute_offsets(shapes) == [0, 16384, 16640, 82176, 82432, 84480]
    assert es.compute_offsets([]) == []


# ---------------------------------------------------------------------------
# Forward
# ---------------------------------------------------------------------------

def _brute_forward(x, w, b, seeds, sigma, offset):
    """Pure-Python loops, one noise element at a time from the Python-int hash."""
    pop = len(seeds)
    out_f, in_f = len(w), len(w[0])
    shared = not isinstance(x[0][0], list)
    batch = len(x) if shared else len(x[0])
    y = [[[0.0] * out_f for _ in range(batch)] for _ in range(pop)]
    for i in range(pop):
        xi = x if shared else x[i]
        for r in range(batch):
            for j in range(out_f):
                acc = 0.0
                for k in range(in_f):
                    acc += xi[r][k] * (w[j][k] + sigma * sm.noise(seeds[i], offset + j * in_f + k))
                if b is not None:
                    acc += b[j] + sigma * sm.noise(seeds[i], offset + out_f * in_f + j)
                y[i][r][j] = acc
    return y


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_forward_matches_brute_force(shared, with_bias):
    rng = np.random.default_rng(10)
    pop, batch, in_f, out_f = 3, 2, 5, 4
    x = rng.standard_normal((batch, in_f) if shared else (pop, batch, in_f))
    w = rng.standard_normal((out_f, in_f))
    b = rng.standard_normal(out_f) if with_bias else None
    seeds = [3, -9, 2 ** 40 + 1]
    sigma, offset = 0.37, (1 << 32) - 7
    got = es.perturbed_linear(x, w, b, np.array(seeds), sigma, offset)
    want = np.array(_brute_forward(x.tolist(), w.tolist(), None if b is None else b.tolist(),
                                   seeds, sigma, offset))
    assert got.shape == (pop, batch, out_f)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_forward_sigma_zero_is_plain_linear():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 3, 6))
    w = rng.standard_normal((5, 6))
    b = rng.standard_normal(5)
    got = es.perturbed_linear(x, w, b, np.arange(4), 0.0, 0)
    want = np.einsum("ibk,jk->ibj", x, w) + b
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def test_forward_one_hot_reads_noise_columns_exactly():
    """X rows = e_k, W = 0, b = 0, sigma = 1 gives Y[i, r, :] = N_i[:, k_r] + nb_i, exactly;
    N_i comes from the dump reshaped row-major ("Noise indexing scheme")."""
    pop, in_f, out_f, offset = 3, 6, 5, 1000
    seeds = np.array([11, 12, -13])
    x = np.zeros((pop, in_f, in_f))
    for i in range(pop):
        x[i] = np.eye(in_f)
    y = es.perturbed_linear(x, np.zeros((out_f, in_f)), np.zeros(out_f), seeds, 1.0, offset)
    dump = es.noise_dump(seeds, out_f * in_f + out_f, offset).astype(np.float64)
    for i in range(pop):
        n_i = dump[i, : out_f * in_f].reshape(out_f, in_f)
        nb_i = dump[i, out_f * in_f:]
        assert np.array_equal(y[i], (n_i + nb_i[:, None]).T)
    # Without a bias there is no bias noise either (reading R6).
    y0 = es.perturbed_linear(x, np.zeros((out_f, in_f)), None, seeds, 1.0, offset)
    for i in range(pop):
        assert np.array_equal(y0[i], dump[i, : out_f * in_f].reshape(out_f, in_f).T)


def test_forward_noise_identity():
    """(Y - X W^T - b) / sigma = X N_i^T + nb_i."""
    rng = np.random.default_rng(12)
    pop, batch, in_f, out_f, sigma, offset = 4, 3, 7, 6, 0.01, 55
    seeds = np.array([1, 2, 3, 4]) * 7919
    x = rng.standard_normal((pop, batch, in_f))
    w = rng.standard_normal((out_f, in_f))
    b = rng.standard_normal(out_f)
    y = es.perturbed_linear(x, w, b, seeds, sigma, offset)
    dump = es.noise_dump(seeds, out_f * in_f + out_f, offset).astype(np.float64)
    for i in range(pop):
        n_i = dump[i, : out_f * in_f].reshape(out_f, in_f)
        nb_i = dump[i, out_f * in_f:]
        lhs = (y[i] - x[i] @ w.T - b) / sigma
        np.testing.assert_allclose(lhs, x[i] @ n_i.T + nb_i, rtol=1e-8, atol=1e-10)


def test_forward_shared_x_equals_broadcast_x():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((3, 8))
    w = rng.standard_normal((4, 8))
    seeds = np.array([5, 6, 7, 8, 9])
    a = es.perturbed_linear(x, w, None, seeds, 0.1, 3)
    b = es.perturbed_linear(np.broadcast_to(x, (5, 3, 8)), w, None, seeds, 0.1, 3)
    assert np.array_equal(a, b)


def test_forward_windows_match_full():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((6, 2, 9))
    w = rng.standard_normal((7, 9))
    b = rng.standard_normal(7)
    seeds = np.arange(6) + 100
    full = es.perturbed_linear(x, w, b, seeds, 0.2, 9)
    win = es.perturbed_linear(x, w, b, seeds, 0.2, 9, individuals=[0, 5], rows=[1, 6])
    assert np.array_equal(win, full[[0, 5]][:, :, [1, 6]])


# ---------------------------------------------------------------------------
# Gradients
# ---------------------------------------------------------------------------

def test_weight_gradient_one_hot_fitness_recovers_noise_exactly():
    """f = e_m * pop * sigma with pop and sigma powers of two gives grad_W == N_m exactly."""
    pop, sigma, out_f, in_f, offset = 8, 2.0 ** -7, 5, 6, 123456789
    seeds = np.arange(1, pop + 1)
    dump = es.noise_dump(seeds, out_f * in_f, offset).astype(np.float64)
    for m in (0, 3, 7):
        f = np.zeros(pop)
        f[m] = pop * sigma
        g = es.weight_gradient(f, seeds, (out_f, in_f), sigma, pop, offset)
        assert np.array_equal(g, dump[m].reshape(out_f, in_f))


def test_weight_gradient_equals_fitness_weighted_dump():
    rng = np.random.default_rng(15)
    pop, out_f, in_f, sigma, offset = 16, 4, 5, 0.05, 31
    seeds = rng.integers(-2 ** 40, 2 ** 40, pop)
    f = rng.standard_normal(pop)
    g = es.weight_gradient(f, seeds, (out_f, in_f), sigma, pop, offset)
    dump = es.noise_dump(seeds, out_f * in_f, offset).astype(np.float64)
    np.testing.assert_allclose(g, (f @ dump).reshape(out_f, in_f) / (pop * sigma), rtol=1e-12, atol=1e-14)
    # Linearity in the fitness.
    f2 = rng.standard_normal(pop)
    g2 = es.weight_gradient(f2, seeds, (out_f, in_f), sigma, pop, offset)
    g12 = es.weight_gradient(2 * f - 3 * f2, seeds, (out_f, in_f), sigma, pop, offset)
    np.testing.assert_allclose(g12, 2 * g - 3 * g2, rtol=1e-10, atol=1e-12)
    # Row windows are the same definition.
    gr = es.weight_gradient(f, seeds, (out_f, in_f), sigma, pop, offset, rows=[3, 1])
    assert np.array_equal(gr, g[[3, 1]])


def test_weight_gradient_expectation_on_a_linear_objective():
    """f_i = <C, W + sigma N_i> with W = 0 gives E[grad_W] = Var(noise) * C = C / 12.

    Catches a wrong scale (sigma, pop), a wrong sign, or noise regenerated at the
    wrong index between the objective and the estimate."""
    rng = np.random.default_rng(16)
    out_f, in_f, pop, sigma, offset = 3, 4, 40000, 0.03, 500
    c = rng.standard_normal((out_f, in_f))
    seeds = np.arange(pop, dtype=np.int64) * 3 + 1
    dump = es.noise_dump(seeds, out_f * in_f, offset).astype(np.float64)
    f = sigma * dump @ c.ravel()
    g = es.weight_gradient(f, seeds, (out_f, in_f), sigma, pop, offset)
    terms = (f[:, None] * dump) / sigma                     # per-individual contributions
    se = terms.std(axis=0) / math.sqrt(pop)
    assert np.all(np.abs(g.ravel() - c.ravel() / 12) < 5 * se)


def test_bias_gradient_matches_forward_bias_noise():
    """virtual_bias_gradient at offset + out*in regenerates the forward's bias noise."""
    pop, sigma, out_f, in_f, offset = 4, 0.25, 6, 3, 40
    seeds = np.array([9, -8, 7, -6])
    y = es.perturbed_linear(np.zeros((pop, 1, in_f)), np.zeros((out_f, in_f)), np.zeros(out_f),
                            seeds, 1.0, offset)                      # Y = nb_i exactly
    for m in range(pop):
        f = np.zeros(pop)
        f[m] = pop * sigma
        g = es.bias_gradient(f, seeds, (out_f,), sigma, pop, offset + out_f * in_f)
        assert np.array_equal(g, y[m, 0])


def test_gradients_refuse_mismatched_population():
    with pytest.raises(ValueError):
        es.weight_gradient(np.ones(3), np.arange(4), (2, 2), 0.1, 4, 0)
    with pytest.raises(ValueError):
        es.bias_gradient(np.ones(4), np.arange(4), (2,), 0.1, 5, 0)


# ---------------------------------------------------------------------------
# Mean-abs reduction metric
# ---------------------------------------------------------------------------

def test_reduce_metric_special_cases_and_brute_force():
    rng = np.random.default_rng(17)
    center = rng.standard_normal(50)
    seeds = np.array([1, 2, 3])
    np.testing.assert_allclose(es.reduce_metric(center, seeds, 0.0, 50, 0), np.abs(center).mean(), rtol=1e-14)
    dump = es.noise_dump(seeds, 50, 7).astype(np.float64)
    np.testing.assert_allclose(es.reduce_metric(np.zeros(50), seeds, 1.0, 50, 7),
                               np.abs(dump).mean(axis=1), rtol=1e-14)
    got = es.reduce_metric(center, seeds, 0.3, 50, 7)
    for i, s in enumerate(seeds.tolist()):
        want = sum(abs(center[k] + 0.3 * sm.noise(s, 7 + k)) for k in range(50)) / 50
        assert abs(got[i] - want) < 1e-13


# ---------------------------------------------------------------------------
# Centered ranks and the parameter update
# ---------------------------------------------------------------------------

def test_centered_ranks_hand_worked_example():
    # ascending order: -1.0 (index 1), 0.3 (index 0), 0.3 (index 2, after the
    # equal value at the lower index), 2.0 (index 3) -> ranks 1, 0, 2, 3
    got = es.centered_ranks(np.array([0.3, -1.0, 0.3, 2.0], dtype=np.float32))
    want = np.array([1, 0, 2, 3], dtype=np.float32) / np.float32(3) - np.float32(0.5)
    assert got.dtype == np.float32 and np.array_equal(got, want)
    assert np.array_equal(es.centered_ranks(np.array([7.0], dtype=np.float32)), np.float32([-0.5]))


def test_centered_ranks_special_values_order():
    vals = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0], dtype=np.float32)
    assert np.signbit(vals[1]) and not np.signbit(vals[0])
    # -NaN < -inf < -0 < +0 < +inf < +NaN
    want = np.array([5, 0, 4, 1, 3, 2], dtype=np.float32) / np.float32(5) - np.float32(0.5)
    assert np.array_equal(es.centered_ranks(vals), want)


def test_centered_ranks_match_a_stable_sort_and_are_a_permutation():
    rng = np.random.default_rng(23)
    f = rng.integers(-20, 20, size=300).astype(np.float32) * np.float32(0.25)  # many ties
    got = es.centered_ranks(f)
    order = np.argsort(f, kind="stable")           # an independent route to the ranks
    rank = np.empty(300, dtype=np.int64)
    rank[order] = np.arange(300)
    assert np.array_equal(got, rank.astype(np.float32) / np.float32(299) - np.float32(0.5))
    assert np.array_equal(np.sort(got), np.arange(300, dtype=np.float32) / np.float32(299) - np.float32(0.5))


def test_es_update_is_theta_plus_lr_grad():
    theta = np.array([1.0, -2.0, 0.5], dtype=np.float32)
    grad = np.array([2.0, 4.0, -1.0], dtype=np.float32)
    assert np.array_equal(es.es_update(theta, grad, 0.5), np.array([2.0, 0.0, 0.0]))
    # lr is used at float32 precision, as the library receives it
    assert es.es_update(np.zeros(1, np.float32), np.ones(1, np.float32), 0.1)[0] == float(np.float32(0.1))


# ---------------------------------------------------------------------------
# Gaussian variant (Box-Muller on the two halves of the finalizer output)
# ---------------------------------------------------------------------------

def test_gaussian_reads_both_halves_hand_values():
    """Choose finalizer outputs, invert them to states, and check Box-Muller's value.

    hi32 -> u1 = 1 - (hi32 >> 9) 2^-23 and lo32 -> u2 = (lo32 >> 9) 2^-23, by hand:
    hi32 = 2^31 gives u1 = 1/2, lo32 = 0 gives u2 = 0 -> g = sqrt(2 ln 2);
    hi32 < 2^9 gives u1 = 1 -> g = 0 whatever u2; lo32 = 2^31 gives u2 = 1/2 -> g = -sqrt(-2 ln u1)."""
    rng = random.Random(11)
    r_half = math.sqrt(2.0 * math.log(2.0))
    cases = [
        (0x80000000_00000000, r_half),
        (0x80000000_000001FF, r_half),                     # bits below 9 of lo32 dropped
        (0x000001FF_12345678, 0.0),                        # u1 = 1
        (0x80000000_80000000, -r_half),                    # u2 = 1/2: cos = -1
        (0xC0000000_00000000, math.sqrt(-2.0 * math.log(0.25))),   # u1 = 1 - 3/4
    ]
    for h, want in cases:
        state = _inverse_finalizer(h, GAMMA_PAGE)
        idx = rng.getrandbits(64)
        seed = (state - (idx + 1) * GAMMA_PAGE) & M64
        assert abs(sm.gaussian_noise(seed, idx) - want) < 1e-15


def test_gaussian_numpy_matches_python_int():
    rng = random.Random(12)
    seeds = _rand_u64(rng, 50) + EDGE
    idx = _rand_u64(rng, 50) + EDGE
    got = sm.gaussian_noise_np(np.array(seeds, dtype=np.uint64), np.array(idx, dtype=np.uint64))
    for g, s, i in zip(got, seeds, idx):
        assert abs(g - sm.gaussian_noise(s, i)) < 1e-12


def test_gaussian_statistics():
    g = es.gaussian_dump(np.arange(4), 250000, 12345).ravel()
    n = g.size
    assert np.all(np.isfinite(g)) and np.max(np.abs(g)) < 5.8   # |g| <= sqrt(2*23*ln 2)
    assert abs(g.mean()) < 5 / math.sqrt(n)
    assert abs(g.var() - 1.0) < 5 * math.sqrt(2.0 / n)
    assert abs(np.mean(np.abs(g) > 2.0) - math.erfc(2.0 / math.sqrt(2.0))) < 5e-4
    # Kolmogorov-Smirnov distance to the standard normal CDF
    s = np.sort(g[:200000])
    cdf = 0.5 * (1.0 + np.vectorize(math.erf)(s / math.sqrt(2.0)))
    emp = np.arange(1, s.size + 1) / s.size
    assert np.max(np.abs(emp - cdf)) < 1.63 / math.sqrt(s.size) * 1.5


def test_gaussian_gradient_one_hot_fitness_recovers_noise():
    seeds = np.array([3, -4, 5, 9])
    pop, sigma, off, n = 4, 2.0 ** -3, 77, 33
    dump = es.gaussian_dump(seeds, n, off)
    for m in range(pop):
        f = np.zeros(pop)
        f[m] = pop * sigma
        np.testing.assert_allclose(es.gaussian_flat_gradient(f, seeds, n, sigma, pop, off), dump[m],
                                   rtol=0, atol=1e-15)


def test_gaussian_forward_one_hot_recovers_the_dump_and_bias_noise():
    """Forward with the Gaussian variant, indexing pinned to the dump's: with X rows
    e_k, W = 0, sigma = 1 and a zero bias, Y[i, r, :] = G(seed_i, offset + j*in + k_r)
    + G(seed_i, offset + out*in + j); without a bias, the column alone."""
    seeds = np.array([5, -2, 17])
    pop, out_f, in_f, off = 3, 6, 5, 999
    dump = es.gaussian_dump(seeds, out_f * in_f + out_f, off)          # [pop, out*in + out]
    x = np.eye(in_f)[None].repeat(pop, axis=0)                          # row r = e_r
    y = es.perturbed_linear(x, np.zeros((out_f, in_f)), None, seeds, 1.0, off, noise="gaussian")
    for i in range(pop):
        n_i = dump[i, :out_f * in_f].reshape(out_f, in_f)
        np.testing.assert_array_equal(y[i], n_i.T)                      # Y[i, k, j] = N_i[j, k]
    yb = es.perturbed_linear(x, np.zeros((out_f, in_f)), np.zeros(out_f), seeds, 1.0, off,
                             noise="gaussian")
    for i in range(pop):
        np.testing.assert_allclose(yb[i] - y[i], np.broadcast_to(dump[i, out_f * in_f:], (in_f, out_f)),
                                   rtol=0, atol=1e-15)


def test_gaussian_forward_identity_and_linearity_in_sigma():
    """(Y - X W^T - b) / sigma = X G_i^T + gb_i: the same for two sigmas, and zero noise
    at sigma = 0 (a plain linear layer, against numpy's matmul)."""
    rng = np.random.default_rng(9)
    pop, batch, in_f, out_f, off = 3, 2, 7, 4, 31
    x = rng.standard_normal((pop, batch, in_f))
    w = rng.standard_normal((out_f, in_f))
    b = rng.standard_normal(out_f)
    seeds = np.arange(pop) + 40
    plain = x @ w.T + b
    np.testing.assert_allclose(es.perturbed_linear(x, w, b, seeds, 0.0, off, noise="gaussian"), plain,
                               rtol=0, atol=1e-12)
    e1 = (es.perturbed_linear(x, w, b, seeds, 0.25, off, noise="gaussian") - plain) / 0.25
    e2 = (es.perturbed_linear(x, w, b, seeds, 0.75, off, noise="gaussian") - plain) / 0.75
    np.testing.assert_allclose(e1, e2, rtol=0, atol=1e-12)
    eu = (es.perturbed_linear(x, w, b, seeds, 0.25, off) - plain) / 0.25       # the uniform kind
    assert np.max(np.abs(eu - e1)) > 0.1                                         # differs from it


# --- the bf16 model of the tensor-core forward and its floor (the perturbed weight,
# and optionally the output, rounded to bfloat16; module description of the page: the
# noise is added to the weight tile that the bf16 contraction then reads)

def test_round_bf16_matches_torchs_conversion_and_ties():
    """On float32 inputs (exact in float64, so one rounding either way) the oracle's
    rounding equals torch's float32 -> bfloat16 conversion (round to nearest, ties to
    even), over many binades and both signs; ties worked by hand."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    a = (rng.standard_normal(200_000) * np.exp2(rng.integers(-60, 60, 200_000))).astype(np.float32)
    # values just around bf16 ties: a bf16 value plus half its spacing, and one float32 ulp either side
    base = torch.tensor(rng.standard_normal(20_000), dtype=torch.bfloat16).float().numpy()
    half = np.abs(base) * np.float32(2.0 ** -8)
    ties = np.concatenate([base + half, np.nextafter(base + half, np.float32(np.inf)),
                           np.nextafter(base + half, np.float32(-np.inf))]).astype(np.float32)
    for v in (a, ties):
        want = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
        assert np.array_equal(es.round_bf16(v.astype(np.float64)), want)
    hand = es.round_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 255.5, 0.0, 2 ** -126]))
    assert list(hand) == [1.0, 1 + 2 ** -6, -1.0, 256.0, 0.0, 2 ** -126]
    with pytest.raises(ValueError):
        es.round_bf16(np.array([2.0 ** -130]))


def test_bf16_model_special_cases():
    """sigma = 0 and bf16-exact weights: rounding W' changes nothing, so the model is the
    exact forward; with round_y it is that forward rounded to bfloat16."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((3, 4, 24))
    w = es.round_bf16(rng.standard_normal((10, 24)) / 5)
    b = rng.standard_normal(10) * 0.1
    seeds = np.array([1, 2, 3])
    exact = es.perturbed_linear(x, w, b, seeds, 0.0, 7)
    assert np.array_equal(es.perturbed_linear_bf16(x, w, b, seeds, 0.0, 7), exact)
    assert np.array_equal(es.perturbed_linear_bf16(x, w, b, seeds, 0.0, 7, round_y=True), es.round_bf16(exact))
    assert es.bf16_floor(x, w, b, seeds, 0.0, 7) == 0.0


def test_bf16_model_one_hot_reads_the_rounded_noise():
    """X rows one-hot at k, W = 0, sigma = 1, no bias: the model's Y[i, r, j] is the
    bfloat16 rounding of noise element j*in + k, i.e. torch's bfloat16 of the float32
    dump (the noise values are exact in float32)."""
    torch = pytest.importorskip("torch")
    pop, in_f, out_f, off = 3, 9, 13, 2 ** 40 + 5
    seeds = np.array([4, -8, 15])
    ks = [0, 4, 8]
    x = np.zeros((pop, len(ks), in_f))
    for r, k in enumerate(ks):
        x[:, r, k] = 1.0
    y = es.perturbed_linear_bf16(x, np.zeros((out_f, in_f)), None, seeds, 1.0, off)
    dump = es.noise_dump(seeds, out_f * in_f, off).reshape(pop, out_f, in_f)
    want = torch.from_numpy(dump).to(torch.bfloat16).double().numpy()
    for r, k in enumerate(ks):
        assert np.array_equal(y[:, r, :], want[:, :, k])


def test_bf16_floor_is_within_the_rounding_bound():
    """Each rounding to bfloat16 has relative error at most 2^-9, so the model deviates
    from the exact forward by at most 2^-9 * (sum_k |x_k| |W'_jk| + |Y|) per output; the
    floor is positive for a generic case and below that bound, and grows when Y is
    rounded too."""
    rng = np.random.default_rng(13)
    x = es.round_bf16(rng.standard_normal((4, 16, 64)))
    w = rng.standard_normal((32, 64)) / 8
    b = rng.standard_normal(32) * 0.1
    seeds = np.arange(4)
    exact = es.perturbed_linear(x, w, b, seeds, 0.05, 3)
    rms = np.sqrt(np.mean(exact ** 2))
    wp = np.stack([w + 0.05 * es.weight_noise(s, 32, 64, 3) for s in seeds])  # [pop, out, in]
    bound_w = 2.0 ** -9 * np.einsum("prk,pjk->prj", np.abs(x), np.abs(wp))
    f_w = es.bf16_floor(x, w, b, seeds, 0.05, 3)
    f_y = es.bf16_floor(x, w, b, seeds, 0.05, 3, round_y=True)
    assert 0.0 < f_w <= np.max(bound_w) / rms
    assert f_w < f_y <= np.max(bound_w * (1 + 2.0 ** -9) + 2.0 ** -9 * np.abs(exact)) / rms
