"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each mutation replaces one oracle function for the duration of one test with a
subtly wrong version (a wrong shift, an off-by-one state, the wrong half of the
hash, a transposed noise index, a dropped term, a wrong scale; in the Gaussian
variant swapped halves, sine for cosine, a missing factor, the uniform kind used by
mistake; in the ES bookkeeping a wrong tie order, divisor, key order, sign or
precision) and runs the pin that should fail.
"""

import math

import numpy as np
import pytest

import tests.test_oracle_pins as pins
from oracle import es, splitmix as sm

_G = np.uint64(sm.GAMMA)


def _mix_wrong_shift(z):
    z &= sm.MASK64
    z = ((z ^ (z >> 29)) * sm.GAMMA) & sm.MASK64
    z = ((z ^ (z >> 27)) * sm.GAMMA) & sm.MASK64
    return z ^ (z >> 31)


def _mix_np_wrong_shift(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _G
        z = (z ^ (z >> np.uint64(28))) * _G
        return z ^ (z >> np.uint64(31))


def _round_bf16_truncating(a):
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)
    return np.ldexp(np.trunc(m * 256.0), e - 8)


def _bf16_model_w_unrounded(x, weight, bias, seeds, sigma, offset, individuals=None, rows=None,
                            round_y=False):
    y = es.perturbed_linear(x, weight, bias, seeds, sigma, offset, individuals=individuals, rows=rows)
    return es.round_bf16(y) if round_y else y


def _state_off_by_one(seed, idx):
    return ((seed & sm.MASK64) + (idx & sm.MASK64) * sm.GAMMA) & sm.MASK64


def _uniform_high_half(h):
    return ((h >> 32) >> 9) * 2.0 ** -23


def _noise_np_high_half(seed_u64, idx_u64):
    h = sm.mix64_np(sm.state64_np(seed_u64, idx_u64))
    return ((h >> np.uint64(41)).astype(np.float64)) * 2.0 ** -23 - 0.5


def _weight_noise_transposed(seed, out_f, in_f, offset, rows=None, noise="uniform"):
    s = sm.seeds_u64([seed])[0]
    rows = range(out_f) if rows is None else list(rows)
    n = np.empty((len(rows), in_f))
    for r, j in enumerate(rows):
        idx = sm.element_indices(offset + j, in_f)  # start at j ...
        idx = sm.element_indices(0, in_f) * np.uint64(out_f) + idx  # ... stride out: k*out + j
        n[r] = sm.noise_np(s, idx)
    return n


def _perturbed_linear_no_bias_noise(x, weight, bias, seeds, sigma, offset, individuals=None, rows=None,
                                    noise="uniform"):
    y = _ORIG["perturbed_linear"](x, weight, None, seeds, sigma, offset, individuals, rows, noise)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        rows_l = list(range(np.asarray(weight).shape[0])) if rows is None else list(rows)
        y = y + b[rows_l][None, None, :]
    return y


def _weight_gradient_missing_sigma(fitness, seeds, weight_shape, sigma, pop_size, offset, rows=None):
    return _ORIG["weight_gradient"](fitness, seeds, weight_shape, sigma, pop_size, offset, rows) * sigma


def _weight_gradient_wrong_sign(fitness, seeds, weight_shape, sigma, pop_size, offset, rows=None):
    return -_ORIG["weight_gradient"](fitness, seeds, weight_shape, sigma, pop_size, offset, rows)


def _bias_gradient_weight_offset(fitness, seeds, bias_shape, sigma, pop_size, offset):
    return _ORIG["bias_gradient"](fitness, seeds, bias_shape, sigma, pop_size, offset - 1)


def _offsets_exclusive_off(param_shapes):
    out, total = [], 0
    for shape in param_shapes:
        total += int(np.prod(shape))
        out.append(total)
    return out


def _weight_gradient_over_pop_minus_one(fitness, seeds, weight_shape, sigma, pop_size, offset, rows=None):
    g = _ORIG["weight_gradient"](fitness, seeds, weight_shape, sigma, pop_size, offset, rows)
    return g * pop_size / (pop_size - 1)


# --- Gaussian variant --------------------------------------------------------

def _u1_u2(h):
    return 1.0 - ((h >> 32) >> 9) * 2.0 ** -23, ((h & sm.MASK32) >> 9) * 2.0 ** -23


def _gauss_halves_swapped(h):
    u1 = 1.0 - ((h & sm.MASK32) >> 9) * 2.0 ** -23
    u2 = ((h >> 32) >> 9) * 2.0 ** -23
    return math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)


def _gauss_sine(h):
    u1, u2 = _u1_u2(h)
    return math.sqrt(-2.0 * math.log(u1)) * math.sin(2.0 * math.pi * u2)


def _gauss_radius_without_two(h):
    u1, u2 = _u1_u2(h)
    return math.sqrt(-math.log(u1)) * math.cos(2.0 * math.pi * u2)


def _gauss_np_u1_not_reflected(seed_u64, idx_u64):
    h = sm.mix64_np(sm.state64_np(seed_u64, idx_u64))
    u1 = ((h >> np.uint64(32)) >> np.uint64(9)).astype(np.float64) * 2.0 ** -23   # [0, 1), not (0, 1]
    u2 = ((h & np.uint64(sm.MASK32)) >> np.uint64(9)).astype(np.float64) * 2.0 ** -23
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def _gauss_dump_uniform(seeds, n_elements, offset):
    return es.noise_dump(seeds, n_elements, offset).astype(np.float64)


def _gauss_gradient_uniform_noise(fitness, seeds, n_elements, sigma, pop_size, offset):
    f = np.asarray(fitness, dtype=np.float64)
    su = sm.seeds_u64(seeds)
    idx = sm.element_indices(offset, n_elements)
    acc = np.zeros(n_elements)
    for i in range(pop_size):
        acc += f[i] * sm.noise_np(su[i], idx)
    return acc / (pop_size * sigma)


def _weight_noise_kind_dropped(seed, out_f, in_f, offset, rows=None, noise="uniform"):
    return _ORIG["weight_noise"](seed, out_f, in_f, offset, rows)        # kind not passed on


def _bias_noise_kind_dropped(seed, out_f, bias_offset, noise="uniform"):
    return _ORIG["bias_noise"](seed, out_f, bias_offset)                 # kind not passed on


# --- centered ranks, update, metric ----------------------------------------

def _ranks(fitness, later_ties_first=False, divisor=None):
    k = es.order_keys(fitness)
    pop = k.shape[0]
    idx = np.arange(pop)
    rank = np.empty(pop, dtype=np.int64)
    for i in range(pop):
        ties = (idx > i) if later_ties_first else (idx < i)
        rank[i] = int(np.count_nonzero(k < k[i])) + int(np.count_nonzero((k == k[i]) & ties))
    d = np.float32(max(pop - 1, 1) if divisor is None else divisor(pop))
    return rank.astype(np.float32) / d - np.float32(0.5)


def _ranks_ties_reversed(fitness):
    return _ranks(fitness, later_ties_first=True)


def _ranks_over_pop(fitness):
    return _ranks(fitness, divisor=lambda pop: pop)


def _order_keys_by_value(values):
    return np.asarray(values, dtype=np.float64)    # -0 equals +0 and NaN compares unordered


def _update_descends(theta, grad, lr):
    return _ORIG["es_update"](theta, grad, -lr)


def _update_lr_in_float64(theta, grad, lr):
    return np.asarray(theta, dtype=np.float64) + lr * np.asarray(grad, dtype=np.float64)


def _metric_without_abs(center, seeds, sigma, n_params, offset=0, individuals=None):
    c = np.asarray(center, dtype=np.float64)
    su = sm.seeds_u64(seeds)
    idx = sm.element_indices(offset, n_params)
    inds = range(su.shape[0]) if individuals is None else list(individuals)
    return np.array([np.mean(c + sigma * sm.noise_np(su[i], idx)) for i in inds])


_ORIG = {
    "perturbed_linear": es.perturbed_linear,
    "weight_gradient": es.weight_gradient,
    "bias_gradient": es.bias_gradient,
    "weight_noise": es.weight_noise,
    "bias_noise": es.bias_noise,
    "es_update": es.es_update,
}

MUTATIONS = [
    # (name, [(module, attribute, replacement)], pin that must fail)
    ("bf16 rounding truncates", [(es, "round_bf16", _round_bf16_truncating)],
     pins.test_round_bf16_matches_torchs_conversion_and_ties),
    ("bf16 model leaves W' unrounded", [(es, "perturbed_linear_bf16", _bf16_model_w_unrounded)],
     pins.test_bf16_model_one_hot_reads_the_rounded_noise),
    ("finalizer shift 30 -> 29", [(sm, "mix64", _mix_wrong_shift)],
     pins.test_finalizer_inverts_with_independent_inverse),
    ("numpy finalizer shift 27 -> 28", [(sm, "mix64_np", _mix_np_wrong_shift)],
     pins.test_finalizer_numpy_matches_python_int),
    ("state uses idx instead of idx + 1", [(sm, "state64", _state_off_by_one)],
     pins.test_zero_state_gives_minus_half),
    ("uniform from the high 32 bits", [(sm, "uniform_from_hash", _uniform_high_half)],
     pins.test_low_32_bits_map_to_the_uniform),
    ("dump from the high 32 bits", [(es, "noise_np", _noise_np_high_half)],
     pins.test_noise_numpy_matches_python_int_including_wrapping),
    ("weight noise indexed k*out + j", [(es, "weight_noise", _weight_noise_transposed)],
     pins.test_forward_one_hot_reads_noise_columns_exactly),
    ("bias noise dropped", [(es, "perturbed_linear", _perturbed_linear_no_bias_noise)],
     pins.test_forward_one_hot_reads_noise_columns_exactly),
    ("gradient not divided by sigma", [(es, "weight_gradient", _weight_gradient_missing_sigma)],
     pins.test_weight_gradient_one_hot_fitness_recovers_noise_exactly),
    ("gradient sign flipped", [(es, "weight_gradient", _weight_gradient_wrong_sign)],
     pins.test_weight_gradient_expectation_on_a_linear_objective),
    ("bias gradient one element early", [(es, "bias_gradient", _bias_gradient_weight_offset)],
     pins.test_bias_gradient_matches_forward_bias_noise),
    ("offsets are end offsets", [(es, "compute_offsets", _offsets_exclusive_off)],
     pins.test_compute_offsets_worked_example),
    ("gradient averaged over pop - 1", [(es, "weight_gradient", _weight_gradient_over_pop_minus_one)],
     pins.test_weight_gradient_one_hot_fitness_recovers_noise_exactly),
    ("gaussian: u1 from the low half, u2 from the high", [(sm, "gaussian_from_hash", _gauss_halves_swapped)],
     pins.test_gaussian_reads_both_halves_hand_values),
    ("gaussian: sine instead of cosine", [(sm, "gaussian_from_hash", _gauss_sine)],
     pins.test_gaussian_reads_both_halves_hand_values),
    ("gaussian: radius sqrt(-ln u1)", [(sm, "gaussian_from_hash", _gauss_radius_without_two)],
     pins.test_gaussian_reads_both_halves_hand_values),
    ("gaussian numpy: u1 not reflected into (0, 1]", [(sm, "gaussian_noise_np", _gauss_np_u1_not_reflected)],
     pins.test_gaussian_numpy_matches_python_int),
    ("gaussian dump made of the uniform", [(es, "gaussian_dump", _gauss_dump_uniform)],
     pins.test_gaussian_statistics),
    ("gaussian gradient on the uniform", [(es, "gaussian_flat_gradient", _gauss_gradient_uniform_noise)],
     pins.test_gaussian_gradient_one_hot_fitness_recovers_noise),
    ("gaussian forward: weight noise of the uniform kind", [(es, "weight_noise", _weight_noise_kind_dropped)],
     pins.test_gaussian_forward_one_hot_recovers_the_dump_and_bias_noise),
    ("gaussian forward: bias noise of the uniform kind", [(es, "bias_noise", _bias_noise_kind_dropped)],
     pins.test_gaussian_forward_one_hot_recovers_the_dump_and_bias_noise),
    ("ranks: later equal value ranked first", [(es, "centered_ranks", _ranks_ties_reversed)],
     pins.test_centered_ranks_hand_worked_example),
    ("ranks divided by pop", [(es, "centered_ranks", _ranks_over_pop)],
     pins.test_centered_ranks_hand_worked_example),
    ("ranks ordered by float value", [(es, "order_keys", _order_keys_by_value)],
     pins.test_centered_ranks_special_values_order),
    ("update descends", [(es, "es_update", _update_descends)],
     pins.test_es_update_is_theta_plus_lr_grad),
    ("update takes lr in float64", [(es, "es_update", _update_lr_in_float64)],
     pins.test_es_update_is_theta_plus_lr_grad),
    ("metric without the absolute value", [(es, "reduce_metric", _metric_without_abs)],
     pins.test_reduce_metric_special_cases_and_brute_force),
]


@pytest.mark.parametrize("name,patches,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, patches, pin):
    for module, attr, repl in patches:
        monkeypatch.setattr(module, attr, repl)
    with pytest.raises(AssertionError):
        pin()
