"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each mutation replaces one oracle function for the duration of one test with a
subtly wrong version (a wrong shift, an off-by-one state, the wrong half of the
hash, a transposed noise index, a dropped term, a wrong scale) and runs the pin
that should fail.
"""

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


_ORIG = {
    "perturbed_linear": es.perturbed_linear,
    "weight_gradient": es.weight_gradient,
    "bias_gradient": es.bias_gradient,
}

MUTATIONS = [
    # (name, [(module, attribute, replacement)], pin that must fail)
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
]


@pytest.mark.parametrize("name,patches,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, patches, pin):
    for module, attr, repl in patches:
        monkeypatch.setattr(module, attr, repl)
    with pytest.raises(AssertionError):
        pin()
