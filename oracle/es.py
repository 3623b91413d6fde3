"""The virtual-noise ES step, written out plainly in float64 on the CPU.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: EvoX API page "evox.triton_kernels.kernels.virtual_noise": the module
description (the model ``Y[i] = X[i] @ (W + sigma*N_i)^T + (b + sigma*nb_i)``
and the estimate ``grad_W[j,k] = sum_i fitness_i*N_i[j,k] / (pop_size*sigma)``),
"Noise indexing scheme", and the API entries ``_cpu_normal_noise``,
``compute_offsets``, ``virtual_perturbed_linear``, ``virtual_weight_gradient``,
``virtual_bias_gradient`` and ``virtual_reduce_metric``.

Every function materialises the noise it needs (one individual at a time) and
does its arithmetic in float64 from the exact input values; there is no
blocking, fusion or reordering beyond the formula. The optional
``individuals`` / ``rows`` arguments only select which outputs to
evaluate, so that large shapes can be checked on windows; each selected output
is computed from the same definition.

Readings (see also ``splitmix``):
  R6 ``bias=None`` means no bias term and no bias noise.
  R7 ``offset`` means the weight block's offset in the forward (bias noise at
     ``offset + out*in + j``) and the bias block's own offset in
     ``bias_gradient`` (``virtual_bias_gradient`` says the caller passes the
     offset of the bias region).
  R8 ``pop_size`` must equal the number of seeds and of fitness values; the
     divisor is ``pop_size``.
  R12 activations between layers are not part of the method.
"""

from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np

from .splitmix import element_indices, gaussian_noise_np, noise_np, seeds_u64


def _check_pop(seeds: np.ndarray, pop_size: int, other: Optional[np.ndarray] = None) -> None:
    if pop_size != seeds.shape[0]:
        raise ValueError(f"pop_size={pop_size} but {seeds.shape[0]} seeds")
    if other is not None and other.shape[0] != pop_size:
        raise ValueError(f"pop_size={pop_size} but {other.shape[0]} fitness values")


def noise_dump(seeds, n_elements: int, offset: int) -> np.ndarray:
    """``_cpu_normal_noise``: ``D[i, t] = PRNG(seed_i, offset + t)``, float32 [pop, n]."""
    s = seeds_u64(seeds)
    idx = element_indices(offset, n_elements)
    out = np.empty((s.shape[0], n_elements), dtype=np.float32)
    for i in range(s.shape[0]):
        out[i] = noise_np(s[i], idx).astype(np.float32)
    return out


def compute_offsets(param_shapes: Sequence[Sequence[int]]) -> list:
    """``compute_offsets``: start offset of each block = elements of all blocks before it."""
    offsets, total = [], 0
    for shape in param_shapes:
        offsets.append(total)
        total += math.prod(int(d) for d in shape)
    return offsets


_NOISE_KINDS = {"uniform": noise_np, "gaussian": gaussian_noise_np}


def weight_noise(seed, out_f: int, in_f: int, offset: int,
                 rows: Optional[Iterable[int]] = None, noise: str = "uniform") -> np.ndarray:
    """N_i[j, k] = PRNG(seed_i, offset + j*in + k) ("Noise indexing scheme"), float64;
    ``noise="gaussian"``: the Gaussian variant's value at the same index (R16).

    ``rows`` selects which j to return (default: all, in order)."""
    s = seeds_u64([seed])[0]
    rows = np.arange(out_f, dtype=np.uint64) if rows is None else np.asarray(list(rows), dtype=np.uint64)
    with np.errstate(over="ignore"):
        idx = (np.uint64(offset & ((1 << 64) - 1)) + rows[:, None] * np.uint64(in_f)
               + np.arange(in_f, dtype=np.uint64)[None, :])        # offset + j*in + k
    return _NOISE_KINDS[noise](s, idx)


def bias_noise(seed, out_f: int, bias_offset: int, noise: str = "uniform") -> np.ndarray:
    """nb_i[j] = PRNG(seed_i, bias_offset + j), float64 (or the Gaussian variant's)."""
    s = seeds_u64([seed])[0]
    return _NOISE_KINDS[noise](s, element_indices(bias_offset, out_f))


def perturbed_linear(x, weight, bias, seeds, sigma: float, offset: int,
                     individuals: Optional[Iterable[int]] = None,
                     rows: Optional[Iterable[int]] = None, noise: str = "uniform") -> np.ndarray:
    """``virtual_perturbed_linear`` in float64.

    x: [B, in] (shared by all individuals) or [pop, B, in]; weight: [out, in];
    bias: [out] or None; seeds: [pop]. Returns [len(individuals), B, len(rows)]
    (the full [pop, B, out] by default):
        Y[i] = X[i] @ (W + sigma*N_i)^T + (b + sigma*nb_i),
    N_i at ``offset + j*in + k`` and nb_i at ``offset + out*in + j``; with
    ``noise="gaussian"`` N_i and nb_i are the Gaussian variant's values at the
    same indices (reading R16).
    """
    w = np.asarray(weight, dtype=np.float64)
    out_f, in_f = w.shape
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(seeds)
    pop = s.shape[0]
    shared = x.ndim == 2
    if x.shape[-1] != in_f or (not shared and x.shape[0] != pop):
        raise ValueError("x / weight / seeds shapes disagree")
    inds = range(pop) if individuals is None else list(individuals)
    rows = list(range(out_f)) if rows is None else list(rows)
    b = None if bias is None else np.asarray(bias, dtype=np.float64)
    batch = x.shape[-2]
    y = np.empty((len(inds), batch, len(rows)), dtype=np.float64)
    for r, i in enumerate(inds):
        n_i = weight_noise(s[i], out_f, in_f, offset, rows, noise)   # [rows, in]
        w_pert = w[rows] + sigma * n_i                                # W + sigma*N_i
        xi = x if shared else x[i]                                    # [B, in]
        yi = xi @ w_pert.T                                            # [B, rows]
        if b is not None:
            nb_i = bias_noise(s[i], out_f, offset + out_f * in_f, noise)[rows]
            yi = yi + (b[rows] + sigma * nb_i)[None, :]
        y[r] = yi
    return y


def round_bf16(a) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to the even one: keep 8
    significant bits (bfloat16's implicit bit and 7 stored bits). Written out on the
    binary exponent: a = m * 2**e with 0.5 <= |m| < 1, so m * 2**8 rounded to an integer
    (numpy's rint: half to even) times 2**(e - 8) is the nearest 8-bit-significand value.
    Defined here for zero and for |a| in bfloat16's normal range [2**-126, 2**128)
    (raises otherwise), which covers every value the bf16 model below rounds."""
    a = np.asarray(a, dtype=np.float64)
    mag = np.abs(a[a != 0])
    if mag.size and (mag.min() < 2.0 ** -126 or mag.max() >= 2.0 ** 128 or not np.all(np.isfinite(mag))):
        raise ValueError("round_bf16: a value outside bfloat16's normal range")
    m, e = np.frexp(a)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def perturbed_linear_bf16(x, weight, bias, seeds, sigma: float, offset: int,
                          individuals: Optional[Iterable[int]] = None,
                          rows: Optional[Iterable[int]] = None, round_y: bool = False) -> np.ndarray:
    """The bf16 model of the tensor-core forward: ``perturbed_linear`` with the perturbed
    weight ``W + sigma*N_i`` rounded to bfloat16 (``round_bf16``) before the product and,
    with ``round_y``, the output (after the bias) rounded to bfloat16 too. Everything else
    is float64 from the exact inputs (bf16 X values are exact in float64), so the model
    differs from ``perturbed_linear`` by those two roundings alone."""
    w = np.asarray(weight, dtype=np.float64)
    out_f, in_f = w.shape
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(seeds)
    pop = s.shape[0]
    shared = x.ndim == 2
    if x.shape[-1] != in_f or (not shared and x.shape[0] != pop):
        raise ValueError("x / weight / seeds shapes disagree")
    inds = range(pop) if individuals is None else list(individuals)
    rows = list(range(out_f)) if rows is None else list(rows)
    b = None if bias is None else np.asarray(bias, dtype=np.float64)
    y = np.empty((len(inds), x.shape[-2], len(rows)), dtype=np.float64)
    for r, i in enumerate(inds):
        n_i = weight_noise(s[i], out_f, in_f, offset, rows)
        w_pert = round_bf16(w[rows] + sigma * n_i)                    # bf16(W + sigma*N_i)
        xi = x if shared else x[i]
        yi = xi @ w_pert.T
        if b is not None:
            nb_i = bias_noise(s[i], out_f, offset + out_f * in_f)[rows]
            yi = yi + (b[rows] + sigma * nb_i)[None, :]
        y[r] = round_bf16(yi) if round_y else yi
    return y


def bf16_floor(x, weight, bias, seeds, sigma: float, offset: int,
               individuals: Optional[Iterable[int]] = None, round_y: bool = False) -> float:
    """The deviation that rounding alone costs a bf16 implementation of the forward:
    max |Y_model - Y| / RMS(Y), with Y = ``perturbed_linear`` (exact up to float64) and
    Y_model = ``perturbed_linear_bf16`` (W + sigma*N_i, and Y when ``round_y``, rounded to
    bfloat16), on the selected individuals."""
    exact = perturbed_linear(x, weight, bias, seeds, sigma, offset, individuals=individuals)
    model = perturbed_linear_bf16(x, weight, bias, seeds, sigma, offset, individuals=individuals,
                                  round_y=round_y)
    rms = float(np.sqrt(np.mean(exact ** 2)))
    return float(np.max(np.abs(model - exact))) / rms


def weight_gradient(fitness, seeds, weight_shape, sigma: float, pop_size: int,
                    offset: int, rows: Optional[Iterable[int]] = None) -> np.ndarray:
    """``virtual_weight_gradient`` in float64:
    grad[j, k] = sum_i fitness_i * N_i[j, k] / (pop_size * sigma)."""
    f = np.asarray(fitness, dtype=np.float64)
    s = np.asarray(seeds)
    _check_pop(s, pop_size, f)
    out_f, in_f = (int(d) for d in weight_shape)
    rows = list(range(out_f)) if rows is None else list(rows)
    acc = np.zeros((len(rows), in_f), dtype=np.float64)
    for i in range(pop_size):
        acc += f[i] * weight_noise(s[i], out_f, in_f, offset, rows)
    return acc / (pop_size * sigma)


def bias_gradient(fitness, seeds, bias_shape, sigma: float, pop_size: int,
                  offset: int) -> np.ndarray:
    """``virtual_bias_gradient`` in float64; ``offset`` already points at the
    bias region (reading R7): grad[j] = sum_i fitness_i * nb_i[j] / (pop_size*sigma)."""
    f = np.asarray(fitness, dtype=np.float64)
    s = np.asarray(seeds)
    _check_pop(s, pop_size, f)
    (out_f,) = (int(d) for d in bias_shape)
    acc = np.zeros(out_f, dtype=np.float64)
    for i in range(pop_size):
        acc += f[i] * bias_noise(s[i], out_f, offset)
    return acc / (pop_size * sigma)


def reduce_metric(center, seeds, sigma: float, n_params: int, offset: int = 0,
                  individuals: Optional[Iterable[int]] = None) -> np.ndarray:
    """``virtual_reduce_metric`` in float64:
    fitness[i] = mean_k | center[k] + sigma * PRNG(seed_i, offset + k) |."""
    c = np.asarray(center, dtype=np.float64)
    if c.shape != (n_params,):
        raise ValueError("center must have n_params elements")
    s = seeds_u64(seeds)
    inds = range(s.shape[0]) if individuals is None else list(individuals)
    idx = element_indices(offset, n_params)
    out = np.empty(len(inds), dtype=np.float64)
    for r, i in enumerate(inds):
        out[r] = np.mean(np.abs(c + sigma * noise_np(s[i], idx)))
    return out


def order_keys(values) -> np.ndarray:
    """A total order on float32 values as unsigned keys: negative below positive,
    -0 below +0, NaNs beyond the infinities on their sign's side. For a set sign bit
    the key is the complement of the bits (larger magnitude -> smaller key); for a
    clear one the bits with the sign bit set."""
    b = np.asarray(values, dtype=np.float32).view(np.uint32).astype(np.uint64)
    neg = (b >> np.uint64(31)) == np.uint64(1)
    return np.where(neg, np.uint64(0xFFFFFFFF) - b, b | np.uint64(0x80000000))


def centered_ranks(fitness) -> np.ndarray:
    """Fitness shaping of the ES workloads ("centered ranks in [-0.5, 0.5]"):
    rank_i = #{j : f_j < f_i} + #{j < i : f_j == f_i} (ascending, ties by index),
    out_i = rank_i / (pop - 1) - 0.5, the division and subtraction in float32.
    Counted one element at a time against the whole population."""
    k = order_keys(fitness)
    pop = k.shape[0]
    idx = np.arange(pop)
    rank = np.empty(pop, dtype=np.int64)
    for i in range(pop):
        rank[i] = int(np.count_nonzero(k < k[i])) + int(np.count_nonzero((k == k[i]) & (idx < i)))
    denom = np.float32(max(pop - 1, 1))
    return rank.astype(np.float32) / denom - np.float32(0.5)


def es_update(theta, grad, lr: float) -> np.ndarray:
    """The ES parameter step theta + lr * grad, in float64 from the float32 inputs
    (lr taken as its float32 value, as the library receives it)."""
    lr32 = float(np.float32(lr))
    return np.asarray(theta, dtype=np.float64) + lr32 * np.asarray(grad, dtype=np.float64)


def gaussian_dump(seeds, n_elements: int, offset: int) -> np.ndarray:
    """The Gaussian variant's dump (reading R16): D[i, t] = G(seed_i, offset + t), float64."""
    s = seeds_u64(seeds)
    idx = element_indices(offset, n_elements)
    return np.stack([gaussian_noise_np(s[i], idx) for i in range(s.shape[0])]) if s.shape[0] else \
        np.zeros((0, n_elements))


def gaussian_flat_gradient(fitness, seeds, n_elements: int, sigma: float, pop_size: int,
                           offset: int) -> np.ndarray:
    """The gradient estimate with Gaussian-variant noise, float64:
    grad[t] = sum_i fitness_i * G(seed_i, offset + t) / (pop_size * sigma)."""
    f = np.asarray(fitness, dtype=np.float64)
    s = np.asarray(seeds)
    _check_pop(s, pop_size, f)
    su = seeds_u64(s)
    idx = element_indices(offset, n_elements)
    acc = np.zeros(n_elements, dtype=np.float64)
    for i in range(pop_size):
        acc += f[i] * gaussian_noise_np(su[i], idx)
    return acc / (pop_size * sigma)
