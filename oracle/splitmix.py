"""splitmix64 hash and centered-uniform noise: the oracle's definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: EvoX API page "evox.triton_kernels.kernels.virtual_noise",
sections "RNG: fast centered-uniform approximation", "Noise indexing scheme",
and the API entries ``_SPLITMIX64_GAMMA``, ``_cpu_logical_rshift``,
``_splitmix64_step`` and ``_cpu_normal_noise``.

What the page fixes:
  * GAMMA = 11400714819323198485 (``_SPLITMIX64_GAMMA``).
  * The finalizer (``_splitmix64_step``): xor with the state shifted right by
    30, multiply by GAMMA, xor with the result shifted right by 27, multiply by
    GAMMA, xor with the result shifted right by 31; all arithmetic wraps mod
    2**64 and every right shift is logical (``_cpu_logical_rshift`` exists only
    to get logical shifts out of signed torch tensors).
  * The uniform in [0, 1) comes from the LOW 32 bits of the hash and the noise
    is that uniform minus 0.5, a value in [-0.5, 0.5) (``_cpu_normal_noise``).
  * Each noise element is PRNG(seed_i, element_index) with
    element_index = offset + flat_index ("Noise indexing scheme").

Readings taken where the page is silent (each also listed in the design notes):
  R1 state mixing: PRNG(seed, idx) is the idx-th output (counting from 0) of a
     splitmix64 generator seeded with ``seed``: the generator adds GAMMA to its
     state before each output, so the hashed state is
     ``seed + (idx + 1) * GAMMA  (mod 2**64)``.
  R2 finalizer: the formula as printed (GAMMA as both multipliers), not the
     textbook finalizer with two distinct multipliers.
  R3 uniform: keep the top 23 of the low 32 bits, ``u = (lo32 >> 9) * 2**-23``.
     It is exact in float32 and can never round up to 1.0, so the stated range
     [-0.5, 0.5) holds exactly.
  R5 seeds: int32 / int64 seeds are taken as signed integers and reduced mod
     2**64 (two's complement), so a negative seed is well defined.
"""

from __future__ import annotations

import math

import numpy as np

#: ``_SPLITMIX64_GAMMA`` as printed on the page (decimal).
GAMMA = 11400714819323198485
MASK64 = (1 << 64) - 1
MASK32 = (1 << 32) - 1

# ----------------------------------------------------------------------------
# Python-int reference (one element at a time)
# ----------------------------------------------------------------------------


def mix64(z: int) -> int:
    """``_splitmix64_step``: the printed 30/27/31 finalizer, wrapping mod 2**64."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * GAMMA) & MASK64
    z = ((z ^ (z >> 27)) * GAMMA) & MASK64
    z = z ^ (z >> 31)
    return z


def state64(seed: int, idx: int) -> int:
    """Reading R1: the state hashed for element ``idx`` of individual ``seed``."""
    return ((seed & MASK64) + ((idx & MASK64) + 1) * GAMMA) & MASK64


def uniform_from_hash(h: int) -> float:
    """Reading R3: low 32 bits -> top 23 of them -> u in [0, 1), exact."""
    lo32 = h & MASK32
    return (lo32 >> 9) * 2.0 ** -23


def noise(seed: int, idx: int) -> float:
    """Centered-uniform noise PRNG(seed, idx) in [-0.5, 0.5) (``_cpu_normal_noise``)."""
    return uniform_from_hash(mix64(state64(seed, idx))) - 0.5


# ----------------------------------------------------------------------------
# numpy uint64 version (bulk work). numpy's uint64 array multiply wraps mod
# 2**64 and ``>>`` on unsigned arrays is a logical shift.
# ----------------------------------------------------------------------------

_G = np.uint64(GAMMA)
_S30, _S27, _S31, _S9 = (np.uint64(s) for s in (30, 27, 31, 9))
_LO32 = np.uint64(MASK32)


def seeds_u64(seeds) -> np.ndarray:
    """Reading R5: signed int32/int64 seeds -> uint64 (two's complement)."""
    a = np.asarray(seeds)
    if a.dtype.kind == "u":
        return a.astype(np.uint64)
    return a.astype(np.int64).view(np.uint64)


def mix64_np(z: np.ndarray) -> np.ndarray:
    """Vectorised ``_splitmix64_step`` on a uint64 array."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> _S30)) * _G
        z = (z ^ (z >> _S27)) * _G
        z = z ^ (z >> _S31)
    return z


def state64_np(seed_u64: np.ndarray, idx_u64: np.ndarray) -> np.ndarray:
    """Reading R1, vectorised with broadcasting: seed + (idx + 1) * GAMMA."""
    with np.errstate(over="ignore"):
        return seed_u64 + (idx_u64 + np.uint64(1)) * _G


def noise_np(seed_u64: np.ndarray, idx_u64: np.ndarray) -> np.ndarray:
    """Noise values (float64, each exactly representable in float32)."""
    h = mix64_np(state64_np(seed_u64, idx_u64))
    m = (h & _LO32) >> _S9
    return m.astype(np.float64) * 2.0 ** -23 - 0.5


def element_indices(offset: int, n: int) -> np.ndarray:
    """``offset + t`` for t in [0, n), as uint64, wrapping mod 2**64."""
    off = np.uint64(offset & MASK64)
    with np.errstate(over="ignore"):
        return off + np.arange(n, dtype=np.uint64)


# ----------------------------------------------------------------------------
# Gaussian variant (reading R16). The page's forward docstring calls the noise
# "Gaussian" while its RNG section uses a centered uniform and names Box-Muller
# as the costly alternative. The variant takes both 32-bit halves of the same
# finalizer output z as two uniforms and applies Box-Muller:
#   u1 = 1 - (hi32(z) >> 9) * 2**-23   in (0, 1]   (never 0: the log is finite)
#   u2 = (lo32(z) >> 9) * 2**-23       in [0, 1)   (the uniform variant's u)
#   g  = sqrt(-2 ln u1) * cos(2 pi u2)
# ----------------------------------------------------------------------------


def gaussian_from_hash(h: int) -> float:
    """Box-Muller on the halves of one finalizer output (reading R16), float64."""
    u1 = 1.0 - ((h >> 32) >> 9) * 2.0 ** -23
    u2 = ((h & MASK32) >> 9) * 2.0 ** -23
    return math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)


def gaussian_noise(seed: int, idx: int) -> float:
    """Gaussian-variant noise for element ``idx`` of individual ``seed``."""
    return gaussian_from_hash(mix64(state64(seed, idx)))


def gaussian_noise_np(seed_u64: np.ndarray, idx_u64: np.ndarray) -> np.ndarray:
    """Gaussian-variant noise values, float64, vectorised."""
    h = mix64_np(state64_np(seed_u64, idx_u64))
    u1 = 1.0 - ((h >> np.uint64(32)) >> _S9).astype(np.float64) * 2.0 ** -23
    u2 = ((h & _LO32) >> _S9).astype(np.float64) * 2.0 ** -23
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
