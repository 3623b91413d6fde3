"""GPU parity of the hash-only measurement kernel (vn_hash_probe) against the oracle.

sums[t] = sum_{e < m} PRNG(seed, offset + t*m + e): the oracle side is its noise dump
of the whole index range (bit-exact to the library's dump, pinned elsewhere), cut into
rows of m and summed in float64. The kernel adds in fp32 as two partial sums (even e
and odd e, each in order of e) and then adds those. The noise values are exact in fp32
and each addition rounds by at most 2^-24 of its result, so each sum is within
m * 2^-24 * (largest even partial sum + largest odd partial sum + 1) of the exact one."""

import numpy as np
import pytest
import torch

from oracle import es
from virtual_noise_perturbed_gb300 import VNError, hash_probe
from virtual_noise_perturbed_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def _want(seed, offset, ts, m):
    rows = []
    bounds = []
    for t in ts:
        d = es.noise_dump(np.array([seed], dtype=np.int64), m, (offset + t * m) % (1 << 64))[0]
        d = d.astype(np.float64)
        rows.append(float(np.sum(d)) if m else 0.0)
        ev, od = np.cumsum(d[0::2]), np.cumsum(d[1::2])
        big = (np.max(np.abs(ev)) if ev.size else 0.0) + (np.max(np.abs(od)) if od.size else 0.0)
        bounds.append(m * 2.0 ** -24 * (big + 1.0))
    return np.array(rows), np.array(bounds)


@pytest.mark.parametrize("seed,offset,n_sums,m", [
    (0, 0, 1, 1),
    (7, 0, 3, 0),                          # empty runs: zeros
    (-3, (1 << 64) - 5, 5, 3),             # indices wrap mod 2^64
    (123, 1 << 32, 300, 37),               # ragged: m not a multiple of the unroll
    (2 ** 62 + 1, 999, 257, 4096),         # two CTAs and one thread more
])
def test_probe_matches_the_oracle(seed, offset, n_sums, m):
    got = hash_probe(seed, offset, n_sums, m, device=DEV).cpu().numpy().astype(np.float64)
    want, bound = _want(seed, offset, range(n_sums), m)
    assert np.all(np.abs(got - want) <= bound), np.max(np.abs(got - want) - bound)


def test_probe_at_the_bench_size_on_sampled_sums():
    """The launch the bench times: 152 SMs x 2048 threads x 4 rounds of sums, 4096
    elements each; sums at both ends and 14 drawn at random against the oracle."""
    n_sums, m, seed, offset = 152 * 2048 * 4, 4096, 1, 0
    got = hash_probe(seed, offset, n_sums, m, device=DEV).cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(5)
    ts = sorted({0, 1, n_sums - 1} | set(rng.integers(2, n_sums - 1, 14).tolist()))
    want, bound = _want(seed, offset, ts, m)
    assert np.all(np.abs(got[ts] - want) <= bound)
    # a property at any size: the sums of a centered uniform stay near 0 (|mean| of
    # 1.2e6 sums with standard deviation sqrt(m/12) ~ 18.5 is below 5 standard errors)
    assert abs(got.mean()) < 5 * np.sqrt(m / 12) / np.sqrt(n_sums)


def test_probe_refusals():
    s = torch.empty(4, device=DEV)
    with pytest.raises(VNError, match="SHAPE"):
        hash_probe(0, 0, 4, -1, out=s)
    with pytest.raises(VNError, match="OVERFLOW"):
        hash_probe(0, 0, 4, 1 << 62, out=s)
