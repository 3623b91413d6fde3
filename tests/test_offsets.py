"""The library's ``compute_offsets`` (host code of the binding) pinned without a GPU.

EvoX API page "evox.triton_kernels.kernels.virtual_noise", API entry
``compute_offsets`` and its "Example": a block's offset is the number of
elements in all blocks before it. The GPU parity tests feed the library's
offsets to both the kernels and the oracle, so a mistake here (end offsets
instead of start offsets, a dropped block, a shape read as its first
dimension) would pass every one of them; these tests compare the library's
function with the page's printed example, with the oracle's own
``compute_offsets`` and with the offsets the ES policy workload is built on.
"""

import json
import math
import os
import random

import pytest

from oracle import es
from virtual_noise_perturbed_gb300 import compute_offsets, workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_matches_the_pages_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "compute_offsets.json")))
    assert compute_offsets([tuple(s) for s in g["param_shapes"]]) == g["offsets"]


def test_policy_layout():
    # 64 -> 256 -> 256 -> 8, weights then bias per layer.
    shapes = [(256, 64), (256,), (256, 256), (256,), (8, 256), (8,)]
    assert compute_offsets(shapes) == [0, 16384, 16640, 82176, 82432, 84480]


@pytest.mark.parametrize("shapes,want", [
    ([], []),
    ([()], [0]),                          # a scalar block holds one element
    ([(), (), (3,)], [0, 1, 2]),
    ([(1,), (1, 1), (1, 1, 1)], [0, 1, 2]),
    ([(0, 5), (4,)], [0, 0]),             # an empty block takes no indices
    ([(7,), (0,), (2, 3)], [0, 7, 7]),
    ([(2, 3, 4)], [0]),
])
def test_hand_worked_cases(shapes, want):
    assert compute_offsets(shapes) == want


def test_agrees_with_the_oracle_on_random_shape_lists():
    rng = random.Random(20261202)
    for _ in range(300):
        n = rng.randrange(0, 12)
        shapes = [tuple(rng.randrange(0, 70) for _ in range(rng.randrange(0, 4))) for _ in range(n)]
        got = compute_offsets(shapes)
        assert got == es.compute_offsets(shapes), shapes
        # and the defining property, block by block
        assert got == [sum(math.prod(s) for s in shapes[:b]) for b in range(n)]


def test_accepts_any_sequence_of_sizes():
    assert compute_offsets([[3, 4], (5,), range(2, 4)]) == [0, 12, 17]
    assert compute_offsets(iter([(2,), (3,)])) == [0, 2]


def test_large_blocks_do_not_overflow():
    shapes = [(1 << 31, 1 << 31), (1 << 20,), (5,)]
    assert compute_offsets(shapes) == [0, 1 << 62, (1 << 62) + (1 << 20)]


def test_workloads_are_laid_out_by_compute_offsets():
    """The layer offsets the policy workload carries (its inputs) are the oracle's
    and the library's compute_offsets over (W_0, b_0, W_1, b_1, ...)."""
    w = workloads.make(2)
    shapes = []
    for l in w.layers:
        shapes += [(l.out_f, l.in_f), (l.out_f,)]
    want = es.compute_offsets(shapes)[0::2]
    assert [l.offset for l in w.layers] == want == compute_offsets(shapes)[0::2] == [0, 16640, 82432]
