"""moe_group_table on the GPU against the oracle's group table: bit-exact,
including the error bits, on exhaustive tiny routings and workload routings."""
import itertools

import numpy as np
import pytest

import oracle
from moe_layer_decode_persistent_b300 import inputs

from gpu_util import group_table_gpu

pytestmark = pytest.mark.gpu


def _same(ids, T, K, E, flags):
    got, gerr = group_table_gpu(ids, T, K, E, flags)
    want, werr = oracle.group_table(np.asarray(ids, np.int32).reshape(-1), T, K, E, flags)
    assert np.array_equal(got, want), (ids, flags)
    assert gerr == werr, (ids, flags, gerr, werr)


@pytest.mark.parametrize("flags", [0, oracle.FLAG_NO_DEDUP])
def test_exhaustive_tiny_routings(flags):
    for T, K, E in [(1, 1, 1), (1, 2, 3), (2, 2, 3), (3, 2, 2), (3, 1, 4), (2, 2, 4)]:
        for flat in itertools.product(range(E), repeat=T * K):
            _same(list(flat), T, K, E, flags)


@pytest.mark.parametrize("flags", [0, oracle.FLAG_NO_DEDUP])
def test_out_of_range_and_repeated_ids(flags):
    for ids, K, E in (([-1, 0], 2, 3), ([0, 5, 5, 0], 2, 3), ([2, 2, -7, 1], 2, 3),
                      ([7, 7, 7, 7, 7, 7], 3, 4)):
        _same(ids, len(ids) // K, K, E, flags)


@pytest.mark.parametrize("T,K,E,routing", [(1, 8, 256, "uniform"), (8, 8, 256, "mtp"),
                                           (64, 8, 256, "zipf"), (256, 8, 384, "uniform"),
                                           (37, 6, 160, "zipf"), (5, 16, 1024, "uniform")])
@pytest.mark.parametrize("flags", [0, oracle.FLAG_NO_DEDUP])
def test_workload_routings(T, K, E, routing, flags):
    for seed in range(3):
        ids = inputs.ROUTINGS[routing](T, K, E, seed).numpy().reshape(-1)
        _same(ids, T, K, E, flags)


def test_zero_rows():
    _same([], 0, 8, 256, 0)
