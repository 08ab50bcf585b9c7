"""The oracle reproduces the stored tiny-layer values (see tests/golden/make_golden.py)."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "golden"))
import make_golden  # noqa: E402


def _load():
    d = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_seed0.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            k, *v = line.split()
            d[k] = v
    return d


def test_tiny_layer_matches_stored_values():
    g = _load()
    L, ref, table, err = make_golden.tiny_reference()
    assert [int(v) for v in g["topk_ids"]] == L.topk_ids.reshape(-1).tolist()
    assert [int(v) for v in g["group_table"]] == table.tolist()
    assert int(g["error_bits"][0]) == err
    for t in range(ref.shape[0]):
        stored = np.array([float(v) for v in g[f"ref_row{t}"]])
        np.testing.assert_allclose(ref[t], stored, rtol=1e-13, atol=1e-13)
