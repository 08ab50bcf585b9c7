"""Writes the stored expected values under tests/golden/.

The pages print no worked numeric example for this layer, so the fixtures here
are values computed by the fp64 oracle (and only by it) on seeded inputs:
they guard the oracle's arithmetic against accidental change. Run from the
repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from moe_layer_decode_persistent_b300 import inputs  # noqa: E402


def _ws(es):
    return oracle.WeightSet(es.fmt, es.w13, es.w2, es.w13_scale, es.w2_scale,
                            es.w13_gscale, es.w2_gscale)


def tiny_reference():
    L = inputs.make_tiny(seed=0)
    s = L.shape
    ref = oracle.moe_layer(L.x, L.topk_ids, L.topk_w, _ws(L.routed), _ws(L.shared),
                           s.T, s.H, s.I, s.I_shared, s.E, s.K)
    table, err = oracle.group_table(L.topk_ids, s.T, s.K, s.E)
    return L, ref, table, err


def main():
    L, ref, table, err = tiny_reference()
    path = os.path.join(HERE, "tiny_seed0.txt")
    with open(path, "w") as f:
        f.write("# tiny all-bf16 layer, seed 0: T=4 H=256 I=128 E=8 K=2 shared I=128\n")
        f.write("# written by tests/golden/make_golden.py from the fp64 oracle\n")
        f.write("topk_ids " + " ".join(str(int(v)) for v in L.topk_ids.reshape(-1)) + "\n")
        f.write("group_table " + " ".join(str(int(v)) for v in table) + "\n")
        f.write(f"error_bits {err}\n")
        for t in range(ref.shape[0]):
            f.write(f"ref_row{t} " + " ".join(repr(float(v)) for v in ref[t]) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
