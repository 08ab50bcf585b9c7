"""Pins of the oracle's FP8 intermediate blocks (the opt-in low-precision
variant) against what the format and the arithmetic fix, independent of the
oracle's own code: torch's float8_e4m3fn conversion, the E4M3 value grid built
from its bit fields, closed forms of the block scale, and the layer assembled
from the oracle's pinned pieces by a numpy matmul."""
import numpy as np
import pytest
import torch

import oracle
from moe_layer_decode_persistent_b300 import inputs


def e4m3_grid():
    """Every finite non-negative E4M3FN value, from the bit fields: normals
    2^(e-7)(1 + m/8) for e = 1..15 except e = 15, m = 7; subnormals m 2^-9."""
    vals = [m * 2.0 ** -9 for m in range(8)]
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append(2.0 ** (e - 7) * (1 + m / 8))
    return np.array(sorted(vals))


def test_every_e4m3_value_maps_to_itself_and_midpoints_go_to_the_even_code():
    g = e4m3_grid()
    assert g[-1] == 448.0 and len(g) == 127
    for v in g:
        assert oracle.e4m3_rne(v) == v and oracle.e4m3_rne(-v) == -v
    # the midpoint of two neighbours goes to the one with the even mantissa,
    # which is the even position on the grid (every binade holds 8 values)
    for i in range(len(g) - 1):
        mid = (g[i] + g[i + 1]) / 2
        want = g[i] if i % 2 == 0 else g[i + 1]
        assert oracle.e4m3_rne(mid) == want, (g[i], g[i + 1])
    assert oracle.e4m3_rne(1000.0) == 448.0 and oracle.e4m3_rne(-1e9) == -448.0


def test_e4m3_rounding_matches_torch_float8_e4m3fn():
    """Random float32 values across the whole range, including subnormals:
    the oracle's rounding equals torch's float8_e4m3fn conversion."""
    rng = np.random.default_rng(0)
    mag = np.exp(rng.uniform(np.log(1e-4), np.log(440.0), 20000))
    v = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_rne(float(x)) for x in v])
    assert np.array_equal(got, want)


def test_block_scale_is_the_smallest_power_of_two_that_fits_448():
    """Closed forms: values already on the E4M3 grid times 2^k stay put; the
    scale steps up exactly when max|mid| passes 448 * 2^k; zeros stay zero."""
    g = e4m3_grid()
    rng = np.random.default_rng(1)
    for k in (-20, -3, 0, 5):
        blk = rng.choice(g, 32) * 2.0 ** k * rng.choice([-1, 1], 32)
        blk[0] = 448.0 * 2.0 ** k  # max|mid| exactly 448 * 2^k: scale 2^k
        assert np.array_equal(oracle.fp8_mid_blocks(blk), blk)
    # just above 448: the scale doubles, so 449 -> 448 (grid step 32 at 2^1 scale: 224.5 -> 224)
    blk = np.zeros(32)
    blk[3] = 449.0
    blk[4] = 1.0
    q = oracle.fp8_mid_blocks(blk)
    assert q[3] == 448.0 and q[4] == 1.0
    assert np.array_equal(oracle.fp8_mid_blocks(np.zeros(64)), np.zeros(64))
    # each block of 32 has its own scale
    a = np.concatenate([np.full(32, 1e-3), np.full(32, 1e3)])
    qa = oracle.fp8_mid_blocks(a)
    assert np.allclose(qa[:32], 1e-3, rtol=2 ** -4) and np.allclose(qa[32:], 1e3, rtol=2 ** -4)


def test_block_quantisation_error_is_within_half_a_grid_step():
    """Every value moves by at most half an E4M3 step at its block's scale:
    2^-4 relative in the normal range, 2^-10 * 2^k below it."""
    rng = np.random.default_rng(2)
    m = rng.standard_normal(4096) * np.exp(rng.uniform(-8, 8, 4096))
    q = oracle.fp8_mid_blocks(m)
    for b in range(0, m.size, 32):
        blk, qb = m[b:b + 32], q[b:b + 32]
        amax = np.abs(blk).max()
        k = int(np.ceil(np.log2(amax / 448.0)))
        bound = np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** (k - 10))
        assert np.all(np.abs(qb - blk) <= bound * (1 + 1e-12))


@pytest.mark.parametrize("fr,fs", [(inputs.FMT_NVFP4, inputs.FMT_FP8_B128), (inputs.FMT_BF16, inputs.FMT_BF16)])
def test_fp8_mid_layer_equals_the_pieces_assembled_by_numpy(fr, fs):
    """The layer with FP8 intermediate blocks equals x + shared + sum of
    weighted routed experts, each down applied (numpy fp64 matmul) to the
    block-quantised intermediate of that expert use."""
    s = inputs.Shape(T=3, H=256, I=128, I_shared=256, E=6, K=2)
    L = inputs.make_layer(s, "uniform", 4, "cpu", fr, fs)
    routed, shared = [oracle.WeightSet(es.fmt, es.w13, es.w2, es.w13_scale, es.w2_scale, es.w13_gscale,
                                       es.w2_gscale) for es in (L.routed, L.shared)]
    got = oracle.moe_layer_fp8mid(L.x, L.topk_ids, L.topk_w, routed, shared, s.T, s.H, s.I, s.I_shared,
                                  s.E, s.K)
    x = L.x.double().numpy()
    want = x.copy()
    for t in range(s.T):
        for ws, I, e, w in [(shared, s.I_shared, 0, 1.0)] + [(routed, s.I, int(L.topk_ids[t, p]),
                                                               float(L.topk_w[t, p])) for p in range(s.K)]:
            mid, _ = oracle.expert_ffn(ws, s.H, I, e, x[t])
            want[t] += w * (oracle.dequant_w2(ws, s.H, I, e) @ oracle.fp8_mid_blocks(mid))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    exact = oracle.moe_layer(L.x, L.topk_ids, L.topk_w, routed, shared, s.T, s.H, s.I, s.I_shared, s.E, s.K)
    rel = np.abs(got - exact).max() / np.abs(exact - x).max()
    assert 0 < rel < 0.1  # the blocks change the result, by about the E4M3 step
