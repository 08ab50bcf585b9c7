"""Pins for the fp64 oracle: checks against facts that do not come from the
oracle itself -- library decodes (torch, CUDA's host fp4 conversion), weights
built from independently chosen factors, the special case that reduces the
layer to a dense SwiGLU MLP (torch fp64 matmul + F.silu), closed forms,
invariants and brute force over tiny routings. CPU only.
"""
import itertools
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from moe_layer_decode_persistent_b300 import inputs

# ---------------------------------------------------------------- decodes


def test_e4m3_exhaustive_matches_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_exhaustive_matches_torch():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16(b) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


_FP4_HOST = r"""
#include <cstdio>
#include <cuda_fp4.h>
int main() {
  for (int c = 0; c < 16; ++c) {
    __nv_fp4_e2m1 v; v.__x = (__nv_fp4_storage_t)c;
    std::printf("%.9g\n", (double)(float)v);
  }
  return 0;
}
"""


def _cuda_host_e2m1():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available for the CUDA host fp4 decode")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "fp4.cu")
        exe = os.path.join(d, "fp4")
        with open(src, "w") as f:
            f.write(_FP4_HOST)
        subprocess.check_call([nvcc, "-o", exe, src], cwd=d)
        out = subprocess.check_output([exe], text=True)
    return np.array([float(v) for v in out.split()])


def test_e2m1_exhaustive_matches_cuda_host_conversion():
    ref = _cuda_host_e2m1()
    got = np.array([oracle.e2m1(c) for c in range(16)])
    assert np.array_equal(got, ref)
    # the encoder used for inputs is consistent with that decode (nearest value)
    vals = torch.tensor(ref, dtype=torch.float32)
    assert torch.equal(vals[inputs.encode_e2m1(vals).long()], vals)


# ---------------------------------------------------- layouts from factors

_E2M1 = None


def _e2m1_table():
    global _E2M1
    if _E2M1 is None:
        _E2M1 = _cuda_host_e2m1()
    return _E2M1


def _e4m3_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _nvfp4_from_factors(rng, E, rows, cols):
    """Random codes / block-scale bytes / tensor scales and the dense matrix they
    stand for, computed from library decode tables, not from the oracle."""
    codes = rng.integers(0, 16, size=(E, rows, cols), dtype=np.uint8)
    # valid (non-NaN, non-zero) E4M3 scale bytes spread over the exponent range
    sbytes = rng.integers(0x08, 0x7E, size=(E, rows, cols // 16), dtype=np.uint8)
    gs = rng.uniform(0.5, 2.0, size=E).astype(np.float32)
    dense = (_e2m1_table()[codes] * np.repeat(_e4m3_table()[sbytes], 16, axis=2)
             * gs.astype(np.float64)[:, None, None])
    packed = (codes[:, :, 0::2] | (codes[:, :, 1::2] << 4)).astype(np.uint8)
    return packed, sbytes, gs, dense


def _fp8_from_factors(rng, E, rows, cols):
    q = rng.integers(0, 256, size=(E, rows, cols), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    s = rng.uniform(0.25, 4.0, size=(E, rows // 128, cols // 128)).astype(np.float32)
    dense = _e4m3_table()[q] * np.repeat(np.repeat(s.astype(np.float64), 128, 1), 128, 2)
    return q, s, dense


def test_nvfp4_layout_from_factors():
    rng = np.random.default_rng(1)
    E, H, I = 2, 64, 32
    p13, s13, g13, d13 = _nvfp4_from_factors(rng, E, 2 * I, H)
    p2, s2, g2, d2 = _nvfp4_from_factors(rng, E, H, I)
    ws = oracle.WeightSet(oracle.FMT_NVFP4, p13, p2, s13, s2, g13, g2)
    for e in range(E):
        assert np.array_equal(oracle.dequant_w13(ws, H, I, e), d13[e])
        assert np.array_equal(oracle.dequant_w2(ws, H, I, e), d2[e])


def test_fp8_block128_layout_from_factors():
    rng = np.random.default_rng(2)
    E, H, I = 1, 256, 128
    q13, s13, d13 = _fp8_from_factors(rng, E, 2 * I, H)
    q2, s2, d2 = _fp8_from_factors(rng, E, H, I)
    ws = oracle.WeightSet(oracle.FMT_FP8_B128, q13, q2, s13, s2)
    assert np.array_equal(oracle.dequant_w13(ws, H, I, 0), d13[0])
    assert np.array_equal(oracle.dequant_w2(ws, H, I, 0), d2[0])


# ------------------------------------------------ layer: special cases


def _dense_swiglu(x64, w13, w2):
    """Textbook SwiGLU MLP in torch fp64: Wd (silu(Wg x) * (Wu x))."""
    x = torch.from_numpy(x64)
    w13 = torch.from_numpy(w13)
    w2 = torch.from_numpy(w2)
    I = w13.shape[0] // 2
    h = torch.nn.functional.silu(x @ w13[:I].T) * (x @ w13[I:].T)
    return (h @ w2.T).numpy()


def _x_bits(T, H, seed):
    x = inputs.activations(T, H, seed)
    return x, x.double().numpy()


def _zero_shared_bf16(H, Is):
    return oracle.WeightSet(oracle.FMT_BF16, np.zeros((1, 2 * Is, H), np.uint16),
                            np.zeros((1, H, Is), np.uint16))


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4"])
def test_top1_weight1_zero_shared_is_dense_swiglu_mlp(fmt):
    """K=1, router weight 1, shared expert zero: out = x + MLP_e(x)."""
    T, H, I, E = 5, 64, 32, 3
    rng = np.random.default_rng(3)
    if fmt == "bf16":
        ex = inputs.make_experts(inputs.FMT_BF16, E, H, I, 7)
        routed = oracle.WeightSet(oracle.FMT_BF16, ex.w13, ex.w2)
        d13 = ex.w13.double().numpy()
        d2 = ex.w2.double().numpy()
    else:
        p13, s13, g13, d13 = _nvfp4_from_factors(rng, E, 2 * I, H)
        p2, s2, g2, d2 = _nvfp4_from_factors(rng, E, H, I)
        routed = oracle.WeightSet(oracle.FMT_NVFP4, p13, p2, s13, s2, g13, g2)
    shared = _zero_shared_bf16(H, 32)
    x, x64 = _x_bits(T, H, 4)
    ids = np.array([[0], [2], [1], [2], [0]], np.int32)
    w = np.ones((T, 1), np.float32)
    ref = oracle.moe_layer(x, ids, w, routed, shared, T, H, I, 32, E, 1)
    for t in range(T):
        want = x64[t] + _dense_swiglu(x64[t:t + 1], d13[ids[t, 0]], d2[ids[t, 0]])[0]
        np.testing.assert_allclose(ref[t], want, rtol=1e-12, atol=1e-12)


def _small_layer(fmt_r, fmt_s, T=6, routing="uniform", seed=0, H=256, I=128, Is=128, E=8, K=3):
    s = inputs.Shape(T=T, H=H, I=I, I_shared=Is, E=E, K=K)
    return inputs.make_layer(s, routing, seed, "cpu", fmt_r, fmt_s)


def _ws(es):
    return oracle.WeightSet(es.fmt, es.w13, es.w2, es.w13_scale, es.w2_scale,
                            es.w13_gscale, es.w2_gscale)


def _ref(L, **kw):
    s = L.shape
    return oracle.moe_layer(L.x, L.topk_ids, L.topk_w, _ws(L.routed), _ws(L.shared),
                            s.T, s.H, s.I, s.I_shared, s.E, s.K, **kw)


FORMATS = [(inputs.FMT_BF16, inputs.FMT_BF16), (inputs.FMT_NVFP4, inputs.FMT_FP8_B128),
           (inputs.FMT_FP8_B128, inputs.FMT_NVFP4)]


@pytest.mark.parametrize("fmts", FORMATS)
def test_fused_equals_four_step_unfused(fmts):
    L = _small_layer(*fmts)
    s = L.shape
    fused = _ref(L)
    unf = oracle.unfused_layer(L.x, L.topk_ids, L.topk_w, _ws(L.routed), _ws(L.shared),
                               s.T, s.H, s.I, s.I_shared, s.E, s.K)
    np.testing.assert_allclose(fused, unf, rtol=1e-12, atol=1e-12)


def test_zero_activations_give_zero_output():
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    L.x.zero_()
    assert np.array_equal(_ref(L), np.zeros((L.shape.T, L.shape.H)))


def test_zero_down_weights_give_residual_exactly():
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    L.routed.w2.zero_()
    L.shared.w2.zero_()
    assert np.array_equal(_ref(L), L.x.double().numpy())


def test_routed_part_is_linear_in_router_weights():
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    w0 = L.topk_w.clone()
    L.topk_w = torch.zeros_like(w0)
    base = _ref(L)
    L.topk_w = w0
    fa = _ref(L) - base
    L.topk_w = 2.0 * w0
    f2 = _ref(L) - base
    np.testing.assert_allclose(f2, 2.0 * fa, rtol=1e-9, atol=1e-11)


def test_down_tensor_scale_scales_routed_part():
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    L0 = torch.zeros_like(L.topk_w)
    w0 = L.topk_w
    L.topk_w = L0
    base = _ref(L)
    L.topk_w = w0
    fa = _ref(L) - base
    L.routed.w2_gscale.mul_(2.0)
    f2 = _ref(L) - base
    np.testing.assert_allclose(f2, 2.0 * fa, rtol=1e-12, atol=1e-12)


def test_duplicate_rows_give_identical_outputs():
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    L.x[3] = L.x[1]
    L.topk_ids[3] = L.topk_ids[1]
    L.topk_w[3] = L.topk_w[1]
    r = _ref(L)
    assert np.array_equal(r[3], r[1])


def test_row_permutation_permutes_outputs():
    L = _small_layer(inputs.FMT_BF16, inputs.FMT_BF16)
    r = _ref(L)
    perm = torch.tensor([4, 2, 0, 5, 1, 3])
    L.x, L.topk_ids, L.topk_w = L.x[perm], L.topk_ids[perm], L.topk_w[perm]
    assert np.array_equal(_ref(L), r[perm.numpy()])


def test_row_subset_matches_full_rows():
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    full = _ref(L)
    sub = _ref(L, rows=np.array([5, 0, 3], np.int32), threads=2)
    assert np.array_equal(sub, full[[5, 0, 3]])


def test_uses_in_parallel_equal_rows_bit_for_bit():
    """The form that runs a row's expert evaluations on separate threads (the
    one the reference arm times) is the row-by-row form, rescheduled."""
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    L.topk_ids[1, 0] = L.shape.E + 1  # an out-of-range pick adds nothing in both
    s = L.shape
    args = (L.x, L.topk_ids, L.topk_w, _ws(L.routed), _ws(L.shared), s.T, s.H, s.I, s.I_shared, s.E, s.K)
    full = oracle.moe_layer(*args)
    for threads in (1, 3):
        assert np.array_equal(oracle.moe_layer_uses(*args, threads=threads), full)
    rows = np.array([4, 1], np.int32)
    assert np.array_equal(oracle.moe_layer_uses(*args, rows=rows, threads=2), full[rows])


# ------------------------------------------------ negative controls


def test_shared_expert_is_not_silently_dropped():
    L = _small_layer(inputs.FMT_NVFP4, inputs.FMT_FP8_B128)
    r = _ref(L)
    L.shared.w2.zero_()
    r0 = _ref(L)
    assert np.all(np.any(r != r0, axis=1))


def test_gate_and_up_are_not_interchangeable():
    L = _small_layer(inputs.FMT_BF16, inputs.FMT_BF16)
    r = _ref(L)
    I = L.shape.I
    L.routed.w13 = torch.cat([L.routed.w13[:, I:], L.routed.w13[:, :I]], dim=1).contiguous()
    assert not np.allclose(_ref(L), r)


def test_out_of_range_pick_contributes_nothing():
    L = _small_layer(inputs.FMT_BF16, inputs.FMT_BF16)
    L.topk_ids[2, 1] = L.shape.E + 3
    r = _ref(L)
    L.topk_w[2, 1] = 0.0
    L.topk_ids[2, 1] = 0
    assert np.array_equal(_ref(L)[2], r[2])


# ------------------------------------------------ group table, brute force


def _check_table(ids, T, K, E, flags):
    table, err = oracle.group_table(ids, T, K, E, flags)
    f = oracle.unpack_table(table, T, K)
    G, U = f["G"], f["U"]
    gexp, gn, g0 = f["group_expert"], f["group_ncols"], f["group_col0"]
    crow, rcol = f["col_row"], f["row_col"]
    valid = [(t, p) for t in range(T) for p in range(K) if 0 <= ids[t][p] < E]
    distinct = []
    for t, p in valid:
        if ids[t][p] not in distinct:
            distinct.append(ids[t][p])
    assert U == T + len(valid)
    if flags & oracle.FLAG_NO_DEDUP:
        assert G == U and list(gn[:G]) == [1] * G
    else:
        assert G == 1 + len(distinct)
        assert gexp[0] == -1 and gn[0] == T
        assert list(gexp[1:G]) == distinct  # distinct, in order of first use
    assert list(g0[:G]) == list(np.cumsum([0] + list(gn[:G - 1]))) if G else True
    assert sum(gn[:G]) == U
    # every column used exactly once, each in the right group, right row
    group_of = np.repeat(np.arange(G), gn[:G])
    seen = []
    for t in range(T):
        c = rcol[t, 0]
        assert gexp[group_of[c]] == -1 and crow[c] == t
        seen.append(c)
        for p in range(K):
            c = rcol[t, 1 + p]
            if 0 <= ids[t][p] < E:
                assert gexp[group_of[c]] == ids[t][p] and crow[c] == t
                seen.append(c)
            else:
                assert c == -1
    assert sorted(seen) == list(range(U))
    # columns inside a group follow (row, slot) order
    key = {}
    for t in range(T):
        for slot in range(K + 1):
            c = rcol[t, slot]
            if c >= 0:
                key[c] = (t, slot)
    for g in range(G):
        ks = [key[c] for c in range(g0[g], g0[g] + gn[g])]
        assert ks == sorted(ks)
    # untouched entries are zero
    C = T * (K + 1)
    for name, n in (("group_expert", G), ("group_ncols", G), ("group_col0", G), ("col_row", U)):
        assert not np.any(f[name][n:C])
    bad = any(not (0 <= ids[t][p] < E) for t in range(T) for p in range(K))
    dup = any(ids[t][p] == ids[t][q] and 0 <= ids[t][p] < E
              for t in range(T) for p in range(K) for q in range(p))
    assert bool(err & oracle.ERR_BAD_EXPERT) == bad
    assert bool(err & oracle.ERR_DUP_EXPERT) == dup


@pytest.mark.parametrize("flags", [0, oracle.FLAG_NO_DEDUP])
def test_group_table_brute_force_all_tiny_routings(flags):
    n = 0
    for T, K, E in [(1, 1, 1), (1, 2, 3), (2, 1, 3), (2, 2, 3), (3, 2, 2), (3, 1, 4), (2, 2, 4), (3, 2, 3)]:
        for flat in itertools.product(range(E), repeat=T * K):
            ids = [list(flat[t * K:(t + 1) * K]) for t in range(T)]
            _check_table(ids, T, K, E, flags)
            n += 1
    # out-of-range ids, negative and too large
    for ids in ([[-1, 0]], [[0, 5], [5, 0]], [[2, 2], [-7, 1]]):
        _check_table(ids, len(ids), 2, 3, flags)
    assert n > 1000


def test_group_table_t0_is_empty():
    table, err = oracle.group_table(np.zeros((0, 4), np.int32), 0, 4, 8)
    assert table[0] == 0 and table[1] == 0 and err == 0


@pytest.mark.parametrize("routing", ["uniform", "mtp", "zipf"])
def test_group_table_on_workload_routings(routing):
    T, K, E = 8, 8, 256
    ids = inputs.ROUTINGS[routing](T, K, E, 0).numpy()
    _check_table(ids.tolist(), T, K, E, 0)
    _check_table(ids.tolist(), T, K, E, oracle.FLAG_NO_DEDUP)


# ------------------------------------------------ tolerance helper


def test_tolerance_rule():
    ref = np.array([1.0, -2.0, 0.0, 4.0])
    rms = np.sqrt(np.mean(ref ** 2))
    ok, _ = oracle.tolerance_ok(ref + 2 ** -7 * np.abs(ref) + 0.999e-3 * rms, ref)
    assert ok
    bad = ref.copy()
    bad[2] += 1.01e-3 * rms
    ok, ratio = oracle.tolerance_ok(bad, ref)
    assert not ok and ratio > 1.0
