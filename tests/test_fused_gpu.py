"""The fused layer on the GPU (through the C ABI) against the fp64 oracle,
plus the invariants the method promises: dedup bitwise equal to the one-row
form, determinism, duplicate rows, row permutation, negative controls,
device error bits and the bounded waits."""
import numpy as np
import pytest
import torch

from moe_layer_decode_persistent_b300 import binding as B
from moe_layer_decode_persistent_b300 import inputs

from gpu_util import (assert_parity, layer, oracle_ref, run_fused, shape_of, workspace)

pytestmark = pytest.mark.gpu

PATHS = {"fma": B.MOE_FLAG_FORCE_FMA, "mma": B.MOE_FLAG_FORCE_MMA, "auto": 0}

SMALL = inputs.Shape(T=5, H=512, I=256, I_shared=512, E=16, K=4)
FORMATS = {"nvfp4/fp8": (inputs.FMT_NVFP4, inputs.FMT_FP8_B128),
           "fp8/nvfp4": (inputs.FMT_FP8_B128, inputs.FMT_NVFP4),
           "bf16/bf16": (inputs.FMT_BF16, inputs.FMT_BF16)}


@pytest.mark.parametrize("path", ["fma", "auto"])
def test_tiny_bf16_layer(path):
    L = inputs.make_tiny(0, "cuda")
    out = run_fused(L, PATHS[path])
    assert_parity(out, oracle_ref(L))


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("fmt", list(FORMATS))
@pytest.mark.parametrize("T", [1, 3, 5, 13])
def test_small_layers_all_formats(path, fmt, T):
    if path == "mma" and fmt == "bf16/bf16":
        pytest.skip("bf16 weights run on the CUDA-core path")
    s = inputs.Shape(T=T, H=SMALL.H, I=SMALL.I, I_shared=SMALL.I_shared, E=SMALL.E, K=SMALL.K)
    L = layer(s, "zipf", seed=T, fr=FORMATS[fmt][0], fs=FORMATS[fmt][1], used_only=False)
    out = run_fused(L, PATHS[path])
    assert_parity(out, oracle_ref(L))


@pytest.mark.parametrize("path", list(PATHS))
def test_non_power_of_two_k(path):
    s = inputs.Shape(T=7, H=256, I=256, I_shared=512, E=12, K=6)
    L = layer(s, "mtp", seed=1, used_only=False)
    assert_parity(run_fused(L, PATHS[path]), oracle_ref(L))


@pytest.mark.parametrize("path", list(PATHS))
def test_dsv3_t1_uniform_full(path):
    L = layer(inputs.dsv3(1), "uniform", seed=0)
    assert_parity(run_fused(L, PATHS[path]), oracle_ref(L))


@pytest.mark.parametrize("path", list(PATHS))
def test_dsv3_t8_mtp_full(path):
    L = layer(inputs.dsv3(8), "mtp", seed=0)
    assert_parity(run_fused(L, PATHS[path]), oracle_ref(L))


@pytest.fixture(scope="module")
def dsv3_t64():
    """DSv3 T=64 Zipf layer and its fp64 oracle output on every row."""
    L = layer(inputs.dsv3(64), "zipf", seed=0)
    return L, oracle_ref(L)


@pytest.mark.parametrize("path", list(PATHS))
def test_dsv3_t64_zipf_all_rows(path, dsv3_t64):
    L, ref = dsv3_t64
    out = run_fused(L, PATHS[path])
    assert_parity(out, ref)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("T", [65, 200])
def test_small_layers_beyond_64_rows(path, T):
    """Above 64 rows the tensor path keeps its per-group tables at the group
    capacity (shared + min(E, T*K) experts), not at T*(K+1)."""
    s = inputs.Shape(T=T, H=SMALL.H, I=SMALL.I, I_shared=SMALL.I_shared, E=SMALL.E, K=SMALL.K)
    L = layer(s, "zipf", seed=T, used_only=False)
    out = run_fused(L, PATHS[path])
    assert_parity(out, oracle_ref(L))
    one_row = run_fused(L, PATHS[path] | B.MOE_FLAG_NO_DEDUP)
    assert torch.equal(out.view(torch.int16), one_row.view(torch.int16))


@pytest.fixture(scope="module")
def wide_t256():
    """Wide-expert layer: E=384 top-8, T=256 uniform rows (about 380 distinct)."""
    return layer(inputs.dsv3(256, E=384), "uniform", seed=0)


WIDE_ROWS = [int(r) for r in np.linspace(0, 255, 32).round()]


@pytest.fixture(scope="module")
def wide_t256_ref(wide_t256):
    return oracle_ref(wide_t256, rows=WIDE_ROWS)


@pytest.mark.parametrize("path", ["mma", "auto"])
def test_wide_expert_T256_32_spread_rows(path, wide_t256, wide_t256_ref):
    out = run_fused(wide_t256, PATHS[path])
    assert_parity(out, wide_t256_ref, rows=WIDE_ROWS)
    assert torch.isfinite(out.float()).all()


def test_wide_expert_T256_dedup_is_bitwise_equal_to_one_row_form(wide_t256):
    a = run_fused(wide_t256, PATHS["mma"])
    b = run_fused(wide_t256, PATHS["mma"] | B.MOE_FLAG_NO_DEDUP)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("case", ["small_zipf_T13", "dsv3_T8_mtp", "dsv3_T64_zipf"])
def test_dedup_is_bitwise_equal_to_one_row_form(path, case):
    if case == "small_zipf_T13":
        s = inputs.Shape(T=13, H=512, I=256, I_shared=512, E=16, K=4)
        L = layer(s, "zipf", seed=2, used_only=False)
    elif case == "dsv3_T8_mtp":
        L = layer(inputs.dsv3(8), "mtp", seed=1)
    else:
        L = layer(inputs.dsv3(64), "zipf", seed=1)
    a = run_fused(L, PATHS[path])
    b = run_fused(L, PATHS[path] | B.MOE_FLAG_NO_DEDUP)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("path", list(PATHS))
def test_repeat_launches_are_identical(path):
    L = layer(inputs.dsv3(8), "mtp", seed=3)
    ws = workspace(L)
    a = run_fused(L, PATHS[path], ws=ws)
    for _ in range(3):
        b = run_fused(L, PATHS[path], ws=ws)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_paths_and_shapes_take_turns_on_one_workspace():
    # The tensor-core kernel keeps launch-wide counters in two sets used by
    # alternate launches, in a region the CUDA-core kernel never writes; a
    # workspace sized for T=8 also serves T=1. Interleave all of it on one
    # workspace and compare with fresh workspaces, bit for bit.
    L8 = layer(inputs.dsv3(8), "mtp", seed=5)
    L1 = layer(inputs.dsv3(1), "uniform", seed=6)
    ws = workspace(L8)
    ref = {(n, p): run_fused(L, PATHS[p]) for n, L in (("t8", L8), ("t1", L1)) for p in ("mma", "fma")}
    order = [("t8", "mma"), ("t8", "fma"), ("t8", "mma"), ("t1", "mma"), ("t1", "fma"), ("t8", "mma"),
             ("t1", "mma"), ("t1", "mma"), ("t8", "fma"), ("t8", "mma")]
    for n, p in order:
        out = run_fused(L8 if n == "t8" else L1, PATHS[p], ws=ws)
        assert torch.equal(out.view(torch.int16), ref[(n, p)].view(torch.int16)), (n, p)


def test_k_and_intermediate_changes_take_turns_on_one_workspace():
    """Launches of different K, I and I_shared (and both paths) on one
    workspace sized for the largest of them give the results of fresh
    workspaces, bit for bit: the tensor path's counters sit at fixed offsets
    that no shape's scratch covers."""
    shapes = {"k8": inputs.Shape(T=16, H=512, I=256, I_shared=512, E=16, K=8),
              "k4": inputs.Shape(T=16, H=512, I=256, I_shared=512, E=16, K=4),
              "i512": inputs.Shape(T=8, H=512, I=512, I_shared=256, E=16, K=8),
              "t3": inputs.Shape(T=3, H=512, I=256, I_shared=256, E=16, K=5)}
    Ls = {n: layer(s, "zipf", seed=i + 20, used_only=False) for i, (n, s) in enumerate(shapes.items())}
    nbytes = max(B.moe_workspace_bytes(shape_of(L)) for L in Ls.values())
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    B.moe_workspace_init(ws)
    ref = {(n, p): run_fused(L, PATHS[p]) for n, L in Ls.items() for p in ("mma", "fma")}
    order = [("k8", "mma"), ("k4", "mma"), ("k8", "mma"), ("i512", "mma"), ("k8", "fma"), ("k8", "mma"),
             ("t3", "mma"), ("k4", "fma"), ("i512", "mma"), ("k8", "mma"), ("t3", "fma"), ("k4", "mma")]
    for n, p in order:
        out = run_fused(Ls[n], PATHS[p], ws=ws)
        assert torch.equal(out.view(torch.int16), ref[(n, p)].view(torch.int16)), (n, p)


@pytest.mark.parametrize("path", list(PATHS))
def test_duplicate_rows_and_permutation(path):
    s = inputs.Shape(T=9, H=512, I=256, I_shared=512, E=16, K=4)
    L = layer(s, "uniform", seed=4, used_only=False)
    L.x[5] = L.x[2]
    L.topk_ids[5] = L.topk_ids[2]
    L.topk_w[5] = L.topk_w[2]
    out = run_fused(L, PATHS[path])
    assert torch.equal(out[5].view(torch.int16), out[2].view(torch.int16))
    perm = torch.randperm(9, generator=torch.Generator().manual_seed(0)).cuda()
    L.x, L.topk_ids, L.topk_w = L.x[perm].contiguous(), L.topk_ids[perm].contiguous(), \
        L.topk_w[perm].contiguous()
    out2 = run_fused(L, PATHS[path])
    assert torch.equal(out2.view(torch.int16), out[perm].view(torch.int16))


@pytest.mark.parametrize("path", list(PATHS))
def test_negative_controls(path):
    """Each perturbation changes exactly the outputs that depend on it."""
    s = inputs.Shape(T=6, H=512, I=256, I_shared=512, E=16, K=4)
    L = layer(s, "uniform", seed=5, used_only=False)
    base = run_fused(L, PATHS[path]).view(torch.int16).clone()

    def rows_changed(out):
        return set(torch.nonzero((out.view(torch.int16) != base).any(dim=1)).flatten().tolist())

    # one activation value negated: only its row
    L.x[3, 100] = -L.x[3, 100]
    assert rows_changed(run_fused(L, PATHS[path])) == {3}
    L.x[3, 100] = -L.x[3, 100]
    # the down tensor scale of a routed expert that only some rows use
    e = int(L.topk_ids[0, 0])
    users = {t for t in range(s.T) if e in L.topk_ids[t].tolist()}
    assert users != set(range(s.T))
    L.routed.w2_gscale[e] *= 4.0
    assert rows_changed(run_fused(L, PATHS[path])) == users
    L.routed.w2_gscale[e] /= 4.0
    # the shared expert zeroed: every row (the silently dropped shared expert)
    saved = L.shared.w2.clone()
    L.shared.w2.zero_()
    assert rows_changed(run_fused(L, PATHS[path])) == set(range(s.T))
    L.shared.w2.copy_(saved)
    assert rows_changed(run_fused(L, PATHS[path])) == set()


ROW_SCALES = [1e-30, 1e-6, 1.0, 1e3, 1e6, 1e12, 1e15]


@pytest.mark.parametrize("path", list(PATHS))
def test_activation_rows_from_tiny_to_huge(path):
    """Rows whose magnitudes span 1e-30 to 1e15 (the output grows like |x|^2,
    so 1e15 is near the top of what bf16 can hold): every row matches the
    oracle within the tolerance taken over that row alone, no device error bit
    is set, and dedup stays bitwise equal to the one-row form."""
    s = inputs.Shape(T=len(ROW_SCALES), H=512, I=256, I_shared=512, E=16, K=4)
    L = layer(s, "uniform", seed=14, used_only=False)
    sc = torch.tensor(ROW_SCALES, dtype=torch.float64, device="cuda")[:, None]
    L.x = (L.x.double() * sc).to(torch.bfloat16)
    out = run_fused(L, PATHS[path])  # asserts the device error word is 0
    ref = oracle_ref(L)
    got = out.float().cpu().double().numpy()
    for r in range(s.T):
        assert_parity(out[r:r + 1], ref[r:r + 1])
    assert np.isfinite(got).all()
    one_row = run_fused(L, PATHS[path] | B.MOE_FLAG_NO_DEDUP)
    assert torch.equal(out.view(torch.int16), one_row.view(torch.int16))


@pytest.mark.parametrize("path", list(PATHS))
def test_zero_down_weights_give_residual(path):
    s = inputs.Shape(T=4, H=256, I=256, I_shared=256, E=8, K=2)
    L = layer(s, "uniform", seed=6, used_only=False)
    L.routed.w2.zero_()
    L.shared.w2.zero_()
    out = run_fused(L, PATHS[path])
    assert torch.equal(out.view(torch.int16), L.x.view(torch.int16))


# H, I and I_shared multiples of 256: the tensor-core path is eligible
ELIGIBLE = inputs.Shape(T=4, H=512, I=256, I_shared=256, E=8, K=2)


@pytest.mark.parametrize("path", list(PATHS))
def test_bad_and_repeated_ids_set_error_bits(path):
    """An id outside [0, E) sets MOE_DEV_BAD_EXPERT and adds nothing; an id
    repeated within a row sets MOE_DEV_DUP_EXPERT and both uses count. Each is
    checked against the oracle, and the dedup form stays bitwise equal to the
    one-row form."""
    L = layer(ELIGIBLE, "uniform", seed=7, used_only=False)
    ref_ok = oracle_ref(L)
    L.topk_ids[1, 1] = 99
    L.topk_ids[2, 0] = -1
    ws = workspace(L)
    out = run_fused(L, PATHS[path], ws=ws, check_err=False)
    assert B.moe_read_error(ws) == B.MOE_DEV_BAD_EXPERT
    ref = oracle_ref(L)
    assert_parity(out, ref)
    assert not np.array_equal(ref[1], ref_ok[1]) and not np.array_equal(ref[2], ref_ok[2])
    one_row = run_fused(L, PATHS[path] | B.MOE_FLAG_NO_DEDUP, ws=ws, check_err=False)
    assert B.moe_read_error(ws) == B.MOE_DEV_BAD_EXPERT
    assert torch.equal(out.view(torch.int16), one_row.view(torch.int16))
    L.topk_ids[1, 1] = L.topk_ids[1, 0]
    L.topk_ids[2, 0] = L.topk_ids[2, 1]
    out = run_fused(L, PATHS[path], ws=ws, check_err=False)
    assert B.moe_read_error(ws) == B.MOE_DEV_DUP_EXPERT
    assert_parity(out, oracle_ref(L))
    one_row = run_fused(L, PATHS[path] | B.MOE_FLAG_NO_DEDUP, ws=ws, check_err=False)
    assert B.moe_read_error(ws) == B.MOE_DEV_DUP_EXPERT
    assert torch.equal(out.view(torch.int16), one_row.view(torch.int16))


@pytest.mark.parametrize("path", ["fma", "mma"])
def test_dropped_arrival_times_out_and_workspace_recovers(path):
    """Fault injection on the host side of the protocol: one CTA skips an
    arrival (CUDA-core kernel: a grid barrier arrival; tensor-core kernel: an
    intermediate-ready arrival), the waits on it run out after their budget and
    set the timeout bit, every role stops and frees what it holds; the context
    stays usable and a re-initialised workspace gives the same output as a
    fresh one."""
    s = ELIGIBLE if path == "mma" else inputs.Shape(T=2, H=256, I=128, I_shared=128, E=8, K=2)
    L = layer(s, "uniform", seed=8, used_only=False)
    ws = workspace(L)
    run_fused(L, PATHS[path] | B.MOE_FLAG_DEBUG_DROP_ARRIVE, ws=ws, check_err=False)
    assert B.moe_read_error(ws) & B.MOE_DEV_WAIT_TIMEOUT
    B.moe_workspace_init(ws)
    out = run_fused(L, PATHS[path], ws=ws)
    assert_parity(out, oracle_ref(L))
    fresh = run_fused(L, PATHS[path])
    assert torch.equal(out.view(torch.int16), fresh.view(torch.int16))
    # and the workspace serves later launches too
    again = run_fused(L, PATHS[path], ws=ws)
    assert torch.equal(again.view(torch.int16), fresh.view(torch.int16))


@pytest.mark.parametrize("T,pinned", [
    (8, "all"),        # page-locked host buffers (asynchronous copies)
    (8, "none"),       # pageable host buffers
    (1, "mixed"),      # some of each
    (20, "all"),
])
def test_host_buffer_entry_matches_device_entry(T, pinned):
    L = layer(inputs.dsv3(T), "mtp" if T == 8 else "uniform", seed=9)
    dev = run_fused(L, 0)
    ws = workspace(L, host=True)

    def host(t, pin):
        t = t.cpu().clone()
        return t.pin_memory() if pin else t

    xh = host(L.x, pinned != "none")
    ih = host(L.topk_ids, pinned != "none")
    wh = host(L.topk_w, pinned == "all")
    oh = host(torch.empty_like(L.x), pinned != "none")
    oh.fill_(7)
    B.moe_fused_decode_host(xh, ih, wh, B.make_weights(L.routed), B.make_weights(L.shared), oh,
                            shape_of(L), ws)
    assert torch.equal(oh.view(torch.int16), dev.cpu().view(torch.int16))
    assert B.moe_read_error(ws) == 0


def test_cuda_graph_replay_equals_eager():
    L = layer(inputs.dsv3(8), "mtp", seed=10)
    eager = run_fused(L, 0)
    ws = workspace(L)
    out = torch.empty_like(eager)
    rw, sw, sh = B.make_weights(L.routed), B.make_weights(L.shared), shape_of(L)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, rw, sw, out, sh, ws)  # warm up (attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, rw, sw, out, sh, ws)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert B.moe_read_error(ws) == 0


def test_zero_rows_launches_nothing():
    L = inputs.make_tiny(0, "cuda")
    sh = B.make_shape(0, 256, 128, 128, 8, 2, 0)
    ws = workspace(L)
    B.moe_fused_decode(None, None, None, B.make_weights(L.routed), B.make_weights(L.shared), None, sh, ws)
    assert B.moe_read_error(ws) == 0
