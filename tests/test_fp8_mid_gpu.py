"""The opt-in FP8 intermediate blocks (MOE_FLAG_FP8_MID) on the GPU against
the oracle's layer with the same blocks, on the tensor-core path: the result
must be within the layer's tolerance of that oracle, away from the exact
layer by about the E4M3 step, and the dedup form bitwise equal to the one-row
form. The CUDA-core path refuses the flag."""
import numpy as np
import pytest
import torch

from moe_layer_decode_persistent_b300 import binding as B
from moe_layer_decode_persistent_b300 import inputs

from gpu_util import assert_parity, layer, oracle_ref, run_fused, shape_of, workspace

pytestmark = pytest.mark.gpu

FP8 = B.MOE_FLAG_FP8_MID
SMALL = inputs.Shape(T=5, H=512, I=256, I_shared=512, E=16, K=4)


@pytest.mark.parametrize("path", ["mma", "auto"])
@pytest.mark.parametrize("case", ["small_nvfp4_fp8", "small_fp8_nvfp4", "small_T13", "dsv3_t1", "dsv3_t8"])
def test_fp8_mid_matches_the_oracle_with_the_same_blocks(path, case):
    flags = FP8 | (B.MOE_FLAG_FORCE_MMA if path == "mma" else 0)
    if case == "small_fp8_nvfp4":
        L = layer(SMALL, "zipf", seed=21, fr=inputs.FMT_FP8_B128, fs=inputs.FMT_NVFP4, used_only=False)
    elif case == "small_T13":
        L = layer(inputs.Shape(T=13, H=512, I=256, I_shared=512, E=16, K=4), "zipf", seed=22, used_only=False)
    elif case.startswith("dsv3"):
        T = int(case[-1])
        L = layer(inputs.dsv3(T), "uniform" if T == 1 else "mtp", seed=23)
    else:
        L = layer(SMALL, "zipf", seed=20, used_only=False)
    out = run_fused(L, flags)
    ref = oracle_ref(L, fp8_mid=True)
    assert_parity(out, ref)
    # the blocks matter: the exact layer differs by far more than the kernel's own rounding
    exact = oracle_ref(L)
    x = L.x.double().cpu().numpy()
    step = np.abs(ref - exact).max() / np.abs(exact - x).max()
    assert 1e-4 < step < 0.1
    one_row = run_fused(L, flags | B.MOE_FLAG_NO_DEDUP)
    assert torch.equal(out.view(torch.int16), one_row.view(torch.int16))


def test_fp8_mid_through_the_routed_entry_equals_the_plain_entry():
    L = layer(SMALL, "uniform", seed=24, used_only=False)
    g = torch.Generator().manual_seed(5)
    wr = (torch.randn(SMALL.E, SMALL.H, generator=g) * (1.5 / SMALL.H ** 0.5)).to(torch.bfloat16).cuda()
    b = (torch.randn(SMALL.E, generator=g) * 0.05).to(torch.bfloat16).cuda()
    ws = workspace(L)
    out = torch.empty(SMALL.T, SMALL.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(SMALL.T, SMALL.K, dtype=torch.int32, device="cuda")
    w = torch.empty(SMALL.T, SMALL.K, dtype=torch.float32, device="cuda")
    B.moe_fused_decode_routed(L.x, B.make_router(wr, b, 2.5, True), B.make_weights(L.routed),
                              B.make_weights(L.shared), out, shape_of(L, FP8), ws, topk_ids=ids, topk_w=w)
    assert B.moe_read_error(ws) == 0
    L.topk_ids, L.topk_w = ids, w
    plain = run_fused(L, FP8)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))


@pytest.mark.parametrize("how", ["force_fma", "bf16_weights"])
def test_fp8_mid_is_refused_off_the_tensor_core_path(how):
    if how == "force_fma":
        L = layer(SMALL, "zipf", seed=25, used_only=False)
        flags = FP8 | B.MOE_FLAG_FORCE_FMA
    else:
        L = inputs.make_tiny(0, "cuda")
        flags = FP8
    ws = workspace(L)
    out = torch.empty(L.shape.T, L.shape.H, dtype=torch.bfloat16, device="cuda")
    st = B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, B.make_weights(L.routed), B.make_weights(L.shared), out,
                            shape_of(L, flags), ws, check=False)
    assert st == B.MOE_ERR_UNSUPPORTED
    assert "FP8_MID" in B.lib().moe_last_error_detail().decode()
