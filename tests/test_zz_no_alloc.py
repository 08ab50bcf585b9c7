"""The no-allocation entry point (moe_fused_decode_noalloc), called through the
C ABI, gives the same output as moe_fused_decode with a caller workspace, on
two calls in a row. It is for callers that may not call cudaMalloc (inside
global-mode graph capture, in plugins whose framework owns device memory, on
paths that cannot take cudaMalloc's device synchronisation); its scratch is an
8 MiB array inside the library. This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
from moe_layer_decode_persistent_b300 import binding as B
from moe_layer_decode_persistent_b300 import inputs

from gpu_util import assert_parity, ensure_built, layer, oracle_ref, run_fused, shape_of

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    ensure_built()
    L = layer(inputs.dsv3(8), "mtp", seed=11)
    want = run_fused(L, 0)
    want_fma = run_fused(L, B.MOE_FLAG_FORCE_FMA)  # the contraction this entry point uses
    rw, sw, sh = B.make_weights(L.routed), B.make_weights(L.shared), shape_of(L)
    err = torch.full((1,), 0xdead, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full_like(want, float("nan"))
        B.moe_fused_decode_noalloc(L.x, L.topk_ids, L.topk_w, rw, sw, out, sh, err_out=err)
        torch.cuda.synchronize()
        ok, ratio = oracle.tolerance_ok(out.float().cpu().double().numpy(),
                                        want.float().cpu().double().numpy())
        assert ok, f"no-alloc output differs beyond tolerance (ratio {ratio:.3f})"
        assert torch.equal(out.view(torch.int16), want_fma.view(torch.int16))
        assert int(err.item()) == 0
    assert_parity(out, oracle_ref(L))


def test_noalloc_size_limit_is_exact_at_dsv3_shapes():
    """The built-in 8 MiB scratch holds DeepSeek-V3 shapes up to T=25: T=25
    runs (and matches the workspace entry's CUDA-core result bit for bit),
    T=26 is refused with MOE_ERR_WORKSPACE before anything is launched."""
    ensure_built()
    L = layer(inputs.dsv3(25), "uniform", seed=13)
    want = run_fused(L, B.MOE_FLAG_FORCE_FMA)
    rw, sw = B.make_weights(L.routed), B.make_weights(L.shared)
    out = torch.full_like(want, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_fused_decode_noalloc(L.x, L.topk_ids, L.topk_w, rw, sw, out, shape_of(L), err_out=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    big = B.make_shape(26, 7168, 2048, 2048, 256, 8, 0)
    st = B.moe_fused_decode_noalloc(L.x, L.topk_ids, L.topk_w, rw, sw, out, big, check=False)
    assert st == B.MOE_ERR_WORKSPACE


def test_noalloc_reports_device_error_bits_and_rejects_large_shapes():
    ensure_built()
    s = inputs.Shape(T=4, H=256, I=128, I_shared=128, E=8, K=2)
    L = layer(s, "uniform", seed=12, used_only=False)
    L.topk_ids[0, 1] = 77
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(4, 256, dtype=torch.bfloat16, device="cuda")
    rw, sw = B.make_weights(L.routed), B.make_weights(L.shared)
    B.moe_fused_decode_noalloc(L.x, L.topk_ids, L.topk_w, rw, sw, out, shape_of(L), err_out=err)
    assert int(err.item()) == B.MOE_DEV_BAD_EXPERT
    # the next call starts clean
    L.topk_ids[0, 1] = 3 if int(L.topk_ids[0, 0]) != 3 else 4
    B.moe_fused_decode_noalloc(L.x, L.topk_ids, L.topk_w, rw, sw, out, shape_of(L), err_out=err)
    assert int(err.item()) == 0
    big = B.make_shape(64, 7168, 2048, 2048, 256, 8, 0)
    st = B.moe_fused_decode_noalloc(L.x, L.topk_ids, L.topk_w, rw, sw, out, big, check=False)
    assert st == B.MOE_ERR_WORKSPACE
    assert "8388608" in B.lib().moe_last_error_detail().decode()
