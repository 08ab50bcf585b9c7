"""The routing front end on the GPU, through the C ABI: moe_route against the
oracle's router, and moe_fused_decode_routed (the router inside the fused
launch) against moe_fused_decode given the same picks, bit for bit, and the
oracle layer.

The picks are compared exactly wherever the oracle's keys are further apart
than the fp32 rounding of the GPU's logits can move them (a bound derived
below); inside that band any order the bound allows is valid, and the test
checks that instead."""
import numpy as np
import pytest
import torch

import oracle
from moe_layer_decode_persistent_b300 import binding as B
from moe_layer_decode_persistent_b300 import inputs

from gpu_util import assert_parity, ensure_built, layer, oracle_ref, run_fused, shape_of, workspace

pytestmark = pytest.mark.gpu

PATHS = {"fma": B.MOE_FLAG_FORCE_FMA, "mma": B.MOE_FLAG_FORCE_MMA, "auto": 0}


def router_weights(E, H, seed, bias=True):
    """bf16 router rows with logits of about unit spread for N(0,1) inputs,
    and a small bf16 correction bias."""
    g = torch.Generator().manual_seed(seed)
    wr = (torch.randn(E, H, generator=g) * (1.5 / np.sqrt(H))).to(torch.bfloat16)
    b = (torch.randn(E, generator=g) * 0.05).to(torch.bfloat16) if bias else None
    return wr, b


def key_error_bound(x, wr):
    """|key_gpu - key_exact| <= this, per (row, expert): the GPU sums each
    logit in fp32 along at most 64 roundings, each within 2^-24 of the running
    sum, which is at most sum_h |x_h w_h|; the sigmoid has slope <= 1/4; the
    sigmoid's own evaluation and the bias add add a few units of 2^-24."""
    ax = x.double().abs()
    aw = wr.double().abs()
    return 0.25 * 64 * 2.0 ** -24 * (ax @ aw.T).numpy() + 16 * 2.0 ** -24


def check_picks(ids, w, x, wr, bias, K, scale, renorm):
    """ids/w from the GPU; returns the number of rows whose picks had to be
    checked inside the error band (0 means every pick was compared exactly)."""
    T, E = ids.shape[0], wr.shape[0]
    ref_ids, ref_w, keys = oracle.route(x, wr, bias, T, x.shape[1], E, K, scale=scale, renorm=renorm)
    delta = key_error_bound(x, wr)
    bias64 = np.zeros(E) if bias is None else bias.double().numpy()
    near = 0
    for t in range(T):
        got = ids[t].tolist()
        assert len(set(got)) == K and all(0 <= e < E for e in got), (t, got)
        order = np.argsort(-keys[t], kind="stable")
        kth = keys[t, order[K - 1]]
        band = 2 * delta[t].max()
        # no pick is clearly outside the top K, and every clearly-inside expert is picked
        assert all(keys[t, e] >= kth - band for e in got), (t, got)
        assert all(e in got for e in order if keys[t, e] > kth + band), t
        if np.array_equal(ref_ids[t], ids[t]):
            pass
        else:
            near += 1
            # picks differ only where the keys are within the band of each other
            for p in range(K):
                a, b_ = got[p], int(ref_ids[t, p])
                assert abs(keys[t, a] - keys[t, b_]) <= band, (t, p, a, b_)
        # weights: the oracle's fp64 weights of the GPU's picks
        s = keys[t, got] - bias64[got]
        want = scale * (s / s.sum() if renorm else s)
        assert np.allclose(w[t], want, rtol=2e-6, atol=1e-7), (t, w[t], want)
    return near


def run_route(x, wr, bias, E, K, scale=1.0, renorm=True):
    ensure_built()
    T, H = x.shape
    sh = B.make_shape(T, H, 256, 256, E, K, 0)
    ws = torch.empty(B.moe_workspace_bytes(sh), dtype=torch.uint8, device="cuda")
    B.moe_workspace_init(ws)
    wr_d, b_d = wr.cuda(), (None if bias is None else bias.cuda())
    ids = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    B.moe_route(x.cuda(), B.make_router(wr_d, b_d, scale, renorm), ids, w, sh, ws)
    assert B.moe_read_error(ws) == 0
    return ids.cpu().numpy(), w.cpu().double().numpy()


@pytest.mark.parametrize("T,H,E,K,bias,renorm", [
    (5, 512, 16, 4, True, True),
    (3, 256, 64, 6, True, True),      # K not a power of two
    (7, 1024, 40, 5, False, False),   # no bias, no renormalisation
    (1, 7168, 256, 8, True, True),    # DeepSeek-V3 shapes
    (8, 7168, 256, 8, True, True),
    (64, 7168, 256, 8, True, True),
    (16, 7168, 384, 8, True, True),   # wide-expert layer
    (2, 512, 1024, 16, True, True),   # the largest E and K
])
def test_route_matches_oracle(T, H, E, K, bias, renorm):
    x = inputs.activations(T, H, T * 7 + E)
    wr, b = router_weights(E, H, E + K, bias)
    ids, w = run_route(x, wr, b, E, K, scale=2.5, renorm=renorm)
    near = check_picks(ids, w, x, wr, b, K, 2.5, renorm)
    assert near <= max(1, T // 16), f"{near} of {T} rows inside the rounding band"


def test_route_exact_ties_go_to_the_lower_expert():
    """x = 0: every logit is exactly 0 and every score exactly 1/2, so the keys
    are 1/2 + bias exactly, with deliberate ties."""
    T, H, E, K = 3, 256, 12, 6
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    wr, _ = router_weights(E, H, 1)
    bias = torch.tensor([0.5, -1, 0.25, 0.5, 0, 3, 0.25, -2, 0.5, 1, 0.25, 0.125]).to(torch.bfloat16)
    ids, w = run_route(x, wr, bias, E, K, scale=2.5)
    assert ids.tolist() == [[5, 9, 0, 3, 8, 2]] * T
    assert np.allclose(w, np.full((T, K), 2.5 / K), rtol=1e-6, atol=0)


def routed_layer(shape, seed, fr=inputs.FMT_NVFP4, fs=inputs.FMT_FP8_B128):
    L = layer(shape, "uniform", seed=seed, fr=fr, fs=fs, used_only=False)
    wr, b = router_weights(shape.E, shape.H, seed + 100)
    return L, wr.cuda(), b.cuda()


def run_routed(L, wr, b, flags=0, ws=None, outputs=True):
    s = L.shape
    ws = workspace(L) if ws is None else ws
    out = torch.empty(s.T, s.H, dtype=torch.bfloat16, device="cuda")
    ids = torch.full((s.T, s.K), -7, dtype=torch.int32, device="cuda") if outputs else None
    w = torch.full((s.T, s.K), float("nan"), dtype=torch.float32, device="cuda") if outputs else None
    B.moe_fused_decode_routed(L.x, B.make_router(wr, b, 2.5, True), B.make_weights(L.routed),
                              B.make_weights(L.shared), out, shape_of(L, flags), ws, topk_ids=ids, topk_w=w)
    assert B.moe_read_error(ws) == 0
    return out, ids, w


SMALL = inputs.Shape(T=5, H=512, I=256, I_shared=512, E=16, K=4)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("case", ["small", "dsv3_t8"])
def test_fused_routed_equals_fused_with_its_picks(path, case):
    """The router inside the launch gives exactly the layer that moe_fused_decode
    computes from the picks and weights it reports; those picks match the
    oracle's router, and the layer matches the oracle layer."""
    shape = SMALL if case == "small" else inputs.dsv3(8)
    L, wr, b = routed_layer(shape, 3)
    out, ids, w = run_routed(L, wr, b, PATHS[path])
    check_picks(ids.cpu().numpy(), w.cpu().double().numpy(), L.x.cpu(), wr.cpu(), b.cpu(), shape.K, 2.5, True)
    L.topk_ids, L.topk_w = ids, w
    plain = run_fused(L, PATHS[path])
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))
    assert_parity(out, oracle_ref(L))


@pytest.mark.parametrize("path", list(PATHS))
def test_fused_routed_dedup_equals_one_row_and_outputs_are_optional(path):
    L, wr, b = routed_layer(inputs.Shape(T=13, H=512, I=256, I_shared=512, E=16, K=4), 5)
    a, _, _ = run_routed(L, wr, b, PATHS[path])
    c, _, _ = run_routed(L, wr, b, PATHS[path] | B.MOE_FLAG_NO_DEDUP, outputs=False)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_fused_routed_repeats_on_one_workspace_alongside_plain_launches():
    L, wr, b = routed_layer(SMALL, 9)
    ws = workspace(L)
    first, ids, w = run_routed(L, wr, b, 0, ws=ws)
    L.topk_ids, L.topk_w = ids, w
    for _ in range(2):
        again, _, _ = run_routed(L, wr, b, 0, ws=ws)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
        plain = run_fused(L, 0, ws=ws)
        assert torch.equal(plain.view(torch.int16), first.view(torch.int16))
