"""Chained launches (MOE_FLAG_CHAIN): layers back to back on one stream, each
launch allowed to start while the previous one still runs (programmatic
dependent launch), every layer on the same workspace.

Each layer's input is the previous layer's output, so a chained launch that
read its input, or the workspace, before the previous grid completed would
see stale data. The chain must give the same bits as the same launches
without the flag, eagerly and replayed from a CUDA graph, on either
contraction and across a switch between them, and the last layer must match
the oracle on the input it was actually given."""
import pytest
import torch

from moe_layer_decode_persistent_b300 import binding as B
from moe_layer_decode_persistent_b300 import inputs

from gpu_util import assert_parity, ensure_built, oracle_ref, shape_of, workspace

pytestmark = pytest.mark.gpu

SMALL = inputs.Shape(T=5, H=512, I=256, I_shared=512, E=16, K=4)
FMA, MMA = B.MOE_FLAG_FORCE_FMA, B.MOE_FLAG_FORCE_MMA


def make_layers(shape, n, seed=0, used_only=True):
    return [inputs.make_layer(shape, "uniform", seed + 11 * l, "cuda", inputs.FMT_NVFP4, inputs.FMT_FP8_B128,
                              layer=l, used_only=used_only) for l in range(n)]


def run_chain(layers, flags, ws, x0=None):
    """Layer l's input is layer l-1's output; flags[l] for launch l. Returns
    every layer's output (the launches are only queued; the caller syncs)."""
    x = layers[0].x if x0 is None else x0
    outs = []
    for L, f in zip(layers, flags):
        out = torch.empty(L.shape.T, L.shape.H, dtype=torch.bfloat16, device="cuda")
        B.moe_fused_decode(x, L.topk_ids, L.topk_w, B.make_weights(L.routed), B.make_weights(L.shared), out,
                           shape_of(L, f), ws)
        outs.append(out)
        x = out
    return outs


def same_bits(a, b):
    return all(torch.equal(u.view(torch.int16), v.view(torch.int16)) for u, v in zip(a, b))


@pytest.mark.parametrize("case,paths", [
    ("small", [FMA] * 4),
    ("small", [MMA] * 4),
    ("small", [FMA, MMA, MMA, FMA]),   # the chained kernel differs from the one before it
    ("dsv3_t1", [0] * 4),
    ("dsv3_t8", [0] * 4),
])
def test_chain_equals_unchained_launches(case, paths):
    ensure_built()
    shape = SMALL if case == "small" else inputs.dsv3(int(case[-1]))
    layers = make_layers(shape, len(paths))
    ws = workspace(layers[0])
    plain = run_chain(layers, paths, ws)
    chained = run_chain(layers, [f | B.MOE_FLAG_CHAIN for f in paths], ws)
    torch.cuda.synchronize()
    assert B.moe_read_error(ws) == 0
    assert same_bits(plain, chained)
    # the last layer against the oracle, on the input the chain gave it
    last = layers[-1]
    last.x = chained[-2]
    assert_parity(chained[-1], oracle_ref(last))


def test_chain_replays_from_a_cuda_graph():
    ensure_built()
    layers = make_layers(inputs.dsv3(1), 4)
    ws = workspace(layers[0])
    x0 = layers[0].x.clone()
    eager = run_chain(layers, [0] * 4, ws, x0)
    assert same_bits(eager, run_chain(layers, [B.MOE_FLAG_CHAIN] * 4, ws, x0))  # also warms the chained launch
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            graphed = run_chain(layers, [B.MOE_FLAG_CHAIN] * 4, ws, x0)
    torch.cuda.synchronize()
    for _ in range(3):
        for o in graphed:
            o.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert B.moe_read_error(ws) == 0
        assert same_bits(eager, graphed)


def test_chain_through_the_routed_entry():
    """The router reads the layer input too: a chained routed launch whose
    input is the previous layer's output picks the same experts and gives the
    same bits as unchained."""
    ensure_built()
    shape = inputs.dsv3(1)
    layers = make_layers(shape, 3, seed=5, used_only=False)
    g = torch.Generator().manual_seed(3)
    routers = []
    for _ in layers:
        wr = (torch.randn(shape.E, shape.H, generator=g) * (1.5 / shape.H ** 0.5)).to(torch.bfloat16).cuda()
        b = (torch.randn(shape.E, generator=g) * 0.05).to(torch.bfloat16).cuda()
        routers.append((wr, b))
    ws = workspace(layers[0])

    def chain(flags):
        x, outs, picks = layers[0].x, [], []
        for L, (wr, b) in zip(layers, routers):
            out = torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device="cuda")
            ids = torch.empty(shape.T, shape.K, dtype=torch.int32, device="cuda")
            B.moe_fused_decode_routed(x, B.make_router(wr, b, 2.5, True), B.make_weights(L.routed),
                                      B.make_weights(L.shared), out, shape_of(L, flags), ws, topk_ids=ids)
            outs.append(out)
            picks.append(ids)
            x = out
        return outs, picks

    a, pa = chain(0)
    c, pc = chain(B.MOE_FLAG_CHAIN)
    torch.cuda.synchronize()
    assert B.moe_read_error(ws) == 0
    assert all(torch.equal(u, v) for u, v in zip(pa, pc))
    assert same_bits(a, c)


def run_chain_next(layers, flags, ws, x0=None):
    """As run_chain, through moe_fused_decode_next: each launch also brings the
    next layer's first shared-expert stages into L2 (the last names the first)."""
    x = layers[0].x if x0 is None else x0
    outs = []
    for l, (L, f) in enumerate(zip(layers, flags)):
        out = torch.empty(L.shape.T, L.shape.H, dtype=torch.bfloat16, device="cuda")
        nxt = layers[(l + 1) % len(layers)]
        B.moe_fused_decode_next(x, L.topk_ids, L.topk_w, B.make_weights(L.routed), B.make_weights(L.shared),
                                B.make_weights(nxt.shared), out, shape_of(L, f), ws)
        outs.append(out)
        x = out
    return outs


@pytest.mark.parametrize("case,paths,fs", [
    ("small", [MMA] * 3, inputs.FMT_NVFP4),        # NVFP4 shared expert: codes and block scales
    ("small", [MMA] * 3, inputs.FMT_FP8_B128),
    ("small", [FMA, MMA, FMA], inputs.FMT_FP8_B128),  # the CUDA-core path ignores the hint
    ("dsv3_t1", [0] * 4, inputs.FMT_FP8_B128),
    ("dsv3_t8", [0] * 4, inputs.FMT_FP8_B128),
])
@pytest.mark.parametrize("chain", [False, True])
def test_next_layer_prefetch_changes_no_bit(case, paths, fs, chain):
    ensure_built()
    shape = SMALL if case == "small" else inputs.dsv3(int(case[-1]))
    layers = [inputs.make_layer(shape, "uniform", 3 + 7 * l, "cuda", inputs.FMT_NVFP4, fs, layer=l, used_only=True)
              for l in range(len(paths))]
    ws = workspace(layers[0])
    plain = run_chain(layers, paths, ws)
    hinted = run_chain_next(layers, [f | (B.MOE_FLAG_CHAIN if chain else 0) for f in paths], ws)
    torch.cuda.synchronize()
    assert B.moe_read_error(ws) == 0
    assert same_bits(plain, hinted)
