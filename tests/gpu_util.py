"""Helpers shared by the GPU tests: run the library through its C ABI and
compute the oracle on CPU copies of only the experts a batch uses."""
import os

import numpy as np
import torch

import oracle
from moe_layer_decode_persistent_b300 import binding as B
from moe_layer_decode_persistent_b300 import build, inputs

_BUILT = False


def ensure_built():
    global _BUILT
    if not _BUILT:
        build.build()
        _BUILT = True


def shape_of(L, flags=0):
    s = L.shape
    return B.make_shape(s.T, s.H, s.I, s.I_shared, s.E, s.K, flags)


def workspace(L, host=False, device="cuda"):
    ensure_built()
    sh = shape_of(L)
    n = B.moe_workspace_bytes_host(sh) if host else B.moe_workspace_bytes(sh)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    B.moe_workspace_init(ws)
    return ws


def run_fused(L, flags=0, ws=None, out=None, check_err=True):
    ensure_built()
    ws = workspace(L) if ws is None else ws
    out = torch.empty(L.shape.T, L.shape.H, dtype=torch.bfloat16, device="cuda") if out is None else out
    B.moe_fused_decode(L.x, L.topk_ids, L.topk_w, B.make_weights(L.routed), B.make_weights(L.shared),
                       out, shape_of(L, flags), ws)
    if check_err:
        err = B.moe_read_error(ws)
        assert err == 0, f"device error word 0x{err:x}"
    return out


def group_table_gpu(ids, T, K, E, flags=0):
    ensure_built()
    sh = B.make_shape(T, 128, 128, 128, E, K, flags)
    n = B.moe_group_table_ints(T, K)
    out = torch.full((n,), -77, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ids_d = torch.as_tensor(np.asarray(ids, np.int32).reshape(T, K)).cuda() if T else \
        torch.zeros((0, K), dtype=torch.int32, device="cuda")
    B.moe_group_table(ids_d, sh, out, ws)
    err = B.moe_read_error(ws)
    return out.cpu().numpy(), err


def oracle_weightset(es):
    return oracle.WeightSet(es.fmt, es.w13, es.w2, es.w13_scale, es.w2_scale, es.w13_gscale,
                            es.w2_gscale)


def oracle_ref(L, rows=None, threads=None, fp8_mid=False):
    """fp64 reference rows, copying to the host only the routed experts used."""
    s = L.shape
    ids = L.topk_ids.cpu().numpy().astype(np.int64)
    used = sorted(set(int(e) for e in ids.reshape(-1) if 0 <= e < s.E))
    remap = {e: i for i, e in enumerate(used)}
    ids2 = np.vectorize(lambda e: remap.get(int(e), -1))(ids).astype(np.int32) if ids.size else \
        ids.astype(np.int32)
    routed = oracle_weightset(L.routed.select(used)) if used else oracle_weightset(L.routed.select([0]))
    shared = oracle_weightset(L.shared.to("cpu"))
    threads = threads or min(32, os.cpu_count() or 1)
    f = oracle.moe_layer_fp8mid if fp8_mid else oracle.moe_layer
    return f(L.x.cpu(), ids2, L.topk_w.cpu(), routed, shared, s.T, s.H, s.I, s.I_shared, max(len(used), 1), s.K,
             rows=rows, threads=threads)


# (test id, worst |err|/bound, elements compared) of every parity check in
# this session; conftest prints them at the end of the run
RATIOS = []


def assert_parity(out, ref, rows=None):
    got = out.float().cpu().double().numpy()
    if rows is not None:
        got = got[np.asarray(rows)]
    ok, ratio = oracle.tolerance_ok(got, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RATIOS.append((test, ratio, int(np.asarray(ref).size)))
    assert ok, f"tolerance exceeded: worst |err|/bound = {ratio:.3f}"
    return ratio


def layer(shape, routing="uniform", seed=0, fr=inputs.FMT_NVFP4, fs=inputs.FMT_FP8_B128, used_only=True):
    return inputs.make_layer(shape, routing, seed, "cuda", fr, fs, used_only=used_only)
