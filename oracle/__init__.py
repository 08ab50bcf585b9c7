"""Test infrastructure: the fp64 CPU oracle of the fused decode MoE layer.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The product path (the CUDA
library and its binding) never imports it, and it imports nothing from the
product package. See ``moe_oracle.c`` for what is computed and which page
passages each function follows.

Functions here take numpy arrays (or objects exposing ``numpy()``), marshal
them to the C library with ctypes, and return numpy results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

FMT_BF16, FMT_NVFP4, FMT_FP8_B128 = 0, 1, 2
ERR_BAD_EXPERT, ERR_DUP_EXPERT = 1, 2
FLAG_NO_DEDUP = 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
             "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Weights(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int),
                ("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w13_gscale", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
                ("w2_gscale", ctypes.c_void_p)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        d, i, p = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
        _lib.oracle_e2m1.restype = d
        _lib.oracle_e2m1.argtypes = [i]
        _lib.oracle_e4m3.restype = d
        _lib.oracle_e4m3.argtypes = [i]
        _lib.oracle_bf16.restype = d
        _lib.oracle_bf16.argtypes = [ctypes.c_uint16]
        _lib.oracle_w13_row.argtypes = [p, i, i, i, i, p]
        _lib.oracle_w2_row.argtypes = [p, i, i, i, i, p]
        _lib.oracle_expert_ffn.argtypes = [p, i, i, i, p, p, p]
        _lib.oracle_group_table_size.restype = i
        _lib.oracle_group_table_size.argtypes = [i, i]
        _lib.oracle_group_table.restype = i
        _lib.oracle_group_table.argtypes = [p, i, i, i, ctypes.c_uint, p, p]
        _lib.oracle_moe_layer_rows.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, i, p, i]
        _lib.oracle_unfused_layer.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p]
        _lib.oracle_moe_layer_uses.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, i, p, i]
        _lib.oracle_route.argtypes = [p, p, p, i, i, i, i, d, i, p, p, p]
        _lib.oracle_e4m3_rne.restype = d
        _lib.oracle_e4m3_rne.argtypes = [d]
        _lib.oracle_fp8_mid_blocks.argtypes = [p, i, i]
        _lib.oracle_moe_layer_fp8mid.argtypes = [p, p, p, p, p, i, i, i, i, i, i, p, i, p, i, i]
    return _lib


def _np(a, dtype):
    """numpy copy/view of a numpy array or a torch tensor, as `dtype`.

    Same-size dtypes are reinterpreted bit for bit (bf16 -> uint16, fp8 ->
    uint8); different sizes are value-converted (int64 ids -> int32)."""
    want = np.dtype(dtype)
    if hasattr(a, "detach"):  # a torch tensor
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype.is_floating_point and want.kind == "f" and t.element_size() == want.itemsize:
            a = t.numpy()
        elif t.dtype.is_floating_point and t.element_size() != want.itemsize:
            a = t.double().numpy()
        else:
            ints = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}
            a = t.view(ints[t.element_size()]).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        same_size = a.dtype.itemsize == want.itemsize
        both_int = a.dtype.kind in "iu" and want.kind in "iu"
        a = a.view(want) if (same_size and both_int) else a.astype(want)
    return a


class WeightSet:
    """Host copies of one expert set in the library's layout (see include/moe.h).

    fields: fmt, w13, w13_scale, w13_gscale, w2, w2_scale, w2_gscale as numpy
    arrays (or None). Keeps them alive while the C side holds pointers.
    """

    def __init__(self, fmt, w13, w2, w13_scale=None, w2_scale=None,
                 w13_gscale=None, w2_gscale=None):
        self.fmt = int(fmt)
        conv = {FMT_BF16: np.uint16, FMT_NVFP4: np.uint8, FMT_FP8_B128: np.uint8}[self.fmt]
        self.w13 = _np(w13, conv)
        self.w2 = _np(w2, conv)
        if self.fmt == FMT_NVFP4:
            self.w13_scale = _np(w13_scale, np.uint8)
            self.w2_scale = _np(w2_scale, np.uint8)
            self.w13_gscale = _np(w13_gscale, np.float32)
            self.w2_gscale = _np(w2_gscale, np.float32)
        elif self.fmt == FMT_FP8_B128:
            self.w13_scale = _np(w13_scale, np.float32)
            self.w2_scale = _np(w2_scale, np.float32)
            self.w13_gscale = self.w2_gscale = None
        else:
            self.w13_scale = self.w2_scale = self.w13_gscale = self.w2_gscale = None

    def cstruct(self) -> _Weights:
        def ptr(a):
            return None if a is None else a.ctypes.data
        return _Weights(self.fmt, ptr(self.w13), ptr(self.w13_scale), ptr(self.w13_gscale),
                        ptr(self.w2), ptr(self.w2_scale), ptr(self.w2_gscale))


def e2m1(code: int) -> float:
    return lib().oracle_e2m1(int(code))


def e4m3(byte: int) -> float:
    return lib().oracle_e4m3(int(byte))


def bf16(bits: int) -> float:
    return lib().oracle_bf16(int(bits) & 0xFFFF)


def w13_row(ws: WeightSet, H, I, e, r) -> np.ndarray:
    out = np.empty(H, np.float64)
    s = ws.cstruct()
    lib().oracle_w13_row(ctypes.byref(s), H, I, e, r, out.ctypes.data)
    return out


def w2_row(ws: WeightSet, H, I, e, h) -> np.ndarray:
    out = np.empty(I, np.float64)
    s = ws.cstruct()
    lib().oracle_w2_row(ctypes.byref(s), H, I, e, h, out.ctypes.data)
    return out


def dequant_w13(ws: WeightSet, H, I, e) -> np.ndarray:
    return np.stack([w13_row(ws, H, I, e, r) for r in range(2 * I)])


def dequant_w2(ws: WeightSet, H, I, e) -> np.ndarray:
    return np.stack([w2_row(ws, H, I, e, h) for h in range(H)])


def expert_ffn(ws: WeightSet, H, I, e, x64):
    x64 = np.ascontiguousarray(x64, np.float64)
    mid = np.empty(I, np.float64)
    y = np.empty(H, np.float64)
    s = ws.cstruct()
    lib().oracle_expert_ffn(ctypes.byref(s), H, I, e, x64.ctypes.data, mid.ctypes.data, y.ctypes.data)
    return mid, y


def group_table(ids, T, K, E, flags=0):
    """Returns (table int32 array, error bits)."""
    ids = _np(ids, np.int32).reshape(-1)
    n = lib().oracle_group_table_size(T, K)
    table = np.zeros(n, np.int32)
    err = ctypes.c_uint32(0)
    lib().oracle_group_table(ids.ctypes.data, T, K, E, flags, table.ctypes.data, ctypes.byref(err))
    return table, int(err.value)


def unpack_table(table, T, K):
    """Split a group table into named fields (views)."""
    C = T * (K + 1)
    G, U = int(table[0]), int(table[1])
    o = 2
    f = {}
    for name in ("group_expert", "group_ncols", "group_col0", "col_row", "row_col"):
        f[name] = table[o:o + C]
        o += C
    f["row_col"] = f["row_col"].reshape(T, K + 1)
    f["G"], f["U"] = G, U
    return f


def moe_layer(x_bf16, ids, topk_w, routed: WeightSet, shared: WeightSet, T, H, I, I_shared, E, K,
              rows=None, threads=1) -> np.ndarray:
    """fp64 reference rows [len(rows)][H] (all rows by default)."""
    x = _np(x_bf16, np.uint16).reshape(-1)
    ids = _np(ids, np.int32).reshape(-1)
    w = _np(topk_w, np.float32).reshape(-1)
    rows = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    out = np.empty((len(rows), H), np.float64)
    rs, ss = routed.cstruct(), shared.cstruct()
    lib().oracle_moe_layer_rows(x.ctypes.data, ids.ctypes.data, w.ctypes.data, ctypes.byref(rs),
                                ctypes.byref(ss), T, H, I, I_shared, E, K, rows.ctypes.data,
                                len(rows), out.ctypes.data, int(threads))
    return out


def moe_layer_uses(x_bf16, ids, topk_w, routed: WeightSet, shared: WeightSet, T, H, I, I_shared, E, K,
                   rows=None, threads=1) -> np.ndarray:
    """moe_layer with the expert evaluations of each row run on separate
    threads (bitwise equal to moe_layer)."""
    x = _np(x_bf16, np.uint16).reshape(-1)
    ids = _np(ids, np.int32).reshape(-1)
    w = _np(topk_w, np.float32).reshape(-1)
    rows = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    out = np.empty((len(rows), H), np.float64)
    rs, ss = routed.cstruct(), shared.cstruct()
    lib().oracle_moe_layer_uses(x.ctypes.data, ids.ctypes.data, w.ctypes.data, ctypes.byref(rs),
                                ctypes.byref(ss), T, H, I, I_shared, E, K, rows.ctypes.data,
                                len(rows), out.ctypes.data, int(threads))
    return out


FP8_MID_BLOCK = 32  # intermediate values per FP8 block (see oracle_fp8_mid_blocks)


def e4m3_rne(v: float) -> float:
    """The nearest E4M3FN value to v (ties to even), saturating at +-448."""
    return lib().oracle_e4m3_rne(float(v))


def fp8_mid_blocks(mid, block=FP8_MID_BLOCK) -> np.ndarray:
    """A copy of mid with each block of `block` values quantised to E4M3 at
    its power-of-two block scale (oracle_fp8_mid_blocks)."""
    m = np.array(mid, np.float64, copy=True)
    lib().oracle_fp8_mid_blocks(m.ctypes.data, len(m), int(block))
    return m


def moe_layer_fp8mid(x_bf16, ids, topk_w, routed: WeightSet, shared: WeightSet, T, H, I, I_shared, E, K,
                     rows=None, threads=1, block=FP8_MID_BLOCK) -> np.ndarray:
    """moe_layer with every expert use's SwiGLU intermediate in FP8 blocks."""
    x = _np(x_bf16, np.uint16).reshape(-1)
    ids = _np(ids, np.int32).reshape(-1)
    w = _np(topk_w, np.float32).reshape(-1)
    rows = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
    out = np.empty((len(rows), H), np.float64)
    rs, ss = routed.cstruct(), shared.cstruct()
    lib().oracle_moe_layer_fp8mid(x.ctypes.data, ids.ctypes.data, w.ctypes.data, ctypes.byref(rs),
                                  ctypes.byref(ss), T, H, I, I_shared, E, K, rows.ctypes.data,
                                  len(rows), out.ctypes.data, int(threads), int(block))
    return out


def route(x_bf16, wr_bf16, bias_bf16, T, H, E, K, scale=1.0, renorm=True):
    """The router: (ids int32 [T][K], weights fp64 [T][K], keys fp64 [T][E]).

    x_bf16 [T][H] and wr_bf16 [E][H] as bf16 bits (or bf16 tensors), bias_bf16
    [E] or None. See oracle_route in moe_oracle.c for the definition."""
    x = _np(x_bf16, np.uint16).reshape(-1)
    wr = _np(wr_bf16, np.uint16).reshape(-1)
    b = None if bias_bf16 is None else _np(bias_bf16, np.uint16).reshape(-1)
    ids = np.zeros((T, K), np.int32)
    w = np.zeros((T, K), np.float64)
    keys = np.zeros((T, E), np.float64)
    lib().oracle_route(x.ctypes.data, wr.ctypes.data, None if b is None else b.ctypes.data, T, H, E, K,
                       float(scale), int(bool(renorm)), ids.ctypes.data, w.ctypes.data, keys.ctypes.data)
    return ids, w, keys


def unfused_layer(x_bf16, ids, topk_w, routed: WeightSet, shared: WeightSet, T, H, I, I_shared, E, K):
    x = _np(x_bf16, np.uint16).reshape(-1)
    ids = _np(ids, np.int32).reshape(-1)
    w = _np(topk_w, np.float32).reshape(-1)
    out = np.empty((T, H), np.float64)
    rs, ss = routed.cstruct(), shared.cstruct()
    lib().oracle_unfused_layer(x.ctypes.data, ids.ctypes.data, w.ctypes.data, ctypes.byref(rs),
                               ctypes.byref(ss), T, H, I, I_shared, E, K, out.ctypes.data)
    return out


def tolerance_ok(gpu, ref):
    """|gpu - ref| <= 2^-7 |ref| + 1e-3 rms(ref), elementwise; returns (ok, worst ratio)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = 2.0 ** -7 * np.abs(ref) + 1e-3 * rms
    err = np.abs(gpu - ref)
    ratio = float(np.max(err / np.maximum(bound, 1e-300))) if ref.size else 0.0
    return bool(np.all(err <= bound)), ratio
