"""ctypes binding of libmoe.so: the C ABI of include/moe.h under the same names.

Argument marshalling only -- every step of the layer runs in the library's
CUDA kernels. torch tensors are accepted for device buffers (their data
pointers are passed) and the current torch CUDA stream is used unless one is
given. If the library is missing, lib() raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = range(5)
MOE_DEV_BAD_EXPERT, MOE_DEV_DUP_EXPERT, MOE_DEV_WAIT_TIMEOUT, MOE_DEV_RANGE = 1, 2, 4, 8
MOE_FLAG_NO_DEDUP, MOE_FLAG_FORCE_FMA, MOE_FLAG_FORCE_MMA, MOE_FLAG_DEBUG_DROP_ARRIVE, MOE_FLAG_CHAIN = 1, 2, 4, 8, 16
MOE_FLAG_FP8_MID = 32
MOE_W_BF16, MOE_W_NVFP4, MOE_W_FP8_B128 = 0, 1, 2

# every symbol include/moe.h declares
EXPORTS = ("moe_workspace_bytes", "moe_workspace_bytes_host", "moe_workspace_init",
           "moe_group_table_ints", "moe_group_table", "moe_fused_decode", "moe_fused_decode_next",
           "moe_fused_decode_host",
           "moe_fused_decode_noalloc", "moe_route", "moe_fused_decode_routed", "moe_read_error",
           "moe_status_string", "moe_last_error_detail")


class moe_weights(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w13_gscale", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("w2_gscale", ctypes.c_void_p)]


class moe_router(ctypes.Structure):
    _fields_ = [("wr", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("scale", ctypes.c_float),
                ("renorm", ctypes.c_int)]


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("I_shared", ctypes.c_int), ("E", ctypes.c_int), ("K", ctypes.c_int),
                ("flags", ctypes.c_uint)]


class MoeError(RuntimeError):
    def __init__(self, status, detail):
        super().__init__(f"{status_string(status)}: {detail}")
        self.status = status


_lib = None


def lib():
    """Load libmoe.so (raises if it is missing: run build.py / __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with "
                               "`python -m moe_layer_decode_persistent_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, S, I, U = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
        sp, wp = ctypes.POINTER(moe_shape), ctypes.POINTER(moe_weights)
        L.moe_workspace_bytes.restype = S
        L.moe_workspace_bytes.argtypes = [sp]
        L.moe_workspace_bytes_host.restype = S
        L.moe_workspace_bytes_host.argtypes = [sp]
        L.moe_workspace_init.restype = I
        L.moe_workspace_init.argtypes = [P, S, P]
        L.moe_group_table_ints.restype = S
        L.moe_group_table_ints.argtypes = [I, I]
        L.moe_group_table.restype = I
        L.moe_group_table.argtypes = [P, sp, P, P, S, P]
        L.moe_fused_decode.restype = I
        L.moe_fused_decode.argtypes = [P, P, P, wp, wp, P, sp, P, S, P]
        L.moe_fused_decode_next.restype = I
        L.moe_fused_decode_next.argtypes = [P, P, P, wp, wp, wp, P, sp, P, S, P]
        L.moe_fused_decode_host.restype = I
        L.moe_fused_decode_host.argtypes = [P, P, P, wp, wp, P, sp, P, S, P]
        L.moe_fused_decode_noalloc.restype = I
        L.moe_fused_decode_noalloc.argtypes = [P, P, P, wp, wp, P, sp, P, P]
        rp = ctypes.POINTER(moe_router)
        L.moe_route.restype = I
        L.moe_route.argtypes = [P, rp, P, P, sp, P, S, P]
        L.moe_fused_decode_routed.restype = I
        L.moe_fused_decode_routed.argtypes = [P, rp, wp, wp, P, P, P, sp, P, S, P]
        L.moe_read_error.restype = I
        L.moe_read_error.argtypes = [P, ctypes.POINTER(U), P]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [I]
        L.moe_last_error_detail.restype = ctypes.c_char_p
        L.moe_last_error_detail.argtypes = []
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(status):
    if status != MOE_OK:
        raise MoeError(status, lib().moe_last_error_detail().decode())
    return status


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def make_shape(T, H, I, I_shared, E, K, flags=0) -> moe_shape:
    return moe_shape(int(T), int(H), int(I), int(I_shared), int(E), int(K), int(flags))


def make_weights(es) -> moe_weights:
    """moe_weights from an object with fmt, w13, w13_scale, w13_gscale, w2, w2_scale, w2_gscale."""
    return moe_weights(int(es.fmt), _ptr(es.w13), _ptr(es.w13_scale), _ptr(es.w13_gscale),
                       _ptr(es.w2), _ptr(es.w2_scale), _ptr(es.w2_gscale))


def moe_workspace_bytes(shape: moe_shape) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(shape))


def moe_workspace_bytes_host(shape: moe_shape) -> int:
    return lib().moe_workspace_bytes_host(ctypes.byref(shape))


def moe_group_table_ints(T: int, K: int) -> int:
    return lib().moe_group_table_ints(T, K)


def moe_workspace_init(ws, nbytes=None, stream=None, check=True):
    n = ws.numel() * ws.element_size() if nbytes is None else nbytes
    st = lib().moe_workspace_init(_ptr(ws), n, _stream(stream))
    return _check(st) if check else st


def moe_group_table(topk_ids, shape: moe_shape, table_out, ws, stream=None, check=True):
    st = lib().moe_group_table(_ptr(topk_ids), ctypes.byref(shape), _ptr(table_out), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream))
    return _check(st) if check else st


def moe_fused_decode(x, topk_ids, topk_w, routed: moe_weights, shared: moe_weights, out,
                     shape: moe_shape, ws, stream=None, ws_bytes=None, check=True):
    n = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    st = lib().moe_fused_decode(_ptr(x), _ptr(topk_ids), _ptr(topk_w), ctypes.byref(routed),
                                ctypes.byref(shared), _ptr(out), ctypes.byref(shape), _ptr(ws), n,
                                _stream(stream))
    return _check(st) if check else st


def moe_fused_decode_next(x, topk_ids, topk_w, routed: moe_weights, shared: moe_weights,
                          next_shared: moe_weights, out, shape: moe_shape, ws, stream=None, check=True):
    """moe_fused_decode that also brings the next layer's first shared-expert
    stages into L2 during its tail (same result bits)."""
    st = lib().moe_fused_decode_next(_ptr(x), _ptr(topk_ids), _ptr(topk_w), ctypes.byref(routed),
                                     ctypes.byref(shared), ctypes.byref(next_shared), _ptr(out),
                                     ctypes.byref(shape), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream))
    return _check(st) if check else st


def moe_fused_decode_host(x_host, ids_host, w_host, routed: moe_weights, shared: moe_weights,
                          out_host, shape: moe_shape, ws, stream=None, check=True):
    st = lib().moe_fused_decode_host(_ptr(x_host), _ptr(ids_host), _ptr(w_host),
                                     ctypes.byref(routed), ctypes.byref(shared), _ptr(out_host),
                                     ctypes.byref(shape), _ptr(ws), ws.numel() * ws.element_size(),
                                     _stream(stream))
    return _check(st) if check else st


def moe_fused_decode_noalloc(x, topk_ids, topk_w, routed: moe_weights, shared: moe_weights, out,
                             shape: moe_shape, err_out=None, stream=None, check=True):
    """The layer with the library's built-in scratch (no workspace, no allocation)."""
    st = lib().moe_fused_decode_noalloc(_ptr(x), _ptr(topk_ids), _ptr(topk_w), ctypes.byref(routed),
                                        ctypes.byref(shared), _ptr(out), ctypes.byref(shape),
                                        _ptr(err_out), _stream(stream))
    return _check(st) if check else st


def make_router(wr, bias=None, scale=1.0, renorm=True) -> moe_router:
    return moe_router(_ptr(wr), _ptr(bias), float(scale), int(bool(renorm)))


def moe_route(x, router: moe_router, topk_ids, topk_w, shape: moe_shape, ws, stream=None, check=True):
    st = lib().moe_route(_ptr(x), ctypes.byref(router), _ptr(topk_ids), _ptr(topk_w), ctypes.byref(shape),
                         _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    return _check(st) if check else st


def moe_fused_decode_routed(x, router: moe_router, routed: moe_weights, shared: moe_weights, out,
                            shape: moe_shape, ws, topk_ids=None, topk_w=None, stream=None, check=True):
    st = lib().moe_fused_decode_routed(_ptr(x), ctypes.byref(router), ctypes.byref(routed),
                                       ctypes.byref(shared), _ptr(out), _ptr(topk_ids), _ptr(topk_w),
                                       ctypes.byref(shape), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream))
    return _check(st) if check else st


def moe_read_error(ws, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().moe_read_error(_ptr(ws), ctypes.byref(v), _stream(stream)))
    return int(v.value)
