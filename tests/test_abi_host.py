"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/moe.h declares, sizes workspaces, and rejects invalid
arguments with the documented status before touching the device."""
import ctypes
import os
import re

import pytest

from moe_layer_decode_persistent_b300 import binding as B
from moe_layer_decode_persistent_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src))


def test_header_declarations_match_binding_list():
    assert _declared() == set(B.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    for name in _declared():
        assert hasattr(lib, name), name


def _shape(**kw):
    d = dict(T=4, H=256, I=128, I_shared=128, E=8, K=2, flags=0)
    d.update(kw)
    return B.make_shape(**d)


def test_workspace_bytes_grow_with_T_and_reject_bad_shapes():
    a = B.moe_workspace_bytes(_shape(T=1))
    b = B.moe_workspace_bytes(_shape(T=8))
    assert 0 < a < b
    assert B.moe_workspace_bytes_host(_shape(T=8)) > b
    for bad in (dict(T=-1), dict(T=257), dict(K=0), dict(K=9, E=8), dict(E=0), dict(H=100),
                dict(I=192 + 1), dict(I_shared=0), dict(flags=1 << 20),
                dict(flags=B.MOE_FLAG_FORCE_FMA | B.MOE_FLAG_FORCE_MMA)):
        assert B.moe_workspace_bytes(_shape(**bad)) == 0, bad


def test_every_declared_flag_is_accepted_and_leaves_the_workspace_size():
    base = B.moe_workspace_bytes(_shape(T=8))
    for f in (B.MOE_FLAG_NO_DEDUP, B.MOE_FLAG_FORCE_FMA, B.MOE_FLAG_FORCE_MMA, B.MOE_FLAG_DEBUG_DROP_ARRIVE,
              B.MOE_FLAG_CHAIN, B.MOE_FLAG_CHAIN | B.MOE_FLAG_FORCE_MMA, B.MOE_FLAG_FP8_MID):
        assert B.moe_workspace_bytes(_shape(T=8, flags=f)) == base, f


def test_workspace_bytes_never_shrink_as_T_grows():
    # the header states that a workspace sized for T serves every smaller T;
    # the tensor path's K-chunk partials change shape at T=3 and T=17
    for dims in (dict(H=7168, I=2048, I_shared=2048, E=256, K=8), dict(H=512, I=256, I_shared=512, E=16, K=4)):
        prev = 0
        for T in range(0, 257):
            n = B.moe_workspace_bytes(_shape(T=T, **dims))
            assert n >= prev, (dims, T, n, prev)
            prev = n


def test_group_table_ints():
    assert B.moe_group_table_ints(4, 2) == 2 + 5 * 4 * 3
    assert B.moe_group_table_ints(0, 8) == 2


def test_status_strings():
    for s in range(5):
        assert B.status_string(s).startswith("MOE_")


class _FakeTensor:
    """Stands in for a device tensor on a GPU-less host: a fake, aligned address."""

    def __init__(self, addr, nbytes):
        self.addr, self.n = addr, nbytes

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.n

    def element_size(self):
        return 1


def _weights(fmt=B.MOE_W_BF16, addr=1 << 20):
    return B.moe_weights(fmt, addr, addr if fmt else None, addr if fmt == 1 else None,
                         addr, addr if fmt else None, addr if fmt == 1 else None)


def _call(shape, x=1 << 24, out=1 << 26, ids=1 << 28, w=1 << 29, routed=None, shared=None,
          ws_addr=1 << 30, ws_bytes=None):
    routed = routed or _weights()
    shared = shared or _weights()
    n = B.moe_workspace_bytes(shape) if ws_bytes is None else ws_bytes
    ws = _FakeTensor(ws_addr, n)
    return B.moe_fused_decode(x, ids, w, routed, shared, out, shape, ws, stream=0, check=False)


def test_invalid_arguments_are_rejected_before_any_launch():
    s = _shape()
    assert _call(s, ws_addr=0) == B.MOE_ERR_INVALID_ARG
    assert _call(s, ws_addr=(1 << 30) + 8) == B.MOE_ERR_INVALID_ARG
    assert _call(s, ws_bytes=1024) == B.MOE_ERR_WORKSPACE
    assert _call(s, x=0) == B.MOE_ERR_INVALID_ARG
    assert _call(s, x=(1 << 24) + 2) == B.MOE_ERR_INVALID_ARG
    assert _call(s, out=(1 << 24) + 64) == B.MOE_ERR_INVALID_ARG  # out overlaps x
    assert _call(s, routed=B.moe_weights(7, 1 << 20, None, None, 1 << 20, None, None)) == \
        B.MOE_ERR_INVALID_ARG
    assert _call(s, shared=B.moe_weights(B.MOE_W_NVFP4, 1 << 20, 1 << 20, None, 1 << 20, 1 << 20,
                                         None)) == B.MOE_ERR_INVALID_ARG
    assert _call(s, routed=_weights(addr=(1 << 20) + 4)) == B.MOE_ERR_INVALID_ARG
    assert _call(_shape(H=192)) == B.MOE_ERR_UNSUPPORTED
    assert _call(_shape(K=0)) == B.MOE_ERR_INVALID_ARG
    detail = B.lib().moe_last_error_detail().decode()
    assert "K=0" in detail


def test_zero_rows_is_a_no_op():
    s = _shape(T=0)
    assert _call(s, x=0, out=0, ids=0, w=0) == B.MOE_OK


def test_host_call_rejects_small_workspace():
    s = _shape()
    ws = _FakeTensor(1 << 30, B.moe_workspace_bytes(s))  # enough for device call, not host
    st = B.lib().moe_fused_decode_host(1, 1, 1, ctypes.byref(_weights()), ctypes.byref(_weights()),
                                       1, ctypes.byref(s), ws.addr, ws.n, 0)
    assert st == B.MOE_ERR_WORKSPACE


def test_next_layer_hint_is_checked_before_any_launch():
    """moe_fused_decode_next rejects a missing, incomplete, misaligned or
    other-format next shared expert on the host, before the device is touched."""
    s = _shape()
    ws = _FakeTensor(1 << 30, B.moe_workspace_bytes(s))

    def call(nxt):
        ref = ctypes.byref(nxt) if nxt is not None else None
        return B.lib().moe_fused_decode_next(1 << 24, 1 << 28, 1 << 29, ctypes.byref(_weights()),
                                             ctypes.byref(_weights()), ref, 1 << 26, ctypes.byref(s),
                                             ws.addr, ws.n, 0)

    assert call(None) == B.MOE_ERR_INVALID_ARG
    assert call(_weights(B.MOE_W_FP8_B128)) == B.MOE_ERR_INVALID_ARG      # another format than `shared`
    assert "format" in B.lib().moe_last_error_detail().decode()
    assert call(_weights(addr=(1 << 20) + 8)) == B.MOE_ERR_INVALID_ARG    # misaligned
    assert call(B.moe_weights(B.MOE_W_BF16, None, None, None, 1 << 20, None, None)) == B.MOE_ERR_INVALID_ARG
