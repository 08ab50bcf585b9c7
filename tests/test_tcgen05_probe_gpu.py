"""Single-CTA probes of the Blackwell building blocks the fused kernel uses:
TMEM store/load, tcgen05.mma (kind::f16, M=128) with A in TMEM or shared
memory and B in shared memory (no-swizzle K-major core matrices), per-column
independence of the MMA result, and TMA swizzled 3-D tiles."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "tc_probe.cu")
LIB = os.path.join(HERE, "csrc", "libtcprobe.so")
_lib = None


def lib():
    global _lib
    if _lib is None:
        hdrs = [os.path.join(HERE, "..", "moe_layer_decode_persistent_b300", "csrc", f)
                for f in ("sm100.cuh", "moe_common.cuh")]
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(p) for p in [SRC] + hdrs):
            subprocess.check_call(["nvcc", "-shared", "-Xcompiler", "-fPIC", "-std=c++17", "-O2",
                                   "-gencode", "arch=compute_103a,code=sm_103a", SRC, "-o", LIB])
        _lib = ctypes.CDLL(LIB)
    return _lib


def _p(a):
    return a.ctypes.data


def test_tmem_store_load_roundtrip():
    out = np.zeros((128, 32), np.uint32)
    assert lib().probe_tmem(ctypes.c_void_p(_p(out))) == 0
    want = np.arange(128)[:, None] * 1000 + np.arange(32)[None, :]
    assert np.array_equal(out, want)


def _mma(A, B, a_in_tmem):
    K = A.shape[1]
    N = B.shape[0]
    D = np.zeros((128, N), np.float32)
    err = np.zeros(1, np.uint32)
    rc = lib().probe_mma(ctypes.c_void_p(_p(A.view(np.uint16))), ctypes.c_void_p(_p(B.view(np.uint16))),
                         K, N, int(a_in_tmem), ctypes.c_void_p(_p(D)), ctypes.c_void_p(_p(err)))
    assert rc == 0 and err[0] == 0, (rc, err)
    return D


@pytest.mark.parametrize("a_in_tmem", [1, 0])
@pytest.mark.parametrize("K,N", [(16, 16), (32, 16), (64, 32), (32, 64), (64, 48)])
def test_mma_small_integers_exact(a_in_tmem, K, N):
    rng = np.random.default_rng(K * 100 + N)
    A = rng.integers(-4, 5, size=(128, K)).astype(np.float16)
    B = rng.integers(-4, 5, size=(N, K)).astype(np.float16)
    D = _mma(A, B, a_in_tmem)
    want = A.astype(np.float64) @ B.astype(np.float64).T
    assert np.array_equal(D.astype(np.float64), want), np.argwhere(D != want)[:5]


def test_mma_column_result_independent_of_other_columns_and_width():
    rng = np.random.default_rng(7)
    K = 64
    A = (rng.standard_normal((128, K)) * 0.05).astype(np.float16)
    B32 = rng.standard_normal((32, K)).astype(np.float16)
    D32 = _mma(A, B32, 1)
    D16 = _mma(A, B32[:16].copy(), 1)
    assert np.array_equal(D32[:, :16].view(np.uint32), D16.view(np.uint32))
    perm = rng.permutation(32)
    Dp = _mma(A, B32[perm].copy(), 1)
    assert np.array_equal(Dp.view(np.uint32), D32[:, perm].view(np.uint32))
    B64 = np.concatenate([B32, rng.standard_normal((32, K)).astype(np.float16)])
    D64 = _mma(A, B64, 1)
    assert np.array_equal(D64[:, :32].view(np.uint32), D32.view(np.uint32))
    # A from TMEM and from shared memory give the same bits
    Ds = _mma(A, B32, 0)
    assert np.array_equal(Ds.view(np.uint32), D32.view(np.uint32))


def _tma(src, box_c, swz, c0, c1, c2):
    E, R, Cb = src.shape
    out = np.zeros(box_c * 128, np.uint8)
    err = np.zeros(1, np.uint32)
    rc = lib().probe_tma(ctypes.c_void_p(_p(src)), E, R, Cb, box_c, swz, c0, c1, c2,
                         ctypes.c_void_p(_p(out)), ctypes.c_void_p(_p(err)))
    assert rc == 0 and err[0] == 0, (rc, err)
    return out.reshape(128, box_c)


@pytest.mark.parametrize("box_c,swz", [(64, 64), (128, 128), (16, 0), (112, 0)])
def test_tma_swizzled_box(box_c, swz):
    rng = np.random.default_rng(box_c + swz)
    E, R, Cb = 3, 300, 448
    src = rng.integers(0, 256, size=(E, R, Cb), dtype=np.uint8)
    c0, c1, c2 = 64, 100, 1
    got = _tma(src, box_c, swz, c0, c1, c2)
    want = np.zeros((128, box_c), np.uint8)
    rows = src[c2, c1:c1 + 128, c0:c0 + box_c]
    want[:rows.shape[0]] = rows
    if swz:
        sw = np.zeros_like(want)
        nchunk = box_c // 16
        for r in range(128):
            x = (r & 7) if swz == 128 else ((r >> 1) & 3)
            for c in range(nchunk):
                sw[r, (c ^ x) * 16:(c ^ x) * 16 + 16] = want[r, c * 16:c * 16 + 16]
        want = sw
    assert np.array_equal(got, want)


def test_tma_rows_past_the_end_read_zero():
    src = np.full((2, 200, 64), 7, np.uint8)
    got = _tma(src, 64, 64, 0, 150, 1)  # rows 150..277 of a 200-row expert
    assert np.all(got.reshape(128, 64)[50:] == 0)
