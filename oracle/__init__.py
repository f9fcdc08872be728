"""Test infrastructure -- Python entry points of the CPU oracle.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may import this package.  The product path (the CUDA library and
its binding) never does.

The arithmetic lives in ``oracle.c`` (plain loops, FP64 accumulation); this
module compiles it with gcc and marshals numpy arrays.  Functions take bf16
tensors as ``np.uint16`` bit patterns and return float64 results that are
not rounded to any narrower type.

Every function is pinned by ``tests/test_oracle.py`` against brute force,
ordinary GEMMs, hand-worked values and invariants of the definitions.

``swiglu`` follows the fused-activation mention in the DeepGEMM issue
thread (wgrad utilities "fused with SwiGLU"); the pages do not define it, so
the standard definition is used: the gate-up output holds the gate half in
columns [0, F) and the up half in [F, 2F), and h = SiLU(gate) * up with
SiLU(z) = z / (1 + exp(-z)), evaluated in FP64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (gcc, OpenMP, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        c_p = ctypes.c_void_p
        lib.oracle_mgemm_rows.argtypes = [c_p, c_p, c_p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          c_p, ctypes.c_int64, c_p]
        lib.oracle_mgemm_rows.restype = ctypes.c_int
        lib.oracle_mgemm_nested_rows.argtypes = [c_p, c_p, c_p, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, c_p, ctypes.c_int64, c_p]
        lib.oracle_mgemm_nested_rows.restype = ctypes.c_int
        lib.oracle_mgemm_mx_rows.argtypes = [c_p, c_p, c_p, c_p, c_p, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             c_p, ctypes.c_int64, c_p]
        lib.oracle_mgemm_mx_rows.restype = ctypes.c_int
        lib.oracle_mx_decode_tables.argtypes = [c_p, c_p]
        lib.oracle_mx_decode_tables.restype = None
        lib.oracle_mx_blocked.argtypes = [c_p, ctypes.c_int64, ctypes.c_int, c_p, ctypes.c_int,
                                          c_p, ctypes.c_int64]
        lib.oracle_mx_blocked.restype = ctypes.c_int64
        lib.oracle_kgemm_mx_rows.argtypes = [c_p, c_p, c_p, c_p, c_p, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_int, ctypes.c_int, c_p, c_p, ctypes.c_int64, c_p]
        lib.oracle_kgemm_mx_rows.restype = ctypes.c_int
        lib.oracle_mx_blocked_k.argtypes = [c_p, ctypes.c_int64, ctypes.c_int, c_p, ctypes.c_int,
                                            c_p, ctypes.c_int64]
        lib.oracle_mx_blocked_k.restype = ctypes.c_int64
        lib.oracle_kgemm_rows.argtypes = [c_p, c_p, c_p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_int,
                                          c_p, c_p, ctypes.c_int64, c_p]
        lib.oracle_kgemm_rows.restype = ctypes.c_int
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def mgemm(x, w, offsets, transpose_B: bool = False, rows=None) -> np.ndarray:
    """M-grouped GEMM.

    x: [M,K] bf16 bits; w: [E,N,K] (or [E,K,N] with transpose_B) bf16 bits;
    offsets: int32 [E+1].  Returns float64 [M,N] with rows >= offsets[E] set
    to NaN (they belong to no expert), or, when ``rows`` is given, float64
    [len(rows), N] for those rows only.
    """
    x, w = _u16(x), _u16(w)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    M, K = x.shape
    E = w.shape[0]
    N = w.shape[2] if transpose_B else w.shape[1]
    assert w.shape == ((E, K, N) if transpose_B else (E, N, K)), w.shape
    assert off.shape == (E + 1,)
    full = rows is None
    if full:
        rows = np.arange(int(off[E]), dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), N), dtype=np.float64)
    rc = _load().oracle_mgemm_rows(_ptr(x), _ptr(w), _ptr(off), E, M, N, K,
                                   int(bool(transpose_B)), _ptr(rows), len(rows), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_mgemm_rows rejected its arguments")
    if full:
        y = np.full((M, N), np.nan, dtype=np.float64)
        y[: int(off[E])] = out
        return y
    return out


def mgemm_nested(x, w, offsets, transpose_B: bool = False, rows=None) -> np.ndarray:
    """Nested grouped GEMM (CUTLASS discussion #1452): O outer groups over
    the columns, L inner groups over the rows.

    x: [M, O*K] bf16 bits; w: [O, L, N, K] (or [O, L, K, N] with
    transpose_B) bf16 bits; offsets: int32 [L+1].  Returns float64 [M, O*N]
    with y[r, o*N + n] = sum_k x[r, o*K + k] * B_{o,l}[k, n] for r in inner
    group l, rows >= offsets[L] set to NaN; or, when ``rows`` is given,
    float64 [len(rows), O*N] for those rows only.
    """
    x, w = _u16(x), _u16(w)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    O, L = w.shape[0], w.shape[1]
    K, N = (w.shape[2], w.shape[3]) if transpose_B else (w.shape[3], w.shape[2])
    M = x.shape[0]
    assert x.shape == (M, O * K), (x.shape, w.shape)
    assert off.shape == (L + 1,)
    full = rows is None
    if full:
        rows = np.arange(int(off[L]), dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), O * N), dtype=np.float64)
    rc = _load().oracle_mgemm_nested_rows(_ptr(x), _ptr(w), _ptr(off), O, L, M, N, K,
                                          int(bool(transpose_B)), _ptr(rows), len(rows), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_mgemm_nested_rows rejected its arguments")
    if full:
        y = np.full((M, O * N), np.nan, dtype=np.float64)
        y[: int(off[L])] = out
        return y
    return out


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8, a.dtype
    return a


def mx_decode_tables() -> tuple[np.ndarray, np.ndarray]:
    """(E4M3 values, E8M0 values) of all 256 codes each, float64."""
    a = np.empty(256, dtype=np.float64)
    b = np.empty(256, dtype=np.float64)
    _load().oracle_mx_decode_tables(_ptr(a), _ptr(b))
    return a, b


def mgemm_mx(xq, sx, wq, sw, offsets, transpose_B: bool = False, rows=None) -> np.ndarray:
    """MXFP8 M-grouped GEMM: E4M3 element codes with one E8M0 scale per 32
    elements along K.

    xq: uint8 [M,K]; sx: uint8 [M,K/32]; wq: uint8 [E,N,K] (or [E,K,N] with
    transpose_B); sw: uint8 [E,N,K/32] (scale of B element (k, n) of expert
    e is sw[e, n, k//32] in both layouts); offsets: int32 [E+1].  Returns
    float64 [M,N] with rows >= offsets[E] set to NaN, or [len(rows), N].
    """
    xq, sx, wq, sw = _u8(xq), _u8(sx), _u8(wq), _u8(sw)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    M, K = xq.shape
    E = wq.shape[0]
    N = wq.shape[2] if transpose_B else wq.shape[1]
    assert wq.shape == ((E, K, N) if transpose_B else (E, N, K)), wq.shape
    assert K % 32 == 0 and sx.shape == (M, K // 32) and sw.shape == (E, N, K // 32)
    assert off.shape == (E + 1,)
    full = rows is None
    if full:
        rows = np.arange(int(off[E]), dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), N), dtype=np.float64)
    rc = _load().oracle_mgemm_mx_rows(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), _ptr(off), E, M, N, K,
                                      int(bool(transpose_B)), _ptr(rows), len(rows), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_mgemm_mx_rows rejected its arguments")
    if full:
        y = np.full((M, N), np.nan, dtype=np.float64)
        y[: int(off[E])] = out
        return y
    return out


def mx_blocked_bytes(R: int, KS: int, G: int) -> int:
    """Upper bound of the blocked layout's size for R rows in G groups."""
    return (R // 128 + G) * ((KS + 3) // 4) * 512


def mx_blocked(scales, offsets, fill: int = 0) -> np.ndarray:
    """Blocked ("128x4") layout of grouped E8M0 scales [R, KS]: see
    oracle_mx_blocked in oracle.c.  Returns uint8 [mx_blocked_bytes(R, KS, G)]
    with bytes past the last block set to ``fill``."""
    src = _u8(scales)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    R, KS = src.shape
    G = len(off) - 1
    dst = np.full(mx_blocked_bytes(R, KS, G), fill, dtype=np.uint8)
    nb = _load().oracle_mx_blocked(_ptr(src), R, KS, _ptr(off), G, _ptr(dst), dst.size)
    if nb < 0:
        raise ValueError("oracle_mx_blocked rejected its arguments")
    return dst


def kgemm_mx(gq, sg, xq, sx, offsets, sel=None) -> np.ndarray:
    """MXFP8 K-grouped weight gradient in FP64.  gq uint8 [M,N], xq uint8
    [M,K] (E4M3), sg uint8 [N,M/32], sx uint8 [K,M/32] (E8M0, one scale per
    column and 32-row block), offsets int32 [E+1], all multiples of 32.
    Returns float64 [E,N,K], or [len(experts), K] for sel = (experts, ns)."""
    gq, sg, xq, sx = _u8(gq), _u8(sg), _u8(xq), _u8(sx)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    M, N = gq.shape
    K = xq.shape[1]
    E = len(off) - 1
    assert xq.shape[0] == M and M % 32 == 0 and sg.shape == (N, M // 32) and sx.shape == (K, M // 32)
    full = sel is None
    if full:
        se = np.repeat(np.arange(E, dtype=np.int32), N)
        sn = np.tile(np.arange(N, dtype=np.int32), E)
    else:
        se = np.ascontiguousarray(sel[0], dtype=np.int32)
        sn = np.ascontiguousarray(sel[1], dtype=np.int32)
    out = np.empty((len(se), K), dtype=np.float64)
    rc = _load().oracle_kgemm_mx_rows(_ptr(gq), _ptr(sg), _ptr(xq), _ptr(sx), _ptr(off), E, M, N, K,
                                      _ptr(se), _ptr(sn), len(se), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_kgemm_mx_rows rejected its arguments")
    return out.reshape(E, N, K) if full else out


def mx_blocked_k_bytes(R: int, KS: int, G: int) -> int:
    """Upper bound of the K-grouped blocked layout's size."""
    return ((R + 127) // 128) * (KS // 4 + G) * 512


def mx_blocked_k(scales, offsets, fill: int = 0) -> np.ndarray:
    """Blocked layout of scales [R, KS] grouped along the contraction by
    offsets (multiples of 32): see oracle_mx_blocked_k in oracle.c."""
    src = _u8(scales)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    R, KS = src.shape
    G = len(off) - 1
    dst = np.full(mx_blocked_k_bytes(R, KS, G), fill, dtype=np.uint8)
    nq = _load().oracle_mx_blocked_k(_ptr(src), R, KS, _ptr(off), G, _ptr(dst), dst.size)
    if nq < 0:
        raise ValueError("oracle_mx_blocked_k rejected its arguments")
    return dst


def kgemm(grad, X, offsets, sel=None) -> np.ndarray:
    """K-grouped FP32 weight gradient, computed in FP64.

    grad: [M,N] bf16 bits; X: [M,K] bf16 bits; offsets: int32 [E+1].
    Returns float64 [E,N,K], or, when ``sel`` = (experts, ns) is given,
    float64 [len(experts), K] with row i = dW[experts[i], ns[i], :].
    """
    grad, X = _u16(grad), _u16(X)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    M, N = grad.shape
    M2, K = X.shape
    assert M == M2
    E = len(off) - 1
    full = sel is None
    if full:
        se = np.repeat(np.arange(E, dtype=np.int32), N)
        sn = np.tile(np.arange(N, dtype=np.int32), E)
    else:
        se = np.ascontiguousarray(sel[0], dtype=np.int32)
        sn = np.ascontiguousarray(sel[1], dtype=np.int32)
    out = np.empty((len(se), K), dtype=np.float64)
    rc = _load().oracle_kgemm_rows(_ptr(grad), _ptr(X), _ptr(off), E, M, N, K,
                                   _ptr(se), _ptr(sn), len(se), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_kgemm_rows rejected its arguments")
    return out.reshape(E, N, K) if full else out


def swiglu(y13) -> np.ndarray:
    """h[r, f] = SiLU(y13[r, f]) * y13[r, F + f] in FP64, for y13 [M, 2F]
    (float64, e.g. the exact output of ``mgemm``); rows of NaN stay NaN."""
    y = np.asarray(y13, dtype=np.float64)
    F = y.shape[1] // 2
    assert y.shape[1] == 2 * F
    gate, up = y[:, :F], y[:, F:]
    return gate / (1.0 + np.exp(-gate)) * up


def swiglu_bwd(dh, y13) -> np.ndarray:
    """Gradient of sum(dh * swiglu(y13)) with respect to y13, in FP64: the
    backward of the activation that is fused after the down projection's
    input gradient (same DeepGEMM issue discussion, "fused with SwiGLU").
    With s = sigmoid(gate): d gate = dh * up * s * (1 + gate * (1 - s)),
    d up = dh * gate * s.  dh [M, F], y13 [M, 2F] -> dy13 [M, 2F]."""
    d = np.asarray(dh, dtype=np.float64)
    y = np.asarray(y13, dtype=np.float64)
    F = y.shape[1] // 2
    assert y.shape[1] == 2 * F and d.shape == (y.shape[0], F)
    gate, up = y[:, :F], y[:, F:]
    s = 1.0 / (1.0 + np.exp(-gate))
    return np.concatenate([d * up * s * (1.0 + gate * (1.0 - s)), d * gate * s], axis=1)
