"""MoE grouped GEMM for GB300 (sm_103a): thin Python binding of librg.so.

The binding only marshals arguments: it checks dtypes and shapes of torch
tensors, passes their device pointers and the current CUDA stream to the C
ABI declared in ``include/rg.h``, and turns error codes into exceptions.
Every step of the computation runs in the library's CUDA kernels; there is
no fallback path.  If the library is not built, ``load()`` raises.

Operations (RapidGEMM README, "Kernels"):

* ``mgemm(x, w, offsets, transpose_B=False)``: M-grouped GEMM for the forward
  pass (``y[rows of e] = x[rows of e] @ w[e].T``, w ``[E,N,K]``) or the input
  gradient (``transpose_B=True``: ``y = x @ w[e]``, w ``[E,K,N]``).
* ``kgemm(grad, X, offsets)``: K-grouped weight gradient
  ``dW[e] = grad[rows of e].T @ X[rows of e]`` in FP32.
* ``mgemm_mxfp8(xq, sx_blocked, wq, sw_blocked, offsets)``: MXFP8 M-grouped
  GEMM (E4M3 codes, E8M0 scale per 32 K elements, scales in the blocked
  layout made by ``mx_scales_blocked``).
* ``mgemm_nested(x, w, offsets)``: nested grouped GEMM (CUTLASS discussion
  #1452): O outer groups over the columns of x ``[M,O*K]`` and y ``[M,O*N]``,
  L inner row groups, w ``[O,L,N,K]``.

``offsets`` is a device int32 tensor ``[E+1]`` of cumulative row offsets
with a leading zero.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = ["load", "mgemm", "mgemm_nested", "mgemm_mxfp8", "mx_scales_blocked", "mx_blocked_bytes", "kgemm_mxfp8", "mx_scales_blocked_k", "mx_blocked_k_bytes", "mgemm_swiglu", "mgemm_swiglu_dgrad", "kgemm", "kgemm_workspace_bytes", "device_status", "shutdown", "set_wait_timeout_ns",
           "selftest_wait_timeout", "RGError", "lib_path", "version",
           "RG_DEV_BAD_OFFSETS", "RG_DEV_TIMEOUT", "EXPORTED_SYMBOLS"]

RG_OK = 0
RG_ERR_INVALID_ARG = -1
RG_ERR_UNSUPPORTED = -2
RG_ERR_CUDA = -3
RG_ERR_SCRATCH = -4
RG_KGEMM_NOALLOC_MAX_FLAGS = 65536
RG_DEV_BAD_OFFSETS = 0x1
RG_DEV_TIMEOUT = 0x2
RG_DEV_LAUNCH_CONFIG = 0x4
RG_DEV_BOUNDS = 0x8
RG_MAX_EXPERTS = 1024
RG_MAX_OUTER = 65536
RG_KGEMM_MAX_EXPERTS = 1024

EXPORTED_SYMBOLS = ("rg_mgemm", "rg_mgemm_nested", "rg_mgemm_mxfp8", "rg_mx_scales_blocked", "rg_mx_blocked_bytes", "rg_kgemm_mxfp8", "rg_mx_scales_blocked_k", "rg_mx_blocked_k_bytes", "rg_mgemm_swiglu", "rg_mgemm_swiglu_dgrad", "rg_kgemm", "rg_kgemm_acc", "rg_kgemm_workspace_bytes", "rg_kgemm_ws", "rg_kgemm_noalloc", "rg_get_device_status", "rg_shutdown", "rg_set_wait_timeout_ns",
                    "rg_selftest_wait_timeout", "rg_last_cuda_error", "rg_device_supported",
                    "rg_version")

_ERRNAMES = {RG_ERR_SCRATCH: "RG_ERR_SCRATCH", RG_ERR_INVALID_ARG: "RG_ERR_INVALID_ARG",
             RG_ERR_UNSUPPORTED: "RG_ERR_UNSUPPORTED",
             RG_ERR_CUDA: "RG_ERR_CUDA"}

_lib = None


class RGError(RuntimeError):
    def __init__(self, fn: str, code: int, cuda_error: int = 0):
        self.code = code
        self.cuda_error = cuda_error
        msg = f"{fn} failed: {_ERRNAMES.get(code, code)}"
        if code == RG_ERR_CUDA:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load librg.so (built in-tree by ``_build.build()``); raise if missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    lib.rg_mgemm.argtypes = [vp, vp, vp, i32, i64, i32, i32, i32, vp, vp]
    lib.rg_mgemm.restype = i32
    lib.rg_mgemm_nested.argtypes = [vp, vp, vp, i32, i32, i64, i32, i32, i32, vp, vp]
    lib.rg_mgemm_nested.restype = i32
    lib.rg_mgemm_mxfp8.argtypes = [vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, vp, vp]
    lib.rg_mgemm_mxfp8.restype = i32
    lib.rg_mx_scales_blocked.argtypes = [vp, vp, i32, i64, i32, vp, i64, vp]
    lib.rg_mx_scales_blocked.restype = i32
    lib.rg_mx_blocked_bytes.argtypes = [i64, i32, i32]
    lib.rg_mx_blocked_bytes.restype = i64
    lib.rg_kgemm_mxfp8.argtypes = [vp, vp, vp, vp, vp, i32, i64, i32, i32, vp, i32, vp]
    lib.rg_kgemm_mxfp8.restype = i32
    lib.rg_mx_scales_blocked_k.argtypes = [vp, vp, i32, i64, i32, vp, i64, vp]
    lib.rg_mx_scales_blocked_k.restype = i32
    lib.rg_mx_blocked_k_bytes.argtypes = [i64, i32, i32]
    lib.rg_mx_blocked_k_bytes.restype = i64
    lib.rg_mgemm_swiglu.argtypes = [vp, vp, vp, i32, i64, i32, i32, vp, vp, vp]
    lib.rg_mgemm_swiglu.restype = i32
    lib.rg_mgemm_swiglu_dgrad.argtypes = [vp, vp, vp, i32, i64, i32, i32, vp, vp, vp]
    lib.rg_mgemm_swiglu_dgrad.restype = i32
    lib.rg_kgemm.argtypes = [vp, vp, vp, i32, i64, i32, i32, vp, vp]
    lib.rg_kgemm.restype = i32
    lib.rg_kgemm_acc.argtypes = [vp, vp, vp, i32, i64, i32, i32, vp, vp]
    lib.rg_kgemm_acc.restype = i32
    lib.rg_kgemm_workspace_bytes.argtypes = [i32, i32, i32]
    lib.rg_kgemm_workspace_bytes.restype = i64
    lib.rg_kgemm_ws.argtypes = [vp, vp, vp, i32, i64, i32, i32, vp, i32, vp, i64, vp]
    lib.rg_kgemm_ws.restype = i32
    lib.rg_kgemm_noalloc.argtypes = [vp, vp, vp, i32, i64, i32, i32, vp, i32, vp]
    lib.rg_kgemm_noalloc.restype = i32
    lib.rg_get_device_status.argtypes = [vp]
    lib.rg_get_device_status.restype = i32
    lib.rg_shutdown.argtypes = []
    lib.rg_shutdown.restype = i32
    lib.rg_set_wait_timeout_ns.argtypes = [u64]
    lib.rg_set_wait_timeout_ns.restype = i32
    lib.rg_selftest_wait_timeout.argtypes = [u64, vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.rg_selftest_wait_timeout.restype = i32
    lib.rg_last_cuda_error.argtypes = []
    lib.rg_last_cuda_error.restype = i32
    lib.rg_device_supported.argtypes = []
    lib.rg_device_supported.restype = i32
    lib.rg_version.argtypes = []
    lib.rg_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def version() -> str:
    return load().rg_version().decode()


def _check(fn: str, rc: int) -> None:
    if rc != RG_OK:
        raise RGError(fn, rc, load().rg_last_cuda_error() if rc == RG_ERR_CUDA else 0)


def _stream_ptr(device, stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need_device(t, name):
    """A contiguous CUDA tensor of any type and shape (raw device memory)."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need(t, name, dtype, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def mgemm(x, w, offsets, transpose_B: bool = False, out=None, stream=None):
    """M-grouped BF16 GEMM.  x [M,K] bf16, w [E,N,K] (or [E,K,N] with
    transpose_B) bf16, offsets int32 [E+1]; returns y [M,N] bf16.  Rows of
    ``out`` at or past offsets[E] are left as they were."""
    import torch
    _need(x, "x", torch.bfloat16, 2)
    _need(w, "w", torch.bfloat16, 3)
    _need(offsets, "offsets", torch.int32, 1)
    M, K = x.shape
    E = w.shape[0]
    if transpose_B:
        if w.shape[1] != K:
            raise ValueError(f"w {tuple(w.shape)} does not match x {tuple(x.shape)} (want [E,K,N])")
        N = w.shape[2]
    else:
        if w.shape[2] != K:
            raise ValueError(f"w {tuple(w.shape)} does not match x {tuple(x.shape)} (want [E,N,K])")
        N = w.shape[1]
    if offsets.shape[0] != E + 1:
        raise ValueError(f"offsets must have E+1 = {E + 1} entries")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    else:
        _need(out, "out", torch.bfloat16, 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must be [{M},{N}]")
    lib = load()
    with torch.cuda.device(x.device):
        rc = lib.rg_mgemm(x.data_ptr(), w.data_ptr(), offsets.data_ptr(), E, M, N, K,
                          int(bool(transpose_B)), out.data_ptr(), _stream_ptr(x.device, stream))
    _check("rg_mgemm", rc)
    return out


def mgemm_nested(x, w, offsets, transpose_B: bool = False, out=None, stream=None):
    """Nested grouped GEMM, flattened into one launch.  x [M, O*K] bf16, w
    [O,L,N,K] (or [O,L,K,N] with transpose_B) bf16, offsets int32 [L+1];
    returns y [M, O*N] bf16 with y[r, o*N:(o+1)*N] = x[r, o*K:(o+1)*K] @ B_{o,l}
    for row r of inner group l.  Rows at or past offsets[L] are left as they
    were."""
    import torch
    _need(x, "x", torch.bfloat16, 2)
    _need(w, "w", torch.bfloat16, 4)
    _need(offsets, "offsets", torch.int32, 1)
    O, L = w.shape[0], w.shape[1]
    if transpose_B:
        K, N = w.shape[2], w.shape[3]
    else:
        N, K = w.shape[2], w.shape[3]
    M = x.shape[0]
    if x.shape[1] != O * K:
        raise ValueError(f"x {tuple(x.shape)} does not match w {tuple(w.shape)} (want [M, O*K])")
    if offsets.shape[0] != L + 1:
        raise ValueError(f"offsets must have L+1 = {L + 1} entries")
    if out is None:
        out = torch.empty((M, O * N), dtype=torch.bfloat16, device=x.device)
    else:
        _need(out, "out", torch.bfloat16, 2)
        if tuple(out.shape) != (M, O * N):
            raise ValueError(f"out must be [{M},{O * N}]")
    lib = load()
    with torch.cuda.device(x.device):
        rc = lib.rg_mgemm_nested(x.data_ptr(), w.data_ptr(), offsets.data_ptr(), O, L, M, N, K,
                                 int(bool(transpose_B)), out.data_ptr(), _stream_ptr(x.device, stream))
    _check("rg_mgemm_nested", rc)
    return out


def mx_blocked_bytes(R: int, KS: int, G: int) -> int:
    """Bytes ``mx_scales_blocked`` may write for R rows of KS scales in G groups."""
    n = load().rg_mx_blocked_bytes(int(R), int(KS), int(G))
    if n < 0:
        raise ValueError("bad arguments to rg_mx_blocked_bytes")
    return int(n)


def mx_scales_blocked(scales, offsets, out=None, stream=None):
    """Blocked ("128x4") layout of grouped E8M0 scales.  scales uint8 [R, KS]
    (device), offsets int32 [G+1] (device); returns uint8
    [mx_blocked_bytes(R, KS, G)] (bytes past the used blocks are unspecified)."""
    import torch
    _need(scales, "scales", torch.uint8, 2)
    _need(offsets, "offsets", torch.int32, 1)
    R, KS = scales.shape
    G = offsets.shape[0] - 1
    nbytes = mx_blocked_bytes(R, KS, G)
    if out is None:
        out = torch.empty((nbytes,), dtype=torch.uint8, device=scales.device)
    else:
        _need(out, "out", torch.uint8, 1)
        if out.numel() < nbytes:
            raise ValueError(f"out must hold at least {nbytes} bytes")
    lib = load()
    with torch.cuda.device(scales.device):
        rc = lib.rg_mx_scales_blocked(scales.data_ptr(), offsets.data_ptr(), G, R, KS, out.data_ptr(),
                                      out.numel(), _stream_ptr(scales.device, stream))
    _check("rg_mx_scales_blocked", rc)
    return out


def mx_weight_offsets(E: int, N: int, device="cuda"):
    """Offsets [E+1] that group a weight stack's scales [E*N, K/32] into E
    groups of N rows (for ``mx_scales_blocked`` of sw)."""
    import torch
    return torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device=device)


def mgemm_mxfp8(xq, sx_blocked, wq, sw_blocked, offsets, transpose_B: bool = False, out=None, stream=None):
    """MXFP8 M-grouped GEMM.  xq uint8 [M,K] E4M3 codes, wq uint8 [E,N,K] (or
    [E,K,N] with transpose_B), sx_blocked / sw_blocked uint8 blocked scales
    (``mx_scales_blocked`` of sx [M,K/32] with ``offsets`` and of sw
    [E*N,K/32] with ``mx_weight_offsets``), offsets int32 [E+1]; returns y
    [M,N] bf16."""
    import torch
    _need(xq, "xq", torch.uint8, 2)
    _need(wq, "wq", torch.uint8, 3)
    _need(sx_blocked, "sx_blocked", torch.uint8, 1)
    _need(sw_blocked, "sw_blocked", torch.uint8, 1)
    _need(offsets, "offsets", torch.int32, 1)
    M, K = xq.shape
    E = wq.shape[0]
    N = wq.shape[2] if transpose_B else wq.shape[1]
    if wq.shape[1 if transpose_B else 2] != K:
        raise ValueError(f"wq {tuple(wq.shape)} does not match xq {tuple(xq.shape)}")
    if offsets.shape[0] != E + 1:
        raise ValueError(f"offsets must have E+1 = {E + 1} entries")
    KS = K // 32
    if sx_blocked.numel() < mx_blocked_bytes(M, KS, E) or sw_blocked.numel() < mx_blocked_bytes(E * N, KS, E):
        raise ValueError("blocked scale buffers are smaller than mx_blocked_bytes")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    else:
        _need(out, "out", torch.bfloat16, 2)
        if tuple(out.shape) != (M, N):
            raise ValueError(f"out must be [{M},{N}]")
    lib = load()
    with torch.cuda.device(xq.device):
        rc = lib.rg_mgemm_mxfp8(xq.data_ptr(), sx_blocked.data_ptr(), wq.data_ptr(), sw_blocked.data_ptr(),
                                offsets.data_ptr(), E, M, N, K, int(bool(transpose_B)), out.data_ptr(),
                                _stream_ptr(xq.device, stream))
    _check("rg_mgemm_mxfp8", rc)
    return out


def mx_blocked_k_bytes(R: int, KS: int, G: int) -> int:
    """Bytes ``mx_scales_blocked_k`` may write for R rows of KS scales in G groups."""
    n = load().rg_mx_blocked_k_bytes(int(R), int(KS), int(G))
    if n < 0:
        raise ValueError("bad arguments to rg_mx_blocked_k_bytes")
    return int(n)


def mx_scales_blocked_k(scales, offsets, out=None, stream=None):
    """Blocked layout of E8M0 scales [R, KS] grouped along the contraction
    by offsets (device int32 [G+1], multiples of 32); returns uint8
    [mx_blocked_k_bytes(R, KS, G)]."""
    import torch
    _need(scales, "scales", torch.uint8, 2)
    _need(offsets, "offsets", torch.int32, 1)
    R, KS = scales.shape
    G = offsets.shape[0] - 1
    nbytes = mx_blocked_k_bytes(R, KS, G)
    if out is None:
        out = torch.empty((nbytes,), dtype=torch.uint8, device=scales.device)
    else:
        _need(out, "out", torch.uint8, 1)
        if out.numel() < nbytes:
            raise ValueError(f"out must hold at least {nbytes} bytes")
    lib = load()
    with torch.cuda.device(scales.device):
        rc = lib.rg_mx_scales_blocked_k(scales.data_ptr(), offsets.data_ptr(), G, R, KS, out.data_ptr(),
                                        out.numel(), _stream_ptr(scales.device, stream))
    _check("rg_mx_scales_blocked_k", rc)
    return out


def kgemm_mxfp8(gq, sg_blocked, xq, sx_blocked, offsets, out=None, accumulate: bool = False, stream=None):
    """MXFP8 K-grouped weight gradient.  gq uint8 [M,N], xq uint8 [M,K] (E4M3
    codes), sg_blocked / sx_blocked: ``mx_scales_blocked_k`` of sg [N,M/32]
    and sx [K,M/32] with ``offsets`` (int32 [E+1], multiples of 32).  Returns
    dW [E,N,K] fp32, overwritten, or added to ``out`` with accumulate=True."""
    import torch
    _need(gq, "gq", torch.uint8, 2)
    _need(xq, "xq", torch.uint8, 2)
    _need(sg_blocked, "sg_blocked", torch.uint8, 1)
    _need(sx_blocked, "sx_blocked", torch.uint8, 1)
    _need(offsets, "offsets", torch.int32, 1)
    M, N = gq.shape
    if xq.shape[0] != M:
        raise ValueError("gq and xq must have the same number of rows")
    K = xq.shape[1]
    E = offsets.shape[0] - 1
    if M % 32:
        raise ValueError("M must be a multiple of 32")
    if M and (sg_blocked.numel() < mx_blocked_k_bytes(N, M // 32, E)
              or sx_blocked.numel() < mx_blocked_k_bytes(K, M // 32, E)):
        raise ValueError("blocked scale buffers are smaller than mx_blocked_k_bytes")
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs the dW to add to as `out`")
        out = torch.empty((E, N, K), dtype=torch.float32, device=gq.device)
    else:
        _need(out, "out", torch.float32, 3)
        if tuple(out.shape) != (E, N, K):
            raise ValueError(f"out must be [{E},{N},{K}]")
    lib = load()
    with torch.cuda.device(gq.device):
        rc = lib.rg_kgemm_mxfp8(gq.data_ptr(), sg_blocked.data_ptr(), xq.data_ptr(), sx_blocked.data_ptr(),
                                offsets.data_ptr(), E, M, N, K, out.data_ptr(), int(bool(accumulate)),
                                _stream_ptr(gq.device, stream))
    _check("rg_kgemm_mxfp8", rc)
    return out


def mgemm_swiglu(x, w13, offsets, out=None, y13=False, stream=None):
    """Forward gate-up GEMM with SwiGLU in the epilogue.  x [M,K] bf16, w13
    [E,2F,K] bf16 (gate rows then up rows), offsets int32 [E+1]; returns h
    [M,F] bf16, or (h, y13) with y13 [M,2F] bf16 when ``y13`` is True (or a
    tensor to write into)."""
    import torch
    _need(x, "x", torch.bfloat16, 2)
    _need(w13, "w13", torch.bfloat16, 3)
    _need(offsets, "offsets", torch.int32, 1)
    M, K = x.shape
    E, N2 = w13.shape[0], w13.shape[1]
    if w13.shape[2] != K or N2 % 2:
        raise ValueError(f"w13 {tuple(w13.shape)} does not match x {tuple(x.shape)} (want [E,2F,K])")
    F = N2 // 2
    if offsets.shape[0] != E + 1:
        raise ValueError(f"offsets must have E+1 = {E + 1} entries")
    h = out if out is not None else torch.empty((M, F), dtype=torch.bfloat16, device=x.device)
    _need(h, "out", torch.bfloat16, 2)
    if tuple(h.shape) != (M, F):
        raise ValueError(f"out must be [{M},{F}]")
    y = None
    if y13 is not False and y13 is not None:
        y = torch.empty((M, N2), dtype=torch.bfloat16, device=x.device) if y13 is True else y13
        _need(y, "y13", torch.bfloat16, 2)
        if tuple(y.shape) != (M, N2):
            raise ValueError(f"y13 must be [{M},{N2}]")
    lib = load()
    with torch.cuda.device(x.device):
        rc = lib.rg_mgemm_swiglu(x.data_ptr(), w13.data_ptr(), offsets.data_ptr(), E, M, F, K,
                                 y.data_ptr() if y is not None else None, h.data_ptr(),
                                 _stream_ptr(x.device, stream))
    _check("rg_mgemm_swiglu", rc)
    return (h, y) if y is not None else h


def mgemm_swiglu_dgrad(dy, w2, offsets, y13, out=None, stream=None):
    """Input gradient of the down projection fused with the SwiGLU backward.
    dy [M,K] bf16, w2 [E,K,F] bf16 (forward layout of the down weight), y13
    [M,2F] bf16 saved by the forward pass; returns dy13 [M,2F] bf16."""
    import torch
    _need(dy, "dy", torch.bfloat16, 2)
    _need(w2, "w2", torch.bfloat16, 3)
    _need(offsets, "offsets", torch.int32, 1)
    _need(y13, "y13", torch.bfloat16, 2)
    M, K = dy.shape
    E, F = w2.shape[0], w2.shape[2]
    if w2.shape[1] != K:
        raise ValueError(f"w2 {tuple(w2.shape)} does not match dy {tuple(dy.shape)} (want [E,K,F])")
    if tuple(y13.shape) != (M, 2 * F):
        raise ValueError(f"y13 must be [{M},{2 * F}]")
    if offsets.shape[0] != E + 1:
        raise ValueError(f"offsets must have E+1 = {E + 1} entries")
    dy13 = out if out is not None else torch.empty((M, 2 * F), dtype=torch.bfloat16, device=dy.device)
    _need(dy13, "out", torch.bfloat16, 2)
    if tuple(dy13.shape) != (M, 2 * F):
        raise ValueError(f"out must be [{M},{2 * F}]")
    lib = load()
    with torch.cuda.device(dy.device):
        rc = lib.rg_mgemm_swiglu_dgrad(dy.data_ptr(), w2.data_ptr(), offsets.data_ptr(), E, M, F, K,
                                       y13.data_ptr(), dy13.data_ptr(), _stream_ptr(dy.device, stream))
    _check("rg_mgemm_swiglu_dgrad", rc)
    return dy13


def kgemm_workspace_bytes(E: int, N: int, K: int) -> int:
    """Bytes of the device workspace ``kgemm(..., workspace=)`` needs."""
    n = load().rg_kgemm_workspace_bytes(int(E), int(N), int(K))
    if n < 0:
        raise ValueError("bad E, N or K")
    return int(n)


def kgemm(grad, X, offsets, out=None, stream=None, accumulate: bool = False, workspace=None):
    """K-grouped weight gradient.  grad [M,N] bf16, X [M,K] bf16, offsets
    int32 [E+1]; returns dW [E,N,K] fp32, overwritten -- or, with
    ``accumulate=True``, added to the given ``out`` (e.g. an FP32 main grad).
    With ``workspace`` (a device tensor of at least kgemm_workspace_bytes
    bytes) the call runs rg_kgemm_ws: the same results, each row of a long
    expert read from DRAM once."""
    import torch
    _need(grad, "grad", torch.bfloat16, 2)
    _need(X, "X", torch.bfloat16, 2)
    _need(offsets, "offsets", torch.int32, 1)
    M, N = grad.shape
    if X.shape[0] != M:
        raise ValueError("grad and X must have the same number of rows")
    K = X.shape[1]
    E = offsets.shape[0] - 1
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs the dW to add to as `out`")
        out = torch.empty((E, N, K), dtype=torch.float32, device=grad.device)
    else:
        _need(out, "out", torch.float32, 3)
        if tuple(out.shape) != (E, N, K):
            raise ValueError(f"out must be [{E},{N},{K}]")
    lib = load()
    if workspace is not None:
        _need_device(workspace, "workspace")
        nbytes = workspace.numel() * workspace.element_size()
        with torch.cuda.device(grad.device):
            rc = lib.rg_kgemm_ws(grad.data_ptr(), X.data_ptr(), offsets.data_ptr(), E, M, N, K, out.data_ptr(),
                                 int(bool(accumulate)), workspace.data_ptr(), nbytes, _stream_ptr(grad.device, stream))
        _check("rg_kgemm_ws", rc)
        return out
    fn = lib.rg_kgemm_acc if accumulate else lib.rg_kgemm
    with torch.cuda.device(grad.device):
        rc = fn(grad.data_ptr(), X.data_ptr(), offsets.data_ptr(), E, M, N, K,
                out.data_ptr(), _stream_ptr(grad.device, stream))
    _check("rg_kgemm_acc" if accumulate else "rg_kgemm", rc)
    return out


def device_status(stream=None) -> int:
    """Return (and clear) the RG_DEV_* bits of the current device after the
    work queued on the stream; synchronises the stream."""
    import torch
    rc = load().rg_get_device_status(_stream_ptr(torch.cuda.current_device(), stream))
    if rc < 0:
        _check("rg_get_device_status", rc)
    return int(rc)


def shutdown() -> None:
    """Forget the per-device set-up (see rg_shutdown in include/rg.h)."""
    _check("rg_shutdown", load().rg_shutdown())


def set_wait_timeout_ns(ns: int) -> None:
    _check("rg_set_wait_timeout_ns", load().rg_set_wait_timeout_ns(int(ns)))


def selftest_wait_timeout(ns: int, stream=None) -> int:
    import torch
    v = ctypes.c_uint32(0)
    _check("rg_selftest_wait_timeout",
           load().rg_selftest_wait_timeout(int(ns), _stream_ptr(torch.cuda.current_device(), stream), ctypes.byref(v)))
    return int(v.value)
