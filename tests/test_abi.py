"""C-ABI checks that need no GPU: the library builds, loads, exports every
entry point include/rg.h declares, and rejects bad arguments on the host
before any CUDA call is made."""
import ctypes
import os
import re

import pytest

import moe_grouped_gemm_device_gb300 as rg
from moe_grouped_gemm_device_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()  # cross-compiles for sm_103a; no GPU needed
    return rg.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "rg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rg_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_symbols() == sorted(rg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert "sm_103a" in rg.version()


DEV = ctypes.c_void_p(0x10000)  # aligned stand-in address: never dereferenced on these paths
BAD = ctypes.c_void_p(0x10001)  # misaligned


@pytest.mark.parametrize(
    "args",
    [
        dict(x=None),                      # null x with rows
        dict(w=None),
        dict(offsets=None),
        dict(y=None),
        dict(x=BAD),                       # misaligned
        dict(offsets=ctypes.c_void_p(0x10002)),
        dict(E=0), dict(E=1025),
        dict(M=-1), dict(M=2**31),
        dict(N=0), dict(N=12), dict(K=4), dict(K=100),
    ],
)
def test_mgemm_rejects_bad_arguments(lib, args):
    a = dict(x=DEV, w=DEV, offsets=DEV, E=4, M=512, N=128, K=256, t=0, y=DEV, s=None)
    a.update(args)
    rc = lib.rg_mgemm(a["x"], a["w"], a["offsets"], a["E"], a["M"], a["N"], a["K"], a["t"], a["y"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


@pytest.mark.parametrize(
    "args",
    [dict(x=None), dict(w13=None), dict(offsets=None), dict(h=None), dict(h=BAD), dict(y13=BAD),
     dict(F=0), dict(F=4), dict(F=100), dict(F=2**30), dict(K=100), dict(E=0), dict(M=-1)],
)
def test_mgemm_swiglu_rejects_bad_arguments(lib, args):
    a = dict(x=DEV, w13=DEV, offsets=DEV, E=4, M=512, F=128, K=256, y13=None, h=DEV, s=None)
    a.update(args)
    rc = lib.rg_mgemm_swiglu(a["x"], a["w13"], a["offsets"], a["E"], a["M"], a["F"], a["K"],
                             a["y13"], a["h"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


@pytest.mark.parametrize(
    "args",
    [dict(dy=None), dict(w2=None), dict(y13=None), dict(dy13=None), dict(y13=BAD), dict(F=4),
     dict(F=100), dict(K=12), dict(E=0), dict(M=-1),
     dict(dy13=ctypes.c_void_p(0x10000 + 512 * 256 * 2 - 16)),  # overlaps y13
     dict(y13=ctypes.c_void_p(0x10000 + 512 * 256 * 2 - 16))],
)
def test_mgemm_swiglu_dgrad_rejects_bad_arguments(lib, args):
    a = dict(dy=DEV, w2=DEV, offsets=DEV, E=4, M=512, F=128, K=256, y13=DEV,
             dy13=ctypes.c_void_p(0x10000 + 512 * 256 * 2), s=None)
    a.update(args)
    rc = lib.rg_mgemm_swiglu_dgrad(a["dy"], a["w2"], a["offsets"], a["E"], a["M"], a["F"], a["K"],
                                   a["y13"], a["dy13"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


@pytest.mark.parametrize(
    "args",
    [dict(grad=None), dict(X=None), dict(dW=None), dict(offsets=None), dict(dW=BAD),
     dict(E=0), dict(E=rg.RG_KGEMM_MAX_EXPERTS + 1), dict(N=7), dict(K=0), dict(M=-5)],
)
@pytest.mark.parametrize("fn", ["rg_kgemm", "rg_kgemm_acc"])
def test_kgemm_rejects_bad_arguments(lib, args, fn):
    a = dict(grad=DEV, X=DEV, offsets=DEV, E=4, M=512, N=128, K=256, dW=DEV, s=None)
    a.update(args)
    rc = getattr(lib, fn)(a["grad"], a["X"], a["offsets"], a["E"], a["M"], a["N"], a["K"], a["dW"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


def test_other_entry_points_validate(lib):
    assert lib.rg_set_wait_timeout_ns(0) == rg.RG_ERR_INVALID_ARG
    assert lib.rg_set_wait_timeout_ns(999_999) == rg.RG_ERR_INVALID_ARG  # below the 1 ms floor
    assert lib.rg_set_wait_timeout_ns(1_000_000) == rg.RG_OK
    assert lib.rg_set_wait_timeout_ns(2_000_000_000) == rg.RG_OK
    assert lib.rg_selftest_wait_timeout(0, None, None) == rg.RG_ERR_INVALID_ARG


def test_kgemm_workspace_entry_points_validate(lib):
    # one 4-byte flag per expert, 256 x 256 dW tile and CTA of the pair
    assert lib.rg_kgemm_workspace_bytes(4, 128, 256) == 4 * 1 * 1 * 2 * 4
    assert lib.rg_kgemm_workspace_bytes(128, 2560, 3072) == 128 * 10 * 12 * 2 * 4
    assert lib.rg_kgemm_workspace_bytes(1024, 257, 1) == 1024 * 2 * 1 * 2 * 4
    for bad in ((0, 128, 128), (1025, 128, 128), (4, 0, 128), (4, 128, 0)):
        assert lib.rg_kgemm_workspace_bytes(*bad) == -1
    need = lib.rg_kgemm_workspace_bytes(4, 128, 256)
    args = (DEV, DEV, DEV, 4, 512, 128, 256, DEV, 0)
    assert lib.rg_kgemm_ws(*args, None, need, None) == rg.RG_ERR_INVALID_ARG       # no workspace
    assert lib.rg_kgemm_ws(*args, ctypes.c_void_p(0x10002), need, None) == rg.RG_ERR_INVALID_ARG  # misaligned
    assert lib.rg_kgemm_ws(*args, DEV, need - 4, None) == rg.RG_ERR_INVALID_ARG    # too small
    bad_e = (DEV, DEV, DEV, 0, 512, 128, 256, DEV, 0)
    assert lib.rg_kgemm_ws(*bad_e, DEV, 1 << 20, None) == rg.RG_ERR_INVALID_ARG


def test_kgemm_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 1024 experts of 32 x 32 dW tiles need 2M flags, more than the fixed
    # scratch holds: refused before any device work
    assert lib.rg_kgemm_workspace_bytes(1024, 8192, 8192) > 4 * rg.RG_KGEMM_NOALLOC_MAX_FLAGS
    rc = lib.rg_kgemm_noalloc(DEV, DEV, DEV, 1024, 512, 8192, 8192, DEV, 0, None)
    assert rc == rg.RG_ERR_SCRATCH
    assert lib.rg_kgemm_noalloc(DEV, DEV, DEV, 0, 512, 128, 128, DEV, 0, None) == rg.RG_ERR_INVALID_ARG


def test_status_and_shutdown_without_a_device(lib):
    """rg_get_device_status returns the bits (>= 0) or a negative error: with
    no device it is an error, never bits; rg_shutdown releases nothing and
    always succeeds."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.rg_get_device_status(None) in (rg.RG_ERR_CUDA, rg.RG_ERR_UNSUPPORTED)
    assert lib.rg_shutdown() == rg.RG_OK
    assert lib.rg_shutdown() == rg.RG_OK


def test_no_device_reports_unsupported_or_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.rg_device_supported() == 0
    # a well-formed call reaches the device query and fails cleanly
    rc = lib.rg_mgemm(DEV, DEV, DEV, 4, 512, 128, 256, 0, DEV, None)
    assert rc in (rg.RG_ERR_CUDA, rg.RG_ERR_UNSUPPORTED)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(rg, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        rg.load()


@pytest.mark.parametrize(
    "args",
    [dict(x=None), dict(w=None), dict(offsets=None), dict(y=None), dict(x=BAD), dict(O=0), dict(O=-2),
     dict(O=rg.RG_MAX_OUTER + 1), dict(L=0), dict(L=1025), dict(N=12), dict(K=4), dict(M=-1),
     dict(O=65536, N=65536)],  # O*N past int32
)
def test_mgemm_nested_rejects_bad_arguments(lib, args):
    a = dict(x=DEV, w=DEV, offsets=DEV, O=2, L=4, M=512, N=128, K=16, t=0, y=DEV, s=None)
    a.update(args)
    rc = lib.rg_mgemm_nested(a["x"], a["w"], a["offsets"], a["O"], a["L"], a["M"], a["N"], a["K"], a["t"],
                             a["y"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


@pytest.mark.parametrize(
    "args",
    [dict(xq=None), dict(sx=None), dict(wq=None), dict(sw=None), dict(offsets=None), dict(y=None),
     dict(xq=BAD), dict(sw=BAD), dict(E=0), dict(E=1025), dict(M=-1), dict(N=8), dict(N=40), dict(K=16),
     dict(K=48)],
)
def test_mgemm_mxfp8_rejects_bad_arguments(lib, args):
    a = dict(xq=DEV, sx=DEV, wq=DEV, sw=DEV, offsets=DEV, E=4, M=512, N=128, K=256, t=0, y=DEV, s=None)
    a.update(args)
    rc = lib.rg_mgemm_mxfp8(a["xq"], a["sx"], a["wq"], a["sw"], a["offsets"], a["E"], a["M"], a["N"], a["K"],
                            a["t"], a["y"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


@pytest.mark.parametrize(
    "args",
    [dict(gq=None), dict(sg=None), dict(xq=None), dict(sx=None), dict(offsets=None), dict(dW=None),
     dict(dW=BAD), dict(E=0), dict(M=-32), dict(M=100), dict(N=8), dict(K=24)],
)
def test_kgemm_mxfp8_rejects_bad_arguments(lib, args):
    a = dict(gq=DEV, sg=DEV, xq=DEV, sx=DEV, offsets=DEV, E=4, M=512, N=128, K=256, dW=DEV, acc=0, s=None)
    a.update(args)
    rc = lib.rg_kgemm_mxfp8(a["gq"], a["sg"], a["xq"], a["sx"], a["offsets"], a["E"], a["M"], a["N"], a["K"],
                            a["dW"], a["acc"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


def test_mx_scale_layout_entry_points_validate(lib):
    assert lib.rg_mx_blocked_bytes(300, 7, 6) == (300 // 128 + 6) * 2 * 512
    assert lib.rg_mx_blocked_bytes(-1, 7, 6) == -1 and lib.rg_mx_blocked_bytes(10, 0, 1) == -1
    assert lib.rg_mx_blocked_k_bytes(300, 10, 3) == 3 * (10 // 4 + 3) * 512
    assert lib.rg_mx_blocked_k_bytes(0, 10, 3) == -1
    need = lib.rg_mx_blocked_bytes(512, 8, 4)
    for fn, n in (("rg_mx_scales_blocked", need), ("rg_mx_scales_blocked_k", lib.rg_mx_blocked_k_bytes(512, 8, 4))):
        f = getattr(lib, fn)
        assert f(DEV, DEV, 4, 512, 8, DEV, n - 1, None) == rg.RG_ERR_INVALID_ARG  # too small
        assert f(DEV, None, 4, 512, 8, DEV, n, None) == rg.RG_ERR_INVALID_ARG
        assert f(DEV, DEV, 4, 512, 8, BAD, n, None) == rg.RG_ERR_INVALID_ARG
        assert f(DEV, DEV, 0, 512, 8, DEV, n, None) == rg.RG_ERR_INVALID_ARG
        assert f(DEV, DEV, 4, 512, 0, DEV, n, None) == rg.RG_ERR_INVALID_ARG


def test_oracle_blocked_sizes_match_the_library(lib):
    """The size bounds the library states equal the oracle's (both written
    from the same definition of the layouts, checked here against each other)."""
    import oracle
    for R, KS, G in ((300, 7, 6), (1, 1, 1), (65536, 96, 128), (0, 3, 2)):
        assert lib.rg_mx_blocked_bytes(R, KS, G) == oracle.mx_blocked_bytes(R, KS, G)
    for R, KS, G in ((300, 10, 3), (2560, 1024, 32), (1, 1, 1)):
        assert lib.rg_mx_blocked_k_bytes(R, KS, G) == oracle.mx_blocked_k_bytes(R, KS, G)


def host_calls():
    """Every compute entry point of the binding, called with host (CPU)
    tensors of the right types and shapes."""
    import torch
    bf, u8, i32 = torch.bfloat16, torch.uint8, torch.int32
    off = torch.tensor([0, 32, 64], dtype=i32)
    x, w = torch.zeros(64, 64, dtype=bf), torch.zeros(2, 64, 64, dtype=bf)
    q, wq, s = torch.zeros(64, 64, dtype=u8), torch.zeros(2, 64, 64, dtype=u8), torch.zeros(4096, dtype=u8)
    return {
        "mgemm": lambda: rg.mgemm(x, w, off),
        "mgemm_dgrad": lambda: rg.mgemm(x, w, off, transpose_B=True),
        "mgemm_nested": lambda: rg.mgemm_nested(torch.zeros(64, 128, dtype=bf),
                                                torch.zeros(2, 2, 64, 64, dtype=bf), off),
        "mgemm_swiglu": lambda: rg.mgemm_swiglu(x, torch.zeros(2, 128, 64, dtype=bf), off),
        "mgemm_swiglu_dgrad": lambda: rg.mgemm_swiglu_dgrad(x, w, off, torch.zeros(64, 128, dtype=bf)),
        "kgemm": lambda: rg.kgemm(x, x, off),
        "mgemm_mxfp8": lambda: rg.mgemm_mxfp8(q, s, wq, s, off),
        "kgemm_mxfp8": lambda: rg.kgemm_mxfp8(q, s, q, s, off),
        "mx_scales_blocked": lambda: rg.mx_scales_blocked(torch.zeros(64, 2, dtype=u8), off),
        "mx_scales_blocked_k": lambda: rg.mx_scales_blocked_k(torch.zeros(64, 2, dtype=u8), off),
    }


@pytest.mark.parametrize("name", sorted(host_calls()))
def test_binding_refuses_host_tensors(lib, name):
    """No CPU fallback: every compute call refuses host tensors loudly
    instead of computing anything."""
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        host_calls()[name]()


def test_binding_checks_types_and_shapes(lib):
    """Type and rank checks come before the device check (host tensors here,
    so only the first argument's checks are reachable)."""
    import torch
    off = torch.tensor([0, 32, 64], dtype=torch.int32)
    x, w = torch.zeros(64, 64, dtype=torch.bfloat16), torch.zeros(2, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="bfloat16"):
        rg.mgemm(x.float(), w, off)
    with pytest.raises(ValueError, match="2-D"):
        rg.mgemm(x[0], w, off)
    with pytest.raises(TypeError, match="torch.Tensor"):
        rg.kgemm([0], x, off)
    with pytest.raises(TypeError, match="uint8"):
        rg.mx_scales_blocked(torch.zeros(64, 2, dtype=torch.int8), off)
