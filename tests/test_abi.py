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
     dict(E=0), dict(N=7), dict(K=0), dict(M=-5)],
)
@pytest.mark.parametrize("fn", ["rg_kgemm", "rg_kgemm_acc"])
def test_kgemm_rejects_bad_arguments(lib, args, fn):
    a = dict(grad=DEV, X=DEV, offsets=DEV, E=4, M=512, N=128, K=256, dW=DEV, s=None)
    a.update(args)
    rc = getattr(lib, fn)(a["grad"], a["X"], a["offsets"], a["E"], a["M"], a["N"], a["K"], a["dW"], a["s"])
    assert rc == rg.RG_ERR_INVALID_ARG


def test_other_entry_points_validate(lib):
    assert lib.rg_set_wait_timeout_ns(0) == rg.RG_ERR_INVALID_ARG
    assert lib.rg_set_wait_timeout_ns(2_000_000_000) == rg.RG_OK
    assert lib.rg_get_device_status(None, None) == rg.RG_ERR_INVALID_ARG
    assert lib.rg_selftest_wait_timeout(0, None, None) == rg.RG_ERR_INVALID_ARG


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
