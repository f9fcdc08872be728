"""The library's per-device set-up across rg_shutdown: the M-grouped GEMM, the
K-grouped weight gradient and its no-alloc form give the same bits before
and after a shutdown (the next call sets the device up again, including the
no-alloc entry point's look-up of its fixed array), with a clean status."""
import ctypes

import numpy as np
import pytest

import workloads as W
from parity import offsets_dev, to_dev

pytestmark = pytest.mark.gpu


def test_calls_before_and_after_shutdown_agree(gpu_lib):
    import torch
    lib = gpu_lib.load()
    counts = [700, 0, 37, 4100, 300]
    off = W.offsets_from_counts(counts)
    E, M, N, K = len(counts), int(off[-1]) + 3, 2560, 2304  # 90 dW tiles per expert: chunk-major
    x = to_dev(W.integer_bf16((M, K), -2, 2, 31, 0))
    w = to_dev(W.integer_bf16((E, N, K), -2, 2, 31, 1))
    g = to_dev(W.integer_bf16((M, N), -2, 2, 31, 2))
    od = offsets_dev(off)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def run():
        y = gpu_lib.mgemm(x, w, od)
        dw = gpu_lib.kgemm(g, x, od)
        dw2 = torch.full((E, N, K), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.rg_kgemm_noalloc(g.data_ptr(), x.data_ptr(), od.data_ptr(), E, M, N, K, dw2.data_ptr(), 0, stream)
        assert rc == gpu_lib.RG_OK
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        return y, dw, dw2

    y0, dw0, nd0 = run()
    assert torch.equal(nd0.view(torch.int32), dw0.view(torch.int32))
    gpu_lib.shutdown()
    y1, dw1, nd1 = run()
    valid = int(off[-1])  # rows past the last group are left untouched (unset here)
    assert torch.equal(y0[:valid].view(torch.int16), y1[:valid].view(torch.int16))
    assert torch.equal(dw0.view(torch.int32), dw1.view(torch.int32))
    assert torch.equal(nd1.view(torch.int32), dw1.view(torch.int32))
    assert np.isfinite(dw1.cpu().numpy()).all()
