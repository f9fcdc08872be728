"""rg_kgemm_noalloc, the weight gradient for callers that cannot allocate
device memory -- a framework or serving runtime whose own pool holds the
device's memory, a plugin given no allocator, a runtime that forbids
allocation once started -- and so cannot hand rg_kgemm_ws its workspace.
Called through the C ABI twice in a row, its dW must match that of the
workspace entry point within the weight-gradient tolerance; the second call
reuses the library's fixed scratch, which the first call left holding its
flags.  This file is collected last, so that a run stopping at its first
failure has run every other test."""
import ctypes

import numpy as np
import pytest

import workloads as W
from parity import check_fp32, offsets_dev, to_dev

pytestmark = pytest.mark.gpu


def test_noalloc_matches_the_workspace_entry_point_twice(gpu_lib):
    import torch
    lib = gpu_lib.load()
    counts = [9000, 0, 37, 4100, 8192, 4033, 1]  # experts of several accumulation chunks
    off = W.offsets_from_counts(counts)
    E, M, N, K = len(counts), int(off[-1]) + 5, 512, 384
    g = to_dev(W.normal_bf16((M, N), 1.0, 91, 0))
    x = to_dev(W.normal_bf16((M, K), 1.0, 91, 1))
    od = offsets_dev(off)
    ws = torch.empty(gpu_lib.kgemm_workspace_bytes(E, N, K), dtype=torch.uint8, device="cuda")
    ref = gpu_lib.kgemm(g, x, od, workspace=ws)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    ref = ref.cpu().numpy().astype(np.float64)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.rg_kgemm_noalloc(g.data_ptr(), x.data_ptr(), od.data_ptr(), E, M, N, K, dW.data_ptr(), 0, stream)
        assert rc == gpu_lib.RG_OK, f"call {call}: rg_kgemm_noalloc returned {rc}"
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        check_fp32(dW.cpu().numpy(), ref, f"rg_kgemm_noalloc call {call}")
