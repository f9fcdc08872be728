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
    # Experts of several accumulation chunks and 90 dW tiles each (more than
    # the grid's CTA pairs), so that the kernel takes the chunk-major
    # schedule and hands tiles over through the flags in the fixed scratch.
    counts = [9000, 0, 37, 4100, 8192, 4033, 1]
    off = W.offsets_from_counts(counts)
    E, M, N, K = len(counts), int(off[-1]) + 5, 2560, 2304
    assert (N // 256) * (K // 256) > torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert gpu_lib.kgemm_workspace_bytes(E, N, K) <= 4 * gpu_lib.RG_KGEMM_NOALLOC_MAX_FLAGS
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
