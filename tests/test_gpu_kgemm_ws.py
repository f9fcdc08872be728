"""rg_kgemm_ws (chunk-major schedule, per-tile hand-over flags in a caller
workspace) against rg_kgemm and the oracle: the results must be
bit-identical to rg_kgemm's -- the same partial sums added in the same row
order -- for experts of one and of many accumulation chunks, overwrite and
accumulate, the 4-D and 3-D operand views, many chunk rounds over the grid,
the largest expert count, and the full-size skewed weight gradient."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import check_fp32, offsets_dev, to_dev

pytestmark = pytest.mark.gpu


def ints(shape, seed, stream):
    return W.integer_bf16(shape, -2, 2, seed, stream)


def both(rg, g, x, off, N, K, accumulate=False, init=None):
    """dW of rg_kgemm and of rg_kgemm_ws on the same inputs."""
    import torch
    E = len(off) - 1
    gd, xd, od = to_dev(g), to_dev(x), offsets_dev(off)
    outs = []
    for ws in (None, torch.empty(rg.kgemm_workspace_bytes(E, N, K), dtype=torch.uint8, device="cuda")):
        if accumulate:
            dW = torch.from_numpy(np.ascontiguousarray(init, dtype=np.float32)).cuda()
        else:
            dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device="cuda")
        rg.kgemm(gd, xd, od, out=dW, accumulate=accumulate, workspace=ws)
        torch.cuda.synchronize()
        assert rg.device_status() == 0
        outs.append(dW.cpu().numpy())
    return outs


LONG = [9000, 0, 37, 4100, 8192, 4032, 4033, 1, 12000]


@pytest.mark.parametrize("N,K", [(256, 320), (200, 136)], ids=["4d-views", "3d-views"])
def test_ws_bit_identical_random(gpu_lib, N, K):
    off = W.offsets_from_counts(LONG)
    M = int(off[-1]) + 3
    g = W.normal_bf16((M, N), 1.0, 41, 0)
    x = W.normal_bf16((M, K), 1.0, 41, 1)
    a, b = both(gpu_lib, g, x, off, N, K)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
    check_fp32(b, oracle.kgemm(g, x, off), f"kgemm_ws N={N} K={K}")


def test_ws_integer_bit_exact(gpu_lib):
    off = W.offsets_from_counts(LONG)
    M, N, K = int(off[-1]), 256, 256
    g, x = ints((M, N), 42, 0), ints((M, K), 42, 1)
    a, b = both(gpu_lib, g, x, off, N, K)
    np.testing.assert_array_equal(b.astype(np.float64), oracle.kgemm(g, x, off))
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_ws_accumulate_bit_identical(gpu_lib):
    off = W.offsets_from_counts(LONG)
    M, N, K = int(off[-1]), 256, 320
    g = W.normal_bf16((M, N), 1.0, 43, 0)
    x = W.normal_bf16((M, K), 1.0, 43, 1)
    init = W.bf16_bits_to_f32(W.normal_bf16((len(LONG), N, K), 1.0, 43, 2))
    a, b = both(gpu_lib, g, x, off, N, K, accumulate=True, init=init)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
    check_fp32(b, oracle.kgemm(g, x, off) + init.astype(np.float64), "kgemm_ws accumulate")
    assert (b[1] == init[1]).all()


def test_ws_many_rounds(gpu_lib):
    """20 tiles per expert and 5-chunk experts: each chunk's items spread
    over the grid and the flags hand tiles between CTAs many times."""
    counts = [20000, 130, 0, 16200, 7, 4032]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 1280, 1024
    g, x = ints((M, N), 44, 0), ints((M, K), 44, 1)
    a, b = both(gpu_lib, g, x, off, N, K)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))
    es = np.array([0, 0, 3, 3, 5], np.int32)
    ns = np.array([0, 1279, 17, 640, 300], np.int32)
    np.testing.assert_array_equal(b[es, ns].astype(np.float64), oracle.kgemm(g, x, off, sel=(es, ns)))


def test_ws_max_experts_and_reuse(gpu_lib):
    """1024 experts (three-stage ring, item tables at their largest), and the
    same workspace used by two calls in a row."""
    import torch
    rng = np.random.default_rng(45)
    counts = rng.integers(0, 6, size=1024)
    counts[[3, 500, 1023]] = [9000, 129, 4100]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 64, 72
    g = W.normal_bf16((M, N), 1.0, 45, 0)
    x = W.normal_bf16((M, K), 1.0, 45, 1)
    ref = oracle.kgemm(g, x, off)
    ws = torch.empty(gpu_lib.kgemm_workspace_bytes(1024, N, K), dtype=torch.uint8, device="cuda")
    plain = gpu_lib.kgemm(to_dev(g), to_dev(x), offsets_dev(off))
    for _ in range(2):
        dW = gpu_lib.kgemm(to_dev(g), to_dev(x), offsets_dev(off), workspace=ws)
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        assert torch.equal(dW.view(torch.int32), plain.view(torch.int32))
    check_fp32(dW.cpu().numpy(), ref, "kgemm_ws E=1024")


@pytest.mark.slow
def test_ws_full_size_skewed_gw13(gpu_lib):
    """The benchmark's skewed gw13 (Zipf experts up to 17.7k rows, 4 GB of
    dW): rg_kgemm_ws gives rg_kgemm's bits."""
    import torch
    wl = W.ALL["skewed"]()
    op = wl.op("wgrad_gw13")
    g, x = to_dev(wl.tensor(op.a)), to_dev(wl.tensor(op.b))
    off = offsets_dev(wl.offsets)
    a = gpu_lib.kgemm(g, x, off)
    ws = torch.empty(gpu_lib.kgemm_workspace_bytes(wl.E, op.N, op.K), dtype=torch.uint8, device="cuda")
    b = gpu_lib.kgemm(g, x, off, workspace=ws)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
