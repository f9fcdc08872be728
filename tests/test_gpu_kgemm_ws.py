"""rg_kgemm_ws (chunk-major schedule, per-tile hand-over flags in a caller
workspace) against rg_kgemm and the oracle: the results must be
bit-identical to rg_kgemm's -- the same partial sums added in the same row
order.  The kernel takes the chunk-major schedule only when an expert has
more dW tiles than the grid has CTA pairs (half the SMs) and some expert is
longer than one accumulation chunk, so the shapes here have more than 76
tiles of 256 x 256 per expert: experts of one and of many chunks, overwrite
and accumulate, the 4-D and 3-D operand views, many chunk rounds, the
largest expert count, the full-size skewed weight gradient.  Shapes with
fewer tiles per expert take rg_kgemm's schedule, also checked."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import check_fp32, offsets_dev, to_dev

pytestmark = pytest.mark.gpu


def ints(shape, seed, stream):
    return W.integer_bf16(shape, -2, 2, seed, stream)


def chunk_mode_shape(N, K):
    """The shape has more tiles per expert than the grid has CTA pairs."""
    import torch
    tpe = -(-N // 256) * -(-K // 256)
    assert tpe > torch.cuda.get_device_properties(0).multi_processor_count // 2, (N, K, tpe)


def sample(off, N, seed, n=48):
    """(experts, ns) for n rows of dW: the first and last row of every
    non-empty expert, the rest at random."""
    counts = np.diff(off)
    live = np.flatnonzero(counts)
    rng = np.random.default_rng(seed)
    es = np.concatenate([live, live, rng.choice(live, n)]).astype(np.int32)
    ns = np.concatenate([np.zeros(len(live)), np.full(len(live), N - 1), rng.integers(0, N, n)]).astype(np.int32)
    return es, ns


def both(rg, g, x, off, N, K, accumulate=False, init=None):
    """dW of rg_kgemm and of rg_kgemm_ws on the same inputs (device tensors)."""
    import torch
    E = len(off) - 1
    gd, xd, od = to_dev(g), to_dev(x), offsets_dev(off)
    outs = []
    for ws in (None, torch.empty(rg.kgemm_workspace_bytes(E, N, K), dtype=torch.uint8, device="cuda")):
        if accumulate:
            dW = init.clone()
        else:
            dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device="cuda")
        rg.kgemm(gd, xd, od, out=dW, accumulate=accumulate, workspace=ws)
        torch.cuda.synchronize()
        assert rg.device_status() == 0
        outs.append(dW)
    return outs


def same_bits(a, b):
    import torch
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def rows(dW, es, ns):
    import torch
    return dW[torch.from_numpy(es).long().cuda(), torch.from_numpy(ns).long().cuda()].cpu().numpy()


LONG = [9000, 0, 37, 4100, 8192, 4032, 4033, 1, 12000]


@pytest.mark.parametrize("N,K", [(2560, 2304), (2248, 2120)], ids=["4d-views", "3d-views"])
def test_ws_bit_identical_random(gpu_lib, N, K):
    chunk_mode_shape(N, K)
    off = W.offsets_from_counts(LONG)
    M = int(off[-1]) + 3
    g = W.normal_bf16((M, N), 1.0, 41, 0)
    x = W.normal_bf16((M, K), 1.0, 41, 1)
    a, b = both(gpu_lib, g, x, off, N, K)
    same_bits(a, b)
    es, ns = sample(off, N, 41)
    check_fp32(rows(b, es, ns), oracle.kgemm(g, x, off, sel=(es, ns)), f"kgemm_ws N={N} K={K}")
    assert bool((b[1] == 0).all())


def test_ws_integer_bit_exact(gpu_lib):
    off = W.offsets_from_counts(LONG)
    M, N, K = int(off[-1]), 2304, 2304
    chunk_mode_shape(N, K)
    g, x = ints((M, N), 42, 0), ints((M, K), 42, 1)
    a, b = both(gpu_lib, g, x, off, N, K)
    same_bits(a, b)
    es, ns = sample(off, N, 42, 96)
    np.testing.assert_array_equal(rows(b, es, ns).astype(np.float64), oracle.kgemm(g, x, off, sel=(es, ns)))


def test_ws_accumulate_bit_identical(gpu_lib):
    import torch
    off = W.offsets_from_counts(LONG)
    M, N, K = int(off[-1]), 2304, 2560
    chunk_mode_shape(N, K)
    g = W.normal_bf16((M, N), 1.0, 43, 0)
    x = W.normal_bf16((M, K), 1.0, 43, 1)
    init = to_dev(W.normal_bf16((len(LONG), N, K), 1.0, 43, 2)).float()
    a, b = both(gpu_lib, g, x, off, N, K, accumulate=True, init=init)
    same_bits(a, b)
    es, ns = sample(off, N, 43)
    ref = oracle.kgemm(g, x, off, sel=(es, ns)) + rows(init, es, ns).astype(np.float64)
    check_fp32(rows(b, es, ns), ref, "kgemm_ws accumulate")
    assert torch.equal(b[1], init[1])


def test_ws_many_rounds(gpu_lib):
    """90 tiles per expert and 5-chunk experts: each chunk's items spread
    over the grid and the flags hand tiles between CTAs many times."""
    counts = [20000, 130, 0, 16200, 7, 4032]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 2560, 2304
    chunk_mode_shape(N, K)
    g, x = ints((M, N), 44, 0), ints((M, K), 44, 1)
    a, b = both(gpu_lib, g, x, off, N, K)
    same_bits(a, b)
    es, ns = sample(off, N, 44)
    np.testing.assert_array_equal(rows(b, es, ns).astype(np.float64), oracle.kgemm(g, x, off, sel=(es, ns)))


@pytest.mark.parametrize("N,K", [(256, 320), (1280, 1024)], ids=["2-tiles", "20-tiles"])
def test_ws_few_tiles_takes_the_tile_schedule(gpu_lib, N, K):
    """Fewer tiles per expert than CTA pairs: rg_kgemm's schedule, the same bits."""
    off = W.offsets_from_counts(LONG)
    M = int(off[-1])
    g = W.normal_bf16((M, N), 1.0, 46, 0)
    x = W.normal_bf16((M, K), 1.0, 46, 1)
    a, b = both(gpu_lib, g, x, off, N, K)
    same_bits(a, b)
    es, ns = sample(off, N, 46)
    check_fp32(rows(b, es, ns), oracle.kgemm(g, x, off, sel=(es, ns)), f"kgemm_ws N={N} K={K}")


def test_ws_max_experts_and_reuse(gpu_lib):
    """1024 experts (three-stage ring, item tables at their largest) of 81
    tiles each, and the same workspace used by two calls in a row."""
    import torch
    rng = np.random.default_rng(45)
    counts = rng.integers(0, 6, size=1024)
    counts[[3, 500, 1023]] = [9000, 129, 4100]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 2304, 2304
    chunk_mode_shape(N, K)
    g = W.normal_bf16((M, N), 1.0, 45, 0)
    x = W.normal_bf16((M, K), 1.0, 45, 1)
    gd, xd, od = to_dev(g), to_dev(x), offsets_dev(off)
    ws = torch.empty(gpu_lib.kgemm_workspace_bytes(1024, N, K), dtype=torch.uint8, device="cuda")
    plain = gpu_lib.kgemm(gd, xd, od)
    dW = torch.empty_like(plain)
    for _ in range(2):
        dW.fill_(float("nan"))
        gpu_lib.kgemm(gd, xd, od, out=dW, workspace=ws)
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        same_bits(dW, plain)
    es, ns = sample(off, N, 45, 64)
    es = np.concatenate([es, [3, 3, 500, 1023, 1023]]).astype(np.int32)
    ns = np.concatenate([ns, [1, 2303, 1000, 0, 2000]]).astype(np.int32)
    check_fp32(rows(dW, es, ns), oracle.kgemm(g, x, off, sel=(es, ns)), "kgemm_ws E=1024")


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
