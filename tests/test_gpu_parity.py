"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span
several tiles with ragged tails, plus the edge cases of grouping."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import (bf16_round_exact, check_bf16, check_fp32, offsets_dev, to_dev,
                    to_host_bits)

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = 0x4640  # 12288.0


def run_mgemm(rg, x, w, off, transpose_B, M, N, sentinel=True):
    import torch
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    if sentinel:
        y.view(torch.int16).fill_(SENTINEL_BF16)
    rg.mgemm(to_dev(x), to_dev(w), offsets_dev(off), transpose_B=transpose_B, out=y)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return to_host_bits(y)


def run_kgemm(rg, g, x, off, N, K):
    import torch
    E = len(off) - 1
    dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device="cuda")
    rg.kgemm(to_dev(g), to_dev(x), offsets_dev(off), out=dW)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return dW.cpu().numpy()


def ints(shape, seed, stream):
    return W.integer_bf16(shape, -2, 2, seed, stream)


# ------------------------------------------------------------ exact integers


INT_COUNTS = [130, 0, 1, 200]  # ragged, empty, single-row groups
INT_TAIL = 7                   # rows past offsets[E]


@pytest.mark.parametrize("transpose_B", [False, True], ids=["fwd", "dgrad"])
def test_mgemm_integer_inputs_bit_exact(gpu_lib, transpose_B):
    off = W.offsets_from_counts(INT_COUNTS)
    M, N, K = int(off[-1]) + INT_TAIL, 384, 320
    x = ints((M, K), 1, 0)
    w = ints((4, K, N) if transpose_B else (4, N, K), 1, 1)
    y = run_mgemm(gpu_lib, x, w, off, transpose_B, M, N)
    ref = oracle.mgemm(x, w, off, transpose_B=transpose_B)
    valid = int(off[-1])
    np.testing.assert_array_equal(y[:valid], bf16_round_exact(ref[:valid]))
    assert (y[valid:] == SENTINEL_BF16).all(), "rows past offsets[E] were written"


def test_kgemm_integer_inputs_bit_exact(gpu_lib):
    off = W.offsets_from_counts(INT_COUNTS)
    M, N, K = int(off[-1]) + INT_TAIL, 384, 320
    g = ints((M, N), 2, 0)
    x = ints((M, K), 2, 1)
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    ref = oracle.kgemm(g, x, off)
    np.testing.assert_array_equal(dW.astype(np.float64), ref)
    assert (dW[1] == 0).all()


@pytest.mark.parametrize("N,K", [(384, 320), (200, 136), (72, 520), (128, 64)],
                         ids=["wide-boxes", "3d-views", "narrow-N", "one-column-block"])
def test_kgemm_operand_views_bit_exact(gpu_lib, N, K):
    """Both operand-view forms: N and K multiples of 64 (one copy per operand
    and stage) and not (one copy per 64-column box, the last one clipped)."""
    counts = [130, 0, 1, 64, 200, 17]
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + 9
    g = ints((M, N), 10, 0)
    x = ints((M, K), 10, 1)
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    np.testing.assert_array_equal(dW.astype(np.float64), oracle.kgemm(g, x, off))


def test_kgemm_ragged_blocks_at_both_ends_bit_exact(gpu_lib):
    """Ragged last blocks of every kind: the first expert's only block starts
    at row 0, blocks of 1, 15, 16, 17, 63 and 65 rows, and the last expert ends
    at the last row of the operands (no rows past offsets[E])."""
    counts = [5, 1, 15, 16, 17, 0, 63, 65, 3]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 320, 384
    g = ints((M, N), 7, 0)
    x = ints((M, K), 7, 1)
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    np.testing.assert_array_equal(dW.astype(np.float64), oracle.kgemm(g, x, off))


def test_kgemm_nonfinite_rows_stay_in_their_expert(gpu_lib):
    """Inf and NaN in one expert's rows of grad and X reach only that expert's
    dW: the neighbouring experts' ragged blocks never contract them."""
    counts = [37, 50, 70, 9]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 256, 256
    g = ints((M, N), 8, 0)
    x = ints((M, K), 8, 1)
    lo, hi = int(off[1]), int(off[2])
    g[lo, 3] = 0x7F80       # +Inf (bf16 bits)
    g[hi - 1, 5] = 0x7FC0   # NaN
    x[lo + 1, 7] = 0xFF80   # -Inf
    x[hi - 1, 0] = 0x7FC0
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    ref = oracle.kgemm(g, x, off)
    for e in (0, 2, 3):
        np.testing.assert_array_equal(dW[e].astype(np.float64), ref[e])
    assert not np.isfinite(dW[1]).all()


def test_kgemm_long_experts_bit_exact(gpu_lib):
    """Experts longer than one accumulation chunk (4032 rows): the partial
    sums folded into dW must reproduce the exact integer result; chunk
    boundaries at 4032, 4033 and 8064 rows."""
    counts = [9000, 0, 4100, 37, 8192, 4032, 4033, 8064]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]) + 5, 256, 320
    g = ints((M, N), 3, 0)
    x = ints((M, K), 3, 1)
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    np.testing.assert_array_equal(dW.astype(np.float64), oracle.kgemm(g, x, off))


def test_kgemm_several_rounds_bit_exact(gpu_lib):
    """More tiles than CTA pairs (160 tiles: E=8 x 5 row blocks x 4 column
    blocks), so tiles of later rounds walk their expert's rows in the other
    direction; multi-chunk, ragged, single-row and empty experts included."""
    counts = [9000, 37, 0, 4100, 130, 1, 5000, 64]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]) + 3, 1280, 1024
    g = ints((M, N), 9, 0)
    x = ints((M, K), 9, 1)
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    np.testing.assert_array_equal(dW.astype(np.float64), oracle.kgemm(g, x, off))


@pytest.mark.parametrize("N,K,ws", [(1280, 1024, False), (2560, 2304, False), (2560, 2304, True)],
                         ids=["20-tiles", "90-tiles", "90-tiles-chunk-major"])
@pytest.mark.parametrize("accumulate", [False, True], ids=["overwrite", "accumulate"])
def test_kgemm_light_and_heavy_experts_bit_exact(gpu_lib, N, K, ws, accumulate):
    """Experts on both sides of the 512-row light/heavy threshold of the issue
    order (511, 512, 513 rows) beside empty, one-row, ragged and multi-chunk
    experts: light tiles run between the heavy tiles' row blocks, in the
    other tensor-memory buffer, and every dW element must still be the exact
    integer result; with 90 tiles per expert and a workspace the long experts
    take the chunk-major schedule at the same time."""
    import torch
    counts = [511, 9000, 0, 512, 1, 513, 4100, 97, 300, 2000, 96, 5000, 7]
    off = W.offsets_from_counts(counts)
    E, M = len(counts), int(off[-1]) + 2
    g, x = ints((M, N), 21, 0), ints((M, K), 21, 1)
    init = W.integer_bf16((E, N, K), -3, 3, 21, 2)
    dW = torch.from_numpy(W.bf16_bits_to_f32(init)).cuda() if accumulate else None
    ws_t = torch.empty(gpu_lib.kgemm_workspace_bytes(E, N, K), dtype=torch.uint8, device="cuda") if ws else None
    out = gpu_lib.kgemm(to_dev(g), to_dev(x), offsets_dev(off), out=dW, accumulate=accumulate, workspace=ws_t)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    got = out.cpu().numpy().astype(np.float64)
    if N * K <= 1280 * 1024:  # every element
        want = oracle.kgemm(g, x, off)
        if accumulate:
            want = want + W.bf16_bits_to_f32(init).astype(np.float64)
        np.testing.assert_array_equal(got, want)
    else:  # the first and last dW row of every expert and 64 others (the oracle row by row)
        rng = np.random.default_rng(21)
        es = np.concatenate([np.arange(E), np.arange(E), rng.integers(0, E, 64)]).astype(np.int32)
        ns = np.concatenate([np.zeros(E), np.full(E, N - 1), rng.integers(0, N, 64)]).astype(np.int32)
        want = oracle.kgemm(g, x, off, sel=(es, ns))
        if accumulate:
            want = want + W.bf16_bits_to_f32(init)[es, ns].astype(np.float64)
        np.testing.assert_array_equal(got[es, ns], want)


def test_kgemm_long_experts_random(gpu_lib):
    counts = [12000, 5000, 4032, 4033, 4096]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 384, 256
    g = W.normal_bf16((M, N), 1.0, 31, 0)
    x = W.normal_bf16((M, K), 1.0, 31, 1)
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    check_fp32(dW, oracle.kgemm(g, x, off), "long experts")


# ------------------------------------------------------------ accumulation


def run_kgemm_acc(rg, g, x, off, init):
    import torch
    dW = torch.from_numpy(np.ascontiguousarray(init, dtype=np.float32)).cuda()
    rg.kgemm(to_dev(g), to_dev(x), offsets_dev(off), out=dW, accumulate=True)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return dW.cpu().numpy()


def test_kgemm_accumulate_bit_exact(gpu_lib):
    """dW += sum: integer data keeps every partial sum exact, including the
    chunk-by-chunk additions of experts longer than 4032 rows; the empty
    expert keeps its initial values."""
    counts = [5000, 0, 130, 1]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]) + 3, 256, 192
    g = ints((M, N), 8, 0)
    x = ints((M, K), 8, 1)
    init = np.random.default_rng(8).integers(-50, 51, size=(4, N, K)).astype(np.float32)
    dW = run_kgemm_acc(gpu_lib, g, x, off, init)
    np.testing.assert_array_equal(dW.astype(np.float64), init.astype(np.float64) + oracle.kgemm(g, x, off))
    np.testing.assert_array_equal(dW[1], init[1])


def test_kgemm_accumulate_random(gpu_lib):
    counts = [3000, 700, 0, 6000]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]), 256, 512
    g = W.normal_bf16((M, N), 1.0, 33, 0)
    x = W.normal_bf16((M, K), 1.0, 33, 1)
    init = np.random.default_rng(9).standard_normal((4, N, K)).astype(np.float32) * 30
    dW = run_kgemm_acc(gpu_lib, g, x, off, init)
    check_fp32(dW, init.astype(np.float64) + oracle.kgemm(g, x, off), "accumulate")
    np.testing.assert_array_equal(dW[2], init[2])


# ------------------------------------------------------------ tiny workload


@pytest.mark.parametrize("opname", ["fwd", "dgrad", "wgrad"])
def test_tiny_workload(gpu_lib, opname):
    wl = W.tiny()
    op = wl.op(opname)
    a, b = wl.tensor(op.a), wl.tensor(op.b)
    off = wl.offsets
    if op.kind == "mgemm":
        y = run_mgemm(gpu_lib, a, b, off, op.transpose_B, wl.M, op.N)
        ref = oracle.mgemm(a, b, off, transpose_B=op.transpose_B)
        check_bf16(y, ref, opname)
    else:
        dW = run_kgemm(gpu_lib, a, b, off, op.N, op.K)
        check_fp32(dW, oracle.kgemm(a, b, off), opname)
        assert (dW[2] == 0).all()


# ------------------------------------------------------------ edge cases

EDGE = {
    "single_expert": dict(counts=[300], tail=0, N=256, K=128),
    "all_empty": dict(counts=[0, 0, 0], tail=64, N=128, K=64),
    "sizes_1_127_128_129": dict(counts=[0, 1, 127, 128, 129, 0], tail=3, N=256, K=192),
    "smallest_dims": dict(counts=[5, 0, 9], tail=2, N=8, K=8),
    "ragged_N_K": dict(counts=[70, 190], tail=0, N=200, K=72),
    "many_experts": dict(counts=list(np.random.default_rng(5).integers(0, 40, size=300)), tail=11, N=128, K=64),
}


@pytest.mark.parametrize("case", sorted(EDGE))
@pytest.mark.parametrize("kind", ["fwd", "dgrad", "wgrad"])
def test_edge_cases(gpu_lib, case, kind):
    c = EDGE[case]
    off = W.offsets_from_counts(c["counts"])
    E = len(c["counts"])
    M = int(off[-1]) + c["tail"]
    N, K = c["N"], c["K"]
    seed = 40 + sorted(EDGE).index(case)
    if kind == "wgrad":
        g = W.normal_bf16((M, N), 1.0, seed, 0)
        x = W.normal_bf16((M, K), 1.0, seed, 1)
        dW = run_kgemm(gpu_lib, g, x, off, N, K)
        check_fp32(dW, oracle.kgemm(g, x, off), f"{case}/{kind}")
        for e in range(E):
            if c["counts"][e] == 0:
                assert (dW[e] == 0).all()
        return
    tb = kind == "dgrad"
    x = W.normal_bf16((M, K), 1.0, seed, 0)
    w = W.normal_bf16((E, K, N) if tb else (E, N, K), 1.0 / np.sqrt(K), seed, 1)
    y = run_mgemm(gpu_lib, x, w, off, tb, M, N)
    valid = int(off[-1])
    if valid:
        check_bf16(y[:valid], oracle.mgemm(x, w, off, transpose_B=tb)[:valid], f"{case}/{kind}")
    assert (y[valid:] == SENTINEL_BF16).all()


def test_zero_rows(gpu_lib):
    import torch
    off = offsets_dev(np.zeros(4, dtype=np.int32))
    w = torch.zeros((3, 64, 64), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    y = gpu_lib.mgemm(x, w, off)
    assert y.shape == (0, 64)
    dW = torch.full((3, 64, 64), float("nan"), device="cuda")
    gpu_lib.kgemm(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"), x, off, out=dW)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    assert (dW == 0).all()


# ------------------------------------------------------------ medium random


def test_medium_random_all_ops(gpu_lib):
    """E=8 Dirichlet-routed rows, several tiles in every dimension."""
    counts = W.counts_dirichlet(8, 3000, 2.0, 21)
    off = W.offsets_from_counts(counts)
    M, D, F = 3000, 768, 512
    x = W.normal_bf16((M, D), 1.0, 21, 1)
    w = W.normal_bf16((8, F, D), 1.0 / np.sqrt(D), 21, 2)
    dy = W.normal_bf16((M, F), 1.0, 21, 3)
    y = run_mgemm(gpu_lib, x, w, off, False, M, F)
    check_bf16(y, oracle.mgemm(x, w, off), "fwd")
    dx = run_mgemm(gpu_lib, dy, w, off, True, M, D)
    check_bf16(dx, oracle.mgemm(dy, w, off, transpose_B=True), "dgrad")
    dW = run_kgemm(gpu_lib, dy, x, off, F, D)
    check_fp32(dW, oracle.kgemm(dy, x, off), "wgrad")


# ------------------------------------------------------------ status / robustness


def test_bad_offsets_set_status_and_write_nothing(gpu_lib):
    import torch
    M, N, K = 64, 128, 64
    x = to_dev(W.normal_bf16((M, K), 1.0, 7, 0))
    w = to_dev(W.normal_bf16((2, N, K), 1.0, 7, 1))
    for bad in ([0, 40, 30], [1, 10, 20], [0, 10, 65]):
        y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
        gpu_lib.mgemm(x, w, offsets_dev(np.array(bad)), out=y)
        assert gpu_lib.device_status() & gpu_lib.RG_DEV_BAD_OFFSETS
        assert (y == 3.0).all()
        dW = torch.full((2, N, K), 5.0, device="cuda")
        gpu_lib.kgemm(to_dev(W.normal_bf16((M, N), 1.0, 7, 2)), x, offsets_dev(np.array(bad)), out=dW)
        assert gpu_lib.device_status() & gpu_lib.RG_DEV_BAD_OFFSETS
        assert (dW == 5.0).all()
    # the status was cleared and good calls still work
    gpu_lib.mgemm(x, w, offsets_dev(np.array([0, 30, 64])))
    assert gpu_lib.device_status() == 0


def test_deterministic(gpu_lib):
    import torch
    wl = W.tiny()
    x = to_dev(wl.tensor("x"))
    w = to_dev(wl.tensor("w"))
    g = to_dev(wl.tensor("grad"))
    off = offsets_dev(wl.offsets)
    y1, y2 = gpu_lib.mgemm(x, w, off), gpu_lib.mgemm(x, w, off)
    d1, d2 = gpu_lib.kgemm(g, x, off), gpu_lib.kgemm(g, x, off)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))


def test_bounded_wait_times_out_with_status(gpu_lib):
    """A barrier nothing signals: the bounded wait gives up after ~50 ms and
    reports RG_DEV_TIMEOUT; the context stays usable."""
    import time
    import torch
    t0 = time.time()
    st = gpu_lib.selftest_wait_timeout(50_000_000)
    assert st == gpu_lib.RG_DEV_TIMEOUT
    assert time.time() - t0 < 10
    assert gpu_lib.device_status() == 0
    a = torch.ones(4, device="cuda")
    assert float(a.sum()) == 4.0


@pytest.mark.parametrize("E", [239, 240, 1024], ids=["deep-ring-limit", "shallow-ring", "max"])
def test_kgemm_most_experts(gpu_lib, E):
    """Many experts, most of them tiny or empty, against the oracle: 239 is
    the most whose tables fit beside the four-stage ring, 240 runs the
    three-stage ring, 1024 is RG_KGEMM_MAX_EXPERTS."""
    assert gpu_lib.RG_KGEMM_MAX_EXPERTS == 1024
    rng = np.random.default_rng(77)
    counts = rng.integers(0, 6, size=E)
    counts[[3, 200, E - 1]] = [400, 129, 64]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]) + 3, 64, 72
    g = W.normal_bf16((M, N), 1.0, 77, 0)
    x = W.normal_bf16((M, K), 1.0, 77, 1)
    dW = run_kgemm(gpu_lib, g, x, off, N, K)
    check_fp32(dW, oracle.kgemm(g, x, off), f"kgemm E={E}")
    assert (dW[np.flatnonzero(counts == 0)] == 0).all()
