"""GPU parity of the nested grouped GEMM (CUTLASS discussion #1452: outer
groups over the columns of x and y, inner row groups over a shared offsets
vector, flattened into one launch) against the CPU oracle, through the C ABI."""
import ctypes
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from parity import bf16_round_exact, check_bf16, offsets_dev, to_dev, to_host_bits

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = 0x4640  # 12288.0


def run_nested(rg, x, w, off, transpose_B, M, O, N):
    import torch
    y = torch.empty((M, O * N), dtype=torch.bfloat16, device="cuda")
    y.view(torch.int16).fill_(SENTINEL_BF16)
    rg.mgemm_nested(to_dev(x), to_dev(w), offsets_dev(off), transpose_B=transpose_B, out=y)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return to_host_bits(y)


@pytest.mark.parametrize("transpose_B", [False, True], ids=["fwd", "dgrad"])
@pytest.mark.parametrize("O", [1, 3])
@pytest.mark.parametrize("K", [320, 16, 32], ids=["k320", "k16", "k32"])
def test_nested_integer_inputs_bit_exact(gpu_lib, transpose_B, O, K):
    """K = 320: pair tiles; K = 16 / 32: single-CTA one-stage tiles with 16- /
    32-column operand boxes, through the outer groups' 3-D activation map."""
    counts = [130, 0, 1, 200, 0]
    off = W.offsets_from_counts(counts)
    L, N = len(counts), 192  # N: one partial 256-column tile per outer group
    M = int(off[-1]) + 9
    x = W.integer_bf16((M, O * K), -2, 2, 21, 0)
    w = W.integer_bf16((O, L, K, N) if transpose_B else (O, L, N, K), -2, 2, 21, 1)
    y = run_nested(gpu_lib, x, w, off, transpose_B, M, O, N)
    ref = oracle.mgemm_nested(x, w, off, transpose_B=transpose_B)
    valid = int(off[-1])
    np.testing.assert_array_equal(y[:valid], bf16_round_exact(ref[:valid]))
    assert (y[valid:] == SENTINEL_BF16).all(), "rows past offsets[L] were written"


@pytest.mark.parametrize("O,N,K", [(2, 640, 16), (3, 16, 512), (2, 8, 8), (4, 136, 72)],
                         ids=["expand_r16", "shrink_N16", "tiny_8x8", "odd_136x72"])
def test_nested_lora_shapes(gpu_lib, O, N, K):
    """LoRA-sized contractions (K = rank) and outputs (N = rank), K and N
    below one 64-wide k-block or 256-wide tile: the outer groups' column
    blocks must not bleed into each other."""
    rng = np.random.default_rng(zlib.crc32(f"lora/{O}/{N}/{K}".encode()))
    L = 12
    counts = rng.multinomial(3000, [1 / L] * L)
    counts[[0, 7]] = 0
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + 3
    x = W.normal_bf16((M, O * K), 1.0, 31, O * 1000 + N)
    w = W.normal_bf16((O, L, N, K), 1.0 / np.sqrt(K), 31, O * 1000 + N + 1)
    y = run_nested(gpu_lib, x, w, off, False, M, O, N)
    ref = oracle.mgemm_nested(x, w, off)
    valid = int(off[-1])
    check_bf16(y[:valid], ref[:valid], f"nested O={O} N={N} K={K}")
    assert (y[valid:] == SENTINEL_BF16).all()


@pytest.mark.parametrize("transpose_B,N,K", [(False, 8, 8), (True, 16, 8), (False, 72, 8)],
                         ids=["fwd-narrow", "dgrad", "fwd-partial-tile"])
def test_nested_max_outer_bit_exact(gpu_lib, transpose_B, N, K):
    """RG_MAX_OUTER outer groups: the tile index (inner tile x O + o) and the
    weight slot (o x L + l) at their largest, every outer group's column
    block in its place."""
    O = gpu_lib.RG_MAX_OUTER
    counts = [3, 0, 130]
    off = W.offsets_from_counts(counts)
    L = len(counts)
    M = int(off[-1]) + 2
    x = W.integer_bf16((M, O * K), -2, 2, 23, 0)
    w = W.integer_bf16((O, L, K, N) if transpose_B else (O, L, N, K), -2, 2, 23, 1)
    y = run_nested(gpu_lib, x, w, off, transpose_B, M, O, N)
    ref = oracle.mgemm_nested(x, w, off, transpose_B=transpose_B)
    valid = int(off[-1])
    np.testing.assert_array_equal(y[:valid], bf16_round_exact(ref[:valid]))
    assert (y[valid:] == SENTINEL_BF16).all()


def test_nested_outer_one_equals_mgemm(gpu_lib):
    """O = 1 is the plain grouped GEMM: same kernel, bit-identical output."""
    import torch
    rng = np.random.default_rng(41)
    counts = rng.multinomial(2000, [0.25] * 4)
    off = W.offsets_from_counts(counts)
    x = to_dev(W.normal_bf16((2000, 256), 1.0, 41, 0))
    w = to_dev(W.normal_bf16((4, 384, 256), 1 / 16, 41, 1))
    d = offsets_dev(off)
    a = gpu_lib.mgemm(x, w, d)
    b = gpu_lib.mgemm_nested(x, w.view(1, 4, 384, 256), d)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_nested_flattened_blocks_equal_separate_calls(gpu_lib):
    """Column block o of one nested launch equals a separate rg_mgemm on x's
    column slice o with the weight stack w[o] (the flattening is exact)."""
    import torch
    rng = np.random.default_rng(42)
    O, L, N, K = 3, 6, 256, 128
    counts = rng.multinomial(1500, [1 / L] * L)
    off = W.offsets_from_counts(counts)
    x = to_dev(W.normal_bf16((1500, O * K), 1.0, 42, 0))
    w = to_dev(W.normal_bf16((O, L, N, K), 1 / np.sqrt(K), 42, 1))
    d = offsets_dev(off)
    y = gpu_lib.mgemm_nested(x, w, d)
    for o in range(O):
        yo = gpu_lib.mgemm(x[:, o * K:(o + 1) * K].contiguous(), w[o].contiguous(), d)
        torch.cuda.synchronize()
        assert torch.equal(y[:, o * N:(o + 1) * N].contiguous().view(torch.int16), yo.view(torch.int16))


def test_nested_bad_arguments(gpu_lib):
    import torch
    lib = gpu_lib.load()
    x = torch.zeros((64, 2 * 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((2, 3, 64, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((64, 2 * 64), dtype=torch.bfloat16, device="cuda")
    d = offsets_dev(np.array([0, 10, 20, 30], dtype=np.int32))
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ok = lib.rg_mgemm_nested(x.data_ptr(), w.data_ptr(), d.data_ptr(), 2, 3, 64, 64, 64, 0, y.data_ptr(), s)
    assert ok == gpu_lib.RG_OK
    for O in (0, -1, gpu_lib.RG_MAX_OUTER + 1):
        assert lib.rg_mgemm_nested(x.data_ptr(), w.data_ptr(), d.data_ptr(), O, 3, 64, 64, 64, 0,
                                   y.data_ptr(), s) == gpu_lib.RG_ERR_INVALID_ARG
    assert lib.rg_mgemm_nested(x.data_ptr() + 2, w.data_ptr(), d.data_ptr(), 2, 3, 64, 64, 64, 0,
                               y.data_ptr(), s) == gpu_lib.RG_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        gpu_lib.mgemm_nested(x[:, :100].contiguous(), w, d)  # x columns != O*K
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0


def test_nested_bad_offsets_flagged(gpu_lib):
    import torch
    x = torch.ones((32, 2 * 64), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((2, 2, 64, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.full((32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    gpu_lib.mgemm_nested(x, w, offsets_dev(np.array([0, 20, 10], dtype=np.int32)), out=y)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == gpu_lib.RG_DEV_BAD_OFFSETS
    assert bool((y == 7.0).all()), "a call with invalid offsets wrote its output"


@pytest.mark.parametrize("N,K,transpose_B", [(48, 320, False), (64, 128, False), (16, 2048, False),
                                             (384, 40, False), (384, 64, True), (200, 16, True), (72, 8, False),
                                             (384, 32, False), (256, 16, True), (320, 24, True), (136, 16, False)],
                         ids=["narrow48", "narrow64", "narrow16_longK", "shallow40", "shallow64_dgrad",
                              "shallow16_dgrad", "shallow8", "shallow32", "shallow16_dgrad_4d",
                              "shallow24_dgrad_4d", "shallow16_136"])
def test_mgemm_small_tile_variants_bit_exact(gpu_lib, N, K, transpose_B):
    """Outputs at most 64 wide (64-column pair tiles) and contractions of one
    64-deep stage (single-CTA 128 x 256 tiles, eight epilogue warps; operand
    boxes 16 K wide with the 32-byte swizzle for K <= 16, 32 wide with the
    64-byte swizzle for K <= 32, both for plain and transposed B) run their
    own tile variants; integer inputs make the expected bf16 outputs exact."""
    counts = [300, 0, 1, 129, 77]
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + 5
    x = W.integer_bf16((M, K), -2, 2, 23, 0)
    w = W.integer_bf16((5, K, N) if transpose_B else (5, N, K), -2, 2, 23, 1)
    y = run_nested(gpu_lib, x, w[None], off, transpose_B, M, 1, N)
    ref = oracle.mgemm(x, w, off, transpose_B=transpose_B)
    valid = int(off[-1])
    np.testing.assert_array_equal(y[:valid], bf16_round_exact(ref[:valid]))
    assert (y[valid:] == SENTINEL_BF16).all()
