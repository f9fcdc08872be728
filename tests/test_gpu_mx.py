"""GPU parity of the MXFP8 grouped GEMM and of the blocked scale layout
(torchao MoE-training PR: MXFP8 grouped GEMMs with E8M0 scales converted to
a blocked format; DeepGEMM issue: block-scaled FP8 GEMMs) against the CPU
oracle, through the C ABI."""
import ctypes
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from parity import bf16_round_exact, check_bf16, offsets_dev, to_host_bits

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = 0x4640  # 12288.0


def u8_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def blocked_dev(rg, scales, off):
    """Blocked layout made on the GPU by rg_mx_scales_blocked."""
    import torch
    out = rg.mx_scales_blocked(u8_dev(scales), offsets_dev(off))
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return out


def run_mx(rg, xq, sx, wq, sw, off, transpose_B, sentinel=True):
    import torch
    E = len(off) - 1
    M, K = xq.shape
    N = wq.shape[2] if transpose_B else wq.shape[1]
    sxb = blocked_dev(rg, sx, off)
    swb = blocked_dev(rg, sw.reshape(E * N, K // 32), np.arange(0, (E + 1) * N, N, dtype=np.int32))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    if sentinel:
        y.view(torch.int16).fill_(SENTINEL_BF16)
    rg.mgemm_mxfp8(u8_dev(xq), sxb, u8_dev(wq), swb, offsets_dev(off), transpose_B=transpose_B, out=y)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return to_host_bits(y)


def mismatch_report(got, want, off):
    bad = np.argwhere(got != want)
    if bad.size == 0:
        return ""
    rows = np.unique(bad[:, 0])
    starts = np.array([off[np.searchsorted(off, r, side="right") - 1] for r in rows])
    local = rows - starts
    return (f"{len(bad)} mismatches in {len(rows)} rows; row-in-expert %128 //32 -> "
            f"{sorted(set(((local % 128) // 32).tolist()))}, %32 sample {sorted(set((local % 32).tolist()))[:8]}; "
            f"cols sample {sorted(set(bad[:, 1].tolist()))[:8]}")


# --------------------------------------------------------------- blocked layout


@pytest.mark.parametrize("counts,KS", [([130, 0, 1, 255, 128, 7], 7), ([512], 96), ([0, 0], 3), ([37] * 9, 80)],
                         ids=["ragged_ks7", "one_group_ks96", "all_empty", "nine_groups_ks80"])
def test_mx_blocked_bit_exact(gpu_lib, counts, KS):
    import torch
    off = W.offsets_from_counts(counts)
    R = int(off[-1]) + 5
    src = W.e8m0_codes((R, KS), 0, 254, 51, len(counts))
    want = oracle.mx_blocked(src, off)
    nblk = sum((c + 127) // 128 for c in counts) * ((KS + 3) // 4) * 512
    out = torch.full((gpu_lib.mx_blocked_bytes(R, KS, len(counts)),), 0xEE, dtype=torch.uint8, device="cuda")
    gpu_lib.mx_scales_blocked(u8_dev(src), offsets_dev(off), out=out)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got[:nblk], want[:nblk])
    assert (got[nblk:] == 0xEE).all(), "bytes past the last block were written"


def test_mx_blocked_bad_offsets(gpu_lib):
    import torch
    out = torch.full((gpu_lib.mx_blocked_bytes(64, 4, 2),), 0xEE, dtype=torch.uint8, device="cuda")
    gpu_lib.mx_scales_blocked(u8_dev(np.zeros((64, 4), np.uint8)), offsets_dev(np.array([0, 40, 20], np.int32)),
                              out=out)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == gpu_lib.RG_DEV_BAD_OFFSETS
    assert bool((out == 0xEE).all())


# ------------------------------------------------------------------- GEMM


def int_codes(shape, seed, stream):
    """E4M3 codes of integers in {-2..2} (decoded by the oracle's table)."""
    e4, _ = oracle.mx_decode_tables()
    table = np.array([int(np.flatnonzero(e4 == v)[0]) for v in (-2.0, -1.0, 0.0, 1.0, 2.0)], dtype=np.uint8)
    rng = np.random.default_rng(np.random.SeedSequence([seed, stream]))
    return table[rng.integers(0, 5, size=shape)]


@pytest.mark.parametrize("transpose_B", [False, True], ids=["fwd", "dgrad"])
def test_mx_integer_inputs_bit_exact(gpu_lib, transpose_B):
    """Integer elements, scales 1/2, 1, 2: every partial sum is exact in
    fp32, so the bf16 output must equal the rounded exact result bit for bit.
    Scales differ per row, per 32-element block and per output column, so a
    misplaced scale shows."""
    counts = [130, 0, 1, 200, 70]
    off = W.offsets_from_counts(counts)
    E, N, K = len(counts), 384, 320
    M = int(off[-1]) + 7
    xq = int_codes((M, K), 61, 0)
    wq = int_codes((E, K, N) if transpose_B else (E, N, K), 61, 1)
    sx = W.e8m0_codes((M, K // 32), 126, 128, 61, 2)
    sw = W.e8m0_codes((E, N, K // 32), 126, 128, 61, 3)
    y = run_mx(gpu_lib, xq, sx, wq, sw, off, transpose_B)
    ref = oracle.mgemm_mx(xq, sx, wq, sw, off, transpose_B=transpose_B)
    valid = int(off[-1])
    want = bf16_round_exact(ref[:valid])
    assert (y[:valid] == want).all(), mismatch_report(y[:valid], want, off)
    assert (y[valid:] == SENTINEL_BF16).all(), "rows past offsets[E] were written"


@pytest.mark.parametrize("transpose_B", [False, True], ids=["fwd", "dgrad"])
@pytest.mark.parametrize("E,N,K,total", [(4, 256, 128, 700), (7, 640, 544, 3000), (3, 16, 32, 200),
                                         (2, 1296, 1024, 900)],
                         ids=["one_chunk", "many_tiles", "min_16x32", "n_tail"])
def test_mx_random_codes(gpu_lib, transpose_B, E, N, K, total):
    rng = np.random.default_rng(zlib.crc32(f"mx/{E}/{N}/{K}/{transpose_B}".encode()))
    counts = rng.multinomial(total, [1 / E] * E)
    counts[0] = 0
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + 3
    s = int(rng.integers(1 << 20))
    xq = W.e4m3_codes((M, K), s, 0)
    wq = W.e4m3_codes((E, K, N) if transpose_B else (E, N, K), s, 1)
    sx = W.e8m0_codes((M, K // 32), *W.MX_ACT_SCALES, s, 2)  # values of RMS ~1 (like N(0,1))
    sw = W.e8m0_codes((E, N, K // 32), *W.mx_weight_scales(K), s, 3)  # RMS ~1/sqrt(K)
    y = run_mx(gpu_lib, xq, sx, wq, sw, off, transpose_B)
    ref = oracle.mgemm_mx(xq, sx, wq, sw, off, transpose_B=transpose_B)
    valid = int(off[-1])
    check_bf16(y[:valid], ref[:valid], f"mxfp8 E={E} N={N} K={K} tB={transpose_B}")
    assert (y[valid:] == SENTINEL_BF16).all()


def test_mx_deterministic(gpu_lib):
    rng = np.random.default_rng(71)
    off = W.offsets_from_counts(rng.multinomial(1000, [0.25] * 4))
    xq, wq = W.e4m3_codes((1000, 256), 71, 0), W.e4m3_codes((4, 512, 256), 71, 1)
    sx, sw = W.e8m0_codes((1000, 8), *W.MX_ACT_SCALES, 71, 2), W.e8m0_codes((4, 512, 8), *W.mx_weight_scales(256), 71, 3)
    a = run_mx(gpu_lib, xq, sx, wq, sw, off, False)
    b = run_mx(gpu_lib, xq, sx, wq, sw, off, False)
    np.testing.assert_array_equal(a, b)


def test_mx_bad_arguments(gpu_lib):
    import torch
    lib = gpu_lib.load()
    xq = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    wq = torch.zeros((2, 64, 64), dtype=torch.uint8, device="cuda")
    sb = torch.zeros((gpu_lib.mx_blocked_bytes(128, 2, 2),), dtype=torch.uint8, device="cuda")
    y = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    d = offsets_dev(np.array([0, 30, 60], dtype=np.int32))
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(M=64, N=64, K=64, E=2, x=xq.data_ptr()):
        return lib.rg_mgemm_mxfp8(x, sb.data_ptr(), wq.data_ptr(), sb.data_ptr(), d.data_ptr(), E, M, N, K, 0,
                                  y.data_ptr(), s)

    assert call() == gpu_lib.RG_OK
    assert call(K=48) == gpu_lib.RG_ERR_INVALID_ARG   # K not a multiple of 32
    assert call(N=40) == gpu_lib.RG_ERR_INVALID_ARG   # N not a multiple of 16
    assert call(E=0) == gpu_lib.RG_ERR_INVALID_ARG
    assert call(x=xq.data_ptr() + 8) == gpu_lib.RG_ERR_INVALID_ARG  # misaligned
    assert lib.rg_mx_blocked_bytes(100, 0, 1) == -1
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0


# ------------------------------------------------ K-grouped MXFP8 (weight gradient)


@pytest.mark.parametrize("off,R,KS", [([0, 96, 96, 320], 130, 10), ([0, 4096], 256, 128), ([0, 0, 0], 8, 3),
                                      ([0, 32, 64, 1024, 1056], 300, 33)],
                         ids=["ragged", "one_group", "all_empty", "mixed"])
def test_mx_blocked_k_bit_exact(gpu_lib, off, R, KS):
    import torch
    off = np.array(off, dtype=np.int32)
    G = len(off) - 1
    src = W.e8m0_codes((R, KS), 0, 254, 52, G)
    want = oracle.mx_blocked_k(src, off)
    nq = sum((int(off[g + 1]) - int(off[g]) + 127) // 128 for g in range(G))
    used = ((R + 127) // 128) * nq * 512
    out = torch.full((gpu_lib.mx_blocked_k_bytes(R, KS, G),), 0xEE, dtype=torch.uint8, device="cuda")
    gpu_lib.mx_scales_blocked_k(u8_dev(src), offsets_dev(off), out=out)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got[:used], want[:used])
    assert (got[used:] == 0xEE).all()


def test_mx_blocked_k_unaligned_offsets_flagged(gpu_lib):
    import torch
    out = torch.full((gpu_lib.mx_blocked_k_bytes(64, 4, 2),), 0xEE, dtype=torch.uint8, device="cuda")
    gpu_lib.mx_scales_blocked_k(u8_dev(np.zeros((64, 4), np.uint8)), offsets_dev(np.array([0, 40, 96], np.int32)),
                                out=out)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == gpu_lib.RG_DEV_BAD_OFFSETS
    assert bool((out == 0xEE).all())


def run_mxk(rg, gq, sg, xq, sx, off, init=None):
    import torch
    E = len(off) - 1
    M, N = gq.shape
    K = xq.shape[1]
    doff = offsets_dev(off)
    sgb = rg.mx_scales_blocked_k(u8_dev(sg), doff)
    sxb = rg.mx_scales_blocked_k(u8_dev(sx), doff)
    if init is None:
        dW = torch.full((E, N, K), float("nan"), dtype=torch.float32, device="cuda")
        rg.kgemm_mxfp8(u8_dev(gq), sgb, u8_dev(xq), sxb, doff, out=dW)
    else:
        dW = torch.from_numpy(init.copy()).cuda()
        rg.kgemm_mxfp8(u8_dev(gq), sgb, u8_dev(xq), sxb, doff, out=dW, accumulate=True)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return dW.cpu().numpy()


def test_mx_kgemm_integer_inputs_bit_exact(gpu_lib):
    """Integer codes and scales 1/2..2 make every fp32 partial sum exact, so
    dW must equal the exact result; the 4160-row expert spans two
    accumulation chunks, N and K end inside a tile."""
    counts = [128, 0, 32, 4160, 96]
    off = W.offsets_from_counts(counts)
    M, N, K = int(off[-1]) + 64, 272, 320
    gq, xq = int_codes((M, N), 62, 0), int_codes((M, K), 62, 1)
    sg = W.e8m0_codes((N, M // 32), 126, 128, 62, 2)
    sx = W.e8m0_codes((K, M // 32), 126, 128, 62, 3)
    dW = run_mxk(gpu_lib, gq, sg, xq, sx, off)
    ref = oracle.kgemm_mx(gq, sg, xq, sx, off)
    np.testing.assert_array_equal(dW.astype(np.float64), ref)
    assert (dW[1] == 0).all()


def mxk_random(seed, counts, N, K, extra=32):
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + extra
    gq, xq = W.e4m3_codes((M, N), seed, 0), W.e4m3_codes((M, K), seed, 1)
    sg = W.e8m0_codes((N, M // 32), *W.MX_ACT_SCALES, seed, 2)
    sx = W.e8m0_codes((K, M // 32), *W.MX_ACT_SCALES, seed, 3)
    return off, gq, sg, xq, sx


@pytest.mark.parametrize("counts,N,K", [([320, 0, 96, 1024, 32], 384, 512), ([64] * 6, 256, 256),
                                        ([2048, 0], 128, 1024), ([32], 16, 16)],
                         ids=["mixed", "six_equal", "one_long", "min_16"])
def test_mx_kgemm_random_codes(gpu_lib, counts, N, K):
    from parity import check_fp32
    off, gq, sg, xq, sx = mxk_random(zlib.crc32(f"mxk/{counts}/{N}/{K}".encode()), counts, N, K)
    dW = run_mxk(gpu_lib, gq, sg, xq, sx, off)
    ref = oracle.kgemm_mx(gq, sg, xq, sx, off)
    check_fp32(dW, ref, f"mxfp8 wgrad counts={counts} N={N} K={K}")
    for e in np.flatnonzero(np.array(counts) == 0):
        assert (dW[e] == 0).all()


def test_mx_kgemm_accumulate(gpu_lib):
    from parity import check_fp32
    off, gq, sg, xq, sx = mxk_random(81, [320, 0, 96, 4224], 256, 384)
    E = len(off) - 1
    init = W.bf16_bits_to_f32(W.normal_bf16((E, 256, 384), 1.0, 81, 9))  # the gradient to add to
    dW = run_mxk(gpu_lib, gq, sg, xq, sx, off, init=init)
    ref = oracle.kgemm_mx(gq, sg, xq, sx, off) + init.astype(np.float64)
    check_fp32(dW, ref, "mxfp8 wgrad accumulate")
    assert (dW[1] == init[1]).all(), "an expert without rows changed dW when accumulating"


def test_mx_kgemm_no_rows_zeroes(gpu_lib):
    import torch
    dW = torch.full((3, 64, 64), 5.0, dtype=torch.float32, device="cuda")
    z = torch.zeros((32, 64), dtype=torch.uint8, device="cuda")
    d = offsets_dev(np.zeros(4, np.int32))
    sb = gpu_lib.mx_scales_blocked_k(torch.zeros((64, 1), dtype=torch.uint8, device="cuda"), d)
    gpu_lib.kgemm_mxfp8(z, sb, z, sb, d, out=dW)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    assert bool((dW == 0).all())


# ------------------------------------------------------------------ edge cases


def test_mx_many_small_experts(gpu_lib):
    """300 experts of 0..7 and a few long ones: the device tile lists and the
    scale-block prefix sums span many groups; empty experts write nothing."""
    rng = np.random.default_rng(91)
    counts = rng.integers(0, 8, size=300)
    counts[[5, 150, 299]] = [300, 260, 129]
    counts[[0, 1, 200]] = 0
    off = W.offsets_from_counts(counts)
    E, N, K = 300, 64, 64
    M = int(off[-1]) + 4
    xq, wq = W.e4m3_codes((M, K), 91, 0), W.e4m3_codes((E, N, K), 91, 1)
    sx = W.e8m0_codes((M, K // 32), *W.MX_ACT_SCALES, 91, 2)
    sw = W.e8m0_codes((E, N, K // 32), *W.mx_weight_scales(K), 91, 3)
    y = run_mx(gpu_lib, xq, sx, wq, sw, off, False)
    ref = oracle.mgemm_mx(xq, sx, wq, sw, off)
    valid = int(off[-1])
    check_bf16(y[:valid], ref[:valid], "mxfp8 300 experts")
    assert (y[valid:] == SENTINEL_BF16).all()


def test_mx_kgemm_many_experts(gpu_lib):
    from parity import check_fp32
    rng = np.random.default_rng(92)
    counts = 32 * rng.integers(0, 3, size=300)
    counts[[7, 100]] = [4128, 320]
    off, gq, sg, xq, sx = mxk_random(92, counts, 32, 48)
    dW = run_mxk(gpu_lib, gq, sg, xq, sx, off)
    ref = oracle.kgemm_mx(gq, sg, xq, sx, off)
    check_fp32(dW, ref, "mxfp8 wgrad 300 experts")
    assert (dW[np.flatnonzero(counts == 0)] == 0).all()


def test_mx_no_rows(gpu_lib):
    """M = 0: the Mgemm writes nothing, the Kgemm zeroes dW."""
    import torch
    E, N, K = 3, 32, 64
    off = offsets_dev(np.zeros(E + 1, np.int32))
    wq = torch.zeros((E, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.zeros((gpu_lib.mx_blocked_bytes(E * N, K // 32, E),), dtype=torch.uint8, device="cuda")
    xq = torch.zeros((0, K), dtype=torch.uint8, device="cuda")
    sa = torch.zeros((gpu_lib.mx_blocked_bytes(0, K // 32, E),), dtype=torch.uint8, device="cuda")
    y = gpu_lib.mgemm_mxfp8(xq, sa, wq, sb, off)
    assert tuple(y.shape) == (0, N)
    dW = torch.full((E, N, K), 3.0, dtype=torch.float32, device="cuda")
    g0 = torch.zeros((0, N), dtype=torch.uint8, device="cuda")
    gpu_lib.kgemm_mxfp8(g0, sb, xq, sb, off, out=dW)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    assert bool((dW == 0).all())
