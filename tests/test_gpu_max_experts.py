"""GPU parity at the largest group count the ABI accepts (RG_MAX_EXPERTS =
1024 experts or inner groups): the per-expert tables beside each kernel's
pipeline are at their largest, the device tile-list scans span 32 lanes x 32
groups, and most groups hold 0..3 rows.  Integer inputs make the bf16
results bit-exact against the oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import bf16_round_exact, offsets_dev, to_dev, to_host_bits
from test_gpu_mx import int_codes, run_mx, run_mxk, u8_dev
from test_gpu_swiglu import check_bwd_case, check_case

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = 0x4640  # 12288.0
E_MAX = 1024


def max_counts(seed, big=(300, 129, 64)):
    """1024 groups of 0..3 rows, with a few longer ones and empty ones at
    both ends and in the middle."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 4, size=E_MAX)
    c[[5, 511, 1000]] = big
    c[[0, 512, E_MAX - 1]] = 0
    return c


def ints(shape, seed, stream):
    return W.integer_bf16(shape, -2, 2, seed, stream)


def test_abi_limit_is_1024(gpu_lib):
    assert gpu_lib.RG_MAX_EXPERTS == E_MAX


@pytest.mark.parametrize("transpose_B,N,K", [(False, 256, 128), (True, 256, 128),   # default tile
                                             (False, 64, 128),                      # 64-column tiles
                                             (False, 256, 64), (True, 320, 64),     # single-CTA one-stage
                                             (False, 256, 32), (True, 320, 16)],    # ... narrow operand boxes
                         ids=["fwd", "dgrad", "fwd-narrow", "fwd-one-stage", "dgrad-one-stage",
                              "fwd-one-stage-k32", "dgrad-one-stage-k16"])
def test_mgemm_max_experts_bit_exact(gpu_lib, transpose_B, N, K):
    import torch
    counts = max_counts(1)
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + 5
    x = ints((M, K), 11, 0)
    w = ints((E_MAX, K, N) if transpose_B else (E_MAX, N, K), 11, 1)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y.view(torch.int16).fill_(SENTINEL_BF16)
    gpu_lib.mgemm(to_dev(x), to_dev(w), offsets_dev(off), transpose_B=transpose_B, out=y)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    got = to_host_bits(y)
    valid = int(off[-1])
    ref = oracle.mgemm(x, w, off, transpose_B=transpose_B)
    np.testing.assert_array_equal(got[:valid], bf16_round_exact(ref[:valid]))
    assert (got[valid:] == SENTINEL_BF16).all()


def test_nested_max_inner_groups_bit_exact(gpu_lib):
    """Two outer groups over 1024 inner row groups (the LoRA expand form)."""
    import torch
    counts = max_counts(2)
    off = W.offsets_from_counts(counts)
    O, N, K = 2, 256, 16
    M = int(off[-1]) + 3
    x = ints((M, O * K), 12, 0)
    w = ints((O, E_MAX, N, K), 12, 1)
    y = torch.empty((M, O * N), dtype=torch.bfloat16, device="cuda")
    y.view(torch.int16).fill_(SENTINEL_BF16)
    gpu_lib.mgemm_nested(to_dev(x), to_dev(w), offsets_dev(off), out=y)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    got = to_host_bits(y)
    valid = int(off[-1])
    ref = oracle.mgemm_nested(x, w, off)
    np.testing.assert_array_equal(got[:valid], bf16_round_exact(ref[:valid]))
    assert (got[valid:] == SENTINEL_BF16).all()


def test_swiglu_max_experts(gpu_lib):
    check_case(gpu_lib, max_counts(3).tolist(), 4, 128, 64, 13)
    check_bwd_case(gpu_lib, max_counts(4).tolist(), 4, 128, 64, 14)


@pytest.mark.parametrize("transpose_B", [False, True], ids=["fwd", "dgrad"])
def test_mx_mgemm_max_experts_bit_exact(gpu_lib, transpose_B):
    counts = max_counts(5)
    off = W.offsets_from_counts(counts)
    N, K = 64, 64
    M = int(off[-1]) + 6
    xq = int_codes((M, K), 15, 0)
    wq = int_codes((E_MAX, K, N) if transpose_B else (E_MAX, N, K), 15, 1)
    sx = W.e8m0_codes((M, K // 32), 126, 128, 15, 2)
    sw = W.e8m0_codes((E_MAX, N, K // 32), 126, 128, 15, 3)
    y = run_mx(gpu_lib, xq, sx, wq, sw, off, transpose_B)
    valid = int(off[-1])
    ref = oracle.mgemm_mx(xq, sx, wq, sw, off, transpose_B=transpose_B)
    assert (y[:valid] == bf16_round_exact(ref[:valid])).all()
    assert (y[valid:] == SENTINEL_BF16).all()


def test_mx_kgemm_max_experts_bit_exact(gpu_lib):
    counts = 32 * max_counts(6, big=(10, 5, 3))
    off = W.offsets_from_counts(counts)
    N, K = 64, 96
    M = int(off[-1]) + 32
    gq, xq = int_codes((M, N), 16, 0), int_codes((M, K), 16, 1)
    sg = W.e8m0_codes((N, M // 32), 126, 128, 16, 2)
    sx = W.e8m0_codes((K, M // 32), 126, 128, 16, 3)
    dW = run_mxk(gpu_lib, gq, sg, xq, sx, off)
    np.testing.assert_array_equal(dW.astype(np.float64), oracle.kgemm_mx(gq, sg, xq, sx, off))
    assert (dW[np.flatnonzero(counts == 0)] == 0).all()


def test_scale_conversions_max_groups(gpu_lib):
    """Both blocked-layout conversions with 1024 groups, byte for byte; no
    byte past the last block is written."""
    import torch
    counts = max_counts(7)
    off = W.offsets_from_counts(counts)
    R, KS = int(off[-1]) + 9, 12
    s = W.e8m0_codes((R, KS), 0, 254, 17, 0)
    nblk = int(sum((int(c) + 127) // 128 for c in counts)) * ((KS + 3) // 4) * 512
    out = torch.full((gpu_lib.mx_blocked_bytes(R, KS, E_MAX),), 0xEE, dtype=torch.uint8, device="cuda")
    gpu_lib.mx_scales_blocked(u8_dev(s), offsets_dev(off), out=out)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got[:nblk], oracle.mx_blocked(s, off)[:nblk])
    assert (got[nblk:] == 0xEE).all()

    ck = 32 * max_counts(8, big=(10, 5, 3))
    offk = W.offsets_from_counts(ck)
    Rk, KSk = 200, int(offk[-1]) // 32 + 3
    sk = W.e8m0_codes((Rk, KSk), 0, 254, 17, 1)
    nq = int(sum((int(c) + 127) // 128 for c in ck))
    used = ((Rk + 127) // 128) * nq * 512
    outk = torch.full((gpu_lib.mx_blocked_k_bytes(Rk, KSk, E_MAX),), 0xEE, dtype=torch.uint8, device="cuda")
    gpu_lib.mx_scales_blocked_k(u8_dev(sk), offsets_dev(offk), out=outk)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    gotk = outk.cpu().numpy()
    np.testing.assert_array_equal(gotk[:used], oracle.mx_blocked_k(sk, offk)[:used])
    assert (gotk[used:] == 0xEE).all()
