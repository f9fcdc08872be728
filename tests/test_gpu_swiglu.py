"""GPU parity of the gate-up forward GEMM with the SwiGLU activation fused
into its epilogue: h against the oracle's SwiGLU of the oracle's exact
gate-up product, and the optional y13 output against the plain grouped GEMM."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import bf16_round_exact, check_bf16, offsets_dev, to_dev, to_host_bits

pytestmark = pytest.mark.gpu

SENTINEL_BF16 = 0x4640  # 12288.0


def run_swiglu(rg, x, w13, off, want_y13=True):
    import torch
    M, F = x.shape[0], w13.shape[1] // 2
    h = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    h.view(torch.int16).fill_(SENTINEL_BF16)
    y13 = None
    if want_y13:
        y13 = torch.empty((M, 2 * F), dtype=torch.bfloat16, device="cuda")
        y13.view(torch.int16).fill_(SENTINEL_BF16)
    rg.mgemm_swiglu(to_dev(x), to_dev(w13), offsets_dev(off), out=h,
                    y13=y13 if want_y13 else False)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return to_host_bits(h), (to_host_bits(y13) if want_y13 else None)


def plain_mgemm(rg, x, w, off):
    import torch
    y = rg.mgemm(to_dev(x), to_dev(w), offsets_dev(off))
    torch.cuda.synchronize()
    return to_host_bits(y)


def check_case(rg, counts, tail, F, K, seed, scale=1.0):
    off = W.offsets_from_counts(counts)
    E = len(counts)
    M = int(off[-1]) + tail
    x = W.normal_bf16((M, K), scale, seed, 0)
    w13 = W.normal_bf16((E, 2 * F, K), 1.0 / np.sqrt(K), seed, 1)
    h, y13 = run_swiglu(rg, x, w13, off)
    valid = int(off[-1])
    if valid:
        y_ref = oracle.mgemm(x, w13, off)
        check_bf16(h[:valid], oracle.swiglu(y_ref[:valid]), "swiglu/h")
        check_bf16(y13[:valid], y_ref[:valid], "swiglu/y13")
        # y13 is the plain forward GEMM's output: same tiles, same MMA order
        y_plain = plain_mgemm(rg, x, w13, off)
        np.testing.assert_array_equal(y13[:valid], y_plain[:valid])
    assert (h[valid:] == SENTINEL_BF16).all(), "rows past offsets[E] were written (h)"
    assert (y13[valid:] == SENTINEL_BF16).all(), "rows past offsets[E] were written (y13)"


def test_swiglu_integer_gate_up_bit_exact(gpu_lib):
    """Integer inputs make every accumulator exact: y13 is the correctly
    rounded product, and h matches SwiGLU of it to bf16 rounding."""
    off = W.offsets_from_counts([130, 0, 1, 200])
    M, F, K = int(off[-1]) + 7, 192, 320
    x = W.integer_bf16((M, K), -2, 2, 3, 0)
    w13 = W.integer_bf16((4, 2 * F, K), -1, 1, 3, 1)
    h, y13 = run_swiglu(gpu_lib, x, w13, off)
    valid = int(off[-1])
    ref = oracle.mgemm(x, w13, off)
    np.testing.assert_array_equal(y13[:valid], bf16_round_exact(ref[:valid]))
    check_bf16(h[:valid], oracle.swiglu(ref[:valid]), "swiglu-int/h")


CASES = {
    "ragged_rows": dict(counts=[300, 0, 1, 129, 77], tail=5, F=256, K=192),
    "F_not_tile_multiple": dict(counts=[200, 90], tail=0, F=200, K=136),
    "F_smallest": dict(counts=[5, 0, 9], tail=2, F=8, K=8),
    "F_136": dict(counts=[40, 300], tail=1, F=136, K=64),
    "all_empty": dict(counts=[0, 0, 0], tail=64, F=128, K=64),
    "many_experts": dict(counts=list(np.random.default_rng(6).integers(0, 40, size=300)), tail=11,
                         F=128, K=64),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_swiglu_cases(gpu_lib, case):
    c = CASES[case]
    check_case(gpu_lib, c["counts"], c["tail"], c["F"], c["K"], 70 + sorted(CASES).index(case))


def test_swiglu_medium_a3b_shape(gpu_lib):
    """Gate-up of one MoE layer at hidden 2048 / expert FFN 768 on 8 experts
    with Dirichlet-routed rows (several tiles in every dimension)."""
    counts = W.counts_dirichlet(8, 2500, 2.0, 31)
    check_case(gpu_lib, counts, 3, 768, 2048, 31)


def test_swiglu_large_activations(gpu_lib):
    """Gate values of magnitude ~10-30 exercise both saturated ends of SiLU."""
    check_case(gpu_lib, [257, 300], 0, 256, 256, 41, scale=16.0)


def test_swiglu_without_y13_matches(gpu_lib):
    off = W.offsets_from_counts([190, 3, 260])
    M, F, K = int(off[-1]), 384, 256
    x = W.normal_bf16((M, K), 1.0, 51, 0)
    w13 = W.normal_bf16((3, 2 * F, K), 1.0 / np.sqrt(K), 51, 1)
    h_only, _ = run_swiglu(gpu_lib, x, w13, off, want_y13=False)
    h_both, _ = run_swiglu(gpu_lib, x, w13, off, want_y13=True)
    np.testing.assert_array_equal(h_only, h_both)
    check_bf16(h_only, oracle.swiglu(oracle.mgemm(x, w13, off)), "swiglu/h_only")


def test_swiglu_zero_rows(gpu_lib):
    import torch
    off = offsets_dev(np.zeros(4, dtype=np.int32))
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    w13 = torch.zeros((3, 256, 64), dtype=torch.bfloat16, device="cuda")
    h, y13 = gpu_lib.mgemm_swiglu(x, w13, off, y13=True)
    torch.cuda.synchronize()
    assert h.shape == (0, 128) and y13.shape == (0, 256)
    assert gpu_lib.device_status() == 0


# ------------------------------------------------------------ backward


def run_swiglu_dgrad(rg, dy, w2, off, y13):
    import torch
    M, F = dy.shape[0], w2.shape[2]
    dy13 = torch.empty((M, 2 * F), dtype=torch.bfloat16, device="cuda")
    dy13.view(torch.int16).fill_(SENTINEL_BF16)
    rg.mgemm_swiglu_dgrad(to_dev(dy), to_dev(w2), offsets_dev(off), to_dev(y13), out=dy13)
    torch.cuda.synchronize()
    assert rg.device_status() == 0
    return to_host_bits(dy13)


def check_bwd_case(rg, counts, tail, F, K, seed, gate_scale=2.0):
    off = W.offsets_from_counts(counts)
    E = len(counts)
    M = int(off[-1]) + tail
    dy = W.normal_bf16((M, K), 1.0, seed, 0)
    w2 = W.normal_bf16((E, K, F), 1.0 / np.sqrt(K), seed, 1)
    y13 = W.normal_bf16((M, 2 * F), gate_scale, seed, 2)
    dy13 = run_swiglu_dgrad(rg, dy, w2, off, y13)
    valid = int(off[-1])
    if valid:
        dh = oracle.mgemm(dy, w2, off, transpose_B=True)
        ref = oracle.swiglu_bwd(dh[:valid], W.bf16_bits_to_f32(y13[:valid]))
        check_bf16(dy13[:valid], ref, "swiglu_dgrad")
    assert (dy13[valid:] == SENTINEL_BF16).all(), "rows past offsets[E] were written"


BWD_CASES = {
    "ragged_rows": dict(counts=[300, 0, 1, 129, 77], tail=5, F=256, K=192),
    "F_not_tile_multiple": dict(counts=[200, 90], tail=0, F=200, K=136),
    "F_smallest": dict(counts=[5, 0, 9], tail=2, F=8, K=8),
    "F_320": dict(counts=[40, 300], tail=1, F=320, K=64),
    "all_empty": dict(counts=[0, 0, 0], tail=64, F=128, K=64),
    "many_experts": dict(counts=list(np.random.default_rng(7).integers(0, 40, size=300)), tail=11,
                         F=128, K=64),
}


@pytest.mark.parametrize("case", sorted(BWD_CASES))
def test_swiglu_dgrad_cases(gpu_lib, case):
    c = BWD_CASES[case]
    check_bwd_case(gpu_lib, c["counts"], c["tail"], c["F"], c["K"], 90 + sorted(BWD_CASES).index(case))


def test_swiglu_dgrad_medium_a3b_shape(gpu_lib):
    """Down-projection input gradient of one layer (hidden 2048 -> F 768) on
    8 experts with Dirichlet-routed rows, then the SwiGLU backward."""
    counts = W.counts_dirichlet(8, 2500, 2.0, 33)
    check_bwd_case(gpu_lib, counts, 3, 768, 2048, 33)


def test_swiglu_dgrad_saturated_gates(gpu_lib):
    check_bwd_case(gpu_lib, [257, 300], 0, 256, 256, 43, gate_scale=20.0)


def test_swiglu_forward_backward_chain(gpu_lib):
    """y13 saved by rg_mgemm_swiglu feeds rg_mgemm_swiglu_dgrad: the result
    matches the oracle's chain on the same bf16 y13."""
    off = W.offsets_from_counts([190, 3, 260, 0])
    M, D, F = int(off[-1]) + 4, 256, 384
    x = W.normal_bf16((M, D), 1.0, 61, 0)
    w13 = W.normal_bf16((4, 2 * F, D), 1.0 / np.sqrt(D), 61, 1)
    w2 = W.normal_bf16((4, D, F), 1.0 / np.sqrt(F), 61, 2)
    dy = W.normal_bf16((M, D), 1.0, 61, 3)
    _, y13 = run_swiglu(gpu_lib, x, w13, off)
    valid = int(off[-1])
    y13[valid:] = 0
    dy13 = run_swiglu_dgrad(gpu_lib, dy, w2, off, y13)
    ref = oracle.swiglu_bwd(oracle.mgemm(dy, w2, off, transpose_B=True)[:valid],
                            W.bf16_bits_to_f32(y13[:valid]))
    check_bf16(dy13[:valid], ref, "swiglu_chain")
