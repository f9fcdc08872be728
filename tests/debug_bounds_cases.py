"""Run the edge-case and tiny cases of every kernel through the debug-bounds
build of the library (every copy and store coordinate checked against its
operand, RG_DEV_BOUNDS on a violation) and check status and results.

    python tests/debug_bounds_cases.py PATH/TO/librg.so

Prints one line per case and exits non-zero if a case sets any status bit or
its output differs from the oracle.  Run in a process of its own: the binding
loads one library per process.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402
from parity import bf16_round_exact, check_bf16, check_fp32, offsets_dev, to_dev, to_host_bits  # noqa: E402


def ints(shape, seed, stream):
    return W.integer_bf16(shape, -2, 2, seed, stream)


def main(lib_path):
    import torch
    from moe_grouped_gemm_device_gb300 import _build
    _build.LIB = lib_path
    import moe_grouped_gemm_device_gb300 as rg
    rg.load()
    results = []

    def status(name):
        torch.cuda.synchronize()
        st = rg.device_status()
        results.append((name, st))
        print(f"{name}: status {st:#x}", flush=True)
        assert st == 0, f"{name}: device status {st:#x}"

    # M-grouped: ragged, empty, single-row and half-tile groups, rows past offsets[E]
    counts = [130, 0, 1, 200, 64, 300]
    off = W.offsets_from_counts(counts)
    doff = offsets_dev(off)
    valid = int(off[-1])
    for tB, N, K in [(False, 384, 320), (True, 320, 384), (True, 200, 136), (False, 64, 320), (False, 256, 64),
                     (True, 256, 64)]:
        M = valid + 7
        x = ints((M, K), 3, 0)
        w = ints((len(counts), K, N) if tB else (len(counts), N, K), 3, 1)
        y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        rg.mgemm(to_dev(x), to_dev(w), doff, transpose_B=tB, out=y)
        status(f"mgemm tB={tB} N={N} K={K}")
        got = to_host_bits(y)
        np.testing.assert_array_equal(got[:valid], bf16_round_exact(oracle.mgemm(x, w, off, transpose_B=tB)[:valid]))
        assert bool((y[valid:] == 7.0).all())
    # nested: three outer groups
    O, N, K = 3, 128, 64
    x = ints((valid + 5, O * K), 4, 0)
    w = ints((O, len(counts), N, K), 4, 1)
    y = rg.mgemm_nested(to_dev(x), to_dev(w), doff)
    status("mgemm_nested O=3")
    np.testing.assert_array_equal(to_host_bits(y)[:valid], bf16_round_exact(oracle.mgemm_nested(x, w, off)[:valid]))
    # fused SwiGLU forward and backward
    F, K = 192, 256
    x = W.normal_bf16((valid, K), 1.0, 5, 0)
    w13 = W.normal_bf16((len(counts), 2 * F, K), 1.0 / 16, 5, 1)
    h, y13 = rg.mgemm_swiglu(to_dev(x), to_dev(w13), doff, y13=True)
    status("mgemm_swiglu")
    yref = oracle.mgemm(x, w13, off)
    check_bf16(to_host_bits(h), oracle.swiglu(yref), "swiglu h")
    dy = W.normal_bf16((valid, K), 1.0, 5, 2)
    w2 = W.normal_bf16((len(counts), K, F), 1.0 / 14, 5, 3)
    dy13 = rg.mgemm_swiglu_dgrad(to_dev(dy), to_dev(w2), doff, y13)
    status("mgemm_swiglu_dgrad")
    dh = oracle.mgemm(dy, w2, off, transpose_B=True)
    check_bf16(to_host_bits(dy13), oracle.swiglu_bwd(dh, W.bf16_bits_to_f32(to_host_bits(y13))), "swiglu dgrad")
    # K-grouped: a long expert (several chunks), ragged blocks, 4-D and 3-D views, accumulation
    kcounts = [130, 0, 1, 200, 4100, 37]
    koff = W.offsets_from_counts(kcounts)
    kdoff = offsets_dev(koff)
    for N, K in [(256, 320), (200, 136)]:
        M = int(koff[-1]) + 5
        g, xx = ints((M, N), 6, 0), ints((M, K), 6, 1)
        dW = rg.kgemm(to_dev(g), to_dev(xx), kdoff)
        status(f"kgemm N={N} K={K}")
        np.testing.assert_array_equal(dW.cpu().numpy().astype(np.float64), oracle.kgemm(g, xx, koff))
        init = torch.ones_like(dW)
        rg.kgemm(to_dev(g), to_dev(xx), kdoff, out=init, accumulate=True)
        status(f"kgemm_acc N={N} K={K}")
        np.testing.assert_array_equal(init.cpu().numpy().astype(np.float64), oracle.kgemm(g, xx, koff) + 1.0)
        ws = torch.empty(rg.kgemm_workspace_bytes(len(kcounts), N, K), dtype=torch.uint8, device="cuda")
        dW2 = rg.kgemm(to_dev(g), to_dev(xx), kdoff, workspace=ws)
        status(f"kgemm_ws N={N} K={K}")
        assert torch.equal(dW2.view(torch.int32), dW.view(torch.int32))
    # K-grouped, chunk-major schedule (more dW tiles per expert than CTA pairs)
    for N, K in [(2560, 2304), (2248, 2120)]:
        M = int(koff[-1]) + 5
        g, xx = ints((M, N), 9, 0), ints((M, K), 9, 1)
        dW = rg.kgemm(to_dev(g), to_dev(xx), kdoff)
        status(f"kgemm N={N} K={K}")
        ws = torch.empty(rg.kgemm_workspace_bytes(len(kcounts), N, K), dtype=torch.uint8, device="cuda")
        dW2 = rg.kgemm(to_dev(g), to_dev(xx), kdoff, workspace=ws)
        status(f"kgemm_ws N={N} K={K}")
        assert torch.equal(dW2.view(torch.int32), dW.view(torch.int32))
        es = np.array([0, 0, 3, 4, 4, 4, 5], np.int32)
        ns = np.array([0, N - 1, 7, 0, 1000, N - 1, 33], np.int32)
        got = dW2[torch.from_numpy(es).long().cuda(), torch.from_numpy(ns).long().cuda()].cpu().numpy()
        np.testing.assert_array_equal(got.astype(np.float64), oracle.kgemm(g, xx, koff, sel=(es, ns)))
    # MXFP8: forward, input gradient and weight gradient
    mcounts = [128, 0, 32, 96, 160]
    moff = W.offsets_from_counts(mcounts)
    mdoff = offsets_dev(moff)
    E = len(mcounts)
    M = int(moff[-1]) + 32
    for tB, N, K in [(False, 256, 256), (True, 256, 256)]:
        xq = W.e4m3_codes((M, K), 7, 0)
        wq = W.e4m3_codes((E, K, N) if tB else (E, N, K), 7, 1)
        sx = W.e8m0_codes((M, K // 32), *W.MX_ACT_SCALES, 7, 2)
        sw = W.e8m0_codes((E, N, K // 32), *W.mx_weight_scales(K), 7, 3)
        sxb = rg.mx_scales_blocked(torch.from_numpy(sx).cuda(), mdoff)
        swb = rg.mx_scales_blocked(torch.from_numpy(sw.reshape(E * N, K // 32)).cuda(), rg.mx_weight_offsets(E, N))
        y = rg.mgemm_mxfp8(torch.from_numpy(xq).cuda(), sxb, torch.from_numpy(wq).cuda(), swb, mdoff, transpose_B=tB)
        status(f"mgemm_mxfp8 tB={tB}")
        v = int(moff[-1])
        check_bf16(to_host_bits(y)[:v], oracle.mgemm_mx(xq, sx, wq, sw, moff, transpose_B=tB)[:v], "mx mgemm")
    N, K = 272, 320
    gq, xq = W.e4m3_codes((M, N), 8, 0), W.e4m3_codes((M, K), 8, 1)
    sg = W.e8m0_codes((N, M // 32), *W.MX_ACT_SCALES, 8, 2)
    sx = W.e8m0_codes((K, M // 32), *W.MX_ACT_SCALES, 8, 3)
    dW = rg.kgemm_mxfp8(torch.from_numpy(gq).cuda(), rg.mx_scales_blocked_k(torch.from_numpy(sg).cuda(), mdoff),
                        torch.from_numpy(xq).cuda(), rg.mx_scales_blocked_k(torch.from_numpy(sx).cuda(), mdoff), mdoff)
    status("kgemm_mxfp8")
    check_fp32(dW.cpu().numpy(), oracle.kgemm_mx(gq, sg, xq, sx, moff), "mx kgemm")
    print(f"ALL OK {len(results)} cases", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
