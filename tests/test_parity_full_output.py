"""GPU parity at the full workload sizes on EVERY output element, one case per
kernel family, in the launch configuration the benchmark times: the M-grouped
forward and input gradient (30B-A3B gate-up), the K-grouped FP32 weight
gradient (30B-A3B gw13, and the skewed workload with tiny and empty experts,
whose 18k-row expert is the longest FP32 accumulation), the MXFP8 forward
(down projection: its oracle decodes every element, the slowest to compute)
and weight gradient, the nested grouped GEMM of the LoRA workload (the
64-column shrink tile and the two-outer-group expand), both fused SwiGLU
kernels (gate-up forward with h and the saved pre-activation, down-projection
input gradient with the SwiGLU backward), the weight gradient accumulated
into an FP32 main grad, and, bit for bit, every scale-layout conversion of
the MXFP8 benchmark step.  The oracle computes every output (chunk by chunk, so host memory
stays bounded) and the relative Frobenius error is that of the whole output;
bf16 outputs also meet the per-element bound everywhere.  Rows of y at or past
offsets[E] must keep their sentinel, and experts without rows must get dW = 0
exactly.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import FullCompare, offsets_dev, to_dev, to_host_bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROW_CHUNK = 4096        # Mgemm rows per oracle call
EXPERT_BYTES = 1 << 29  # float64 bytes of dW per oracle call (Kgemm)

MG = [("a3b", "fwd_gate_up"), ("a3b", "dgrad_gate_up")]
KG = [("a3b", "wgrad_gw13"), ("skewed_tail", "wgrad_gw13")]


@pytest.mark.parametrize("wname,opname", MG, ids=[f"{w}-{o}" for w, o in MG])
def test_full_output_mgemm(gpu_lib, wname, opname):
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    a_h, b_h = wl.tensor(op.a), wl.tensor(op.b)
    y = torch.full((wl.M, op.N), 7.0, dtype=torch.bfloat16, device="cuda")  # sentinel
    gpu_lib.mgemm(to_dev(a_h), to_dev(b_h), offsets_dev(off), transpose_B=op.transpose_B, out=y)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp = FullCompare("bf16", f"{wname}/{opname}/full")
    n = int(off[-1])
    for r0 in range(0, n, ROW_CHUNK):
        rows = np.arange(r0, min(n, r0 + ROW_CHUNK), dtype=np.int64)
        ref = oracle.mgemm(a_h, b_h, off, transpose_B=op.transpose_B, rows=rows)
        cmp.add(to_host_bits(y[r0:r0 + len(rows)]), ref)
    rec = cmp.finish()
    assert rec["elements"] == n * op.N
    if n < wl.M:
        assert bool((y[n:] == 7.0).all()), "rows past offsets[E] were written"


@pytest.mark.parametrize("wname,opname", KG, ids=[f"{w}-{o}" for w, o in KG])
def test_full_output_kgemm(gpu_lib, wname, opname):
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    a_h, b_h = wl.tensor(op.a), wl.tensor(op.b)
    dW = gpu_lib.kgemm(to_dev(a_h), to_dev(b_h), offsets_dev(off))
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp = FullCompare("fp32", f"{wname}/{opname}/full")
    per = max(1, EXPERT_BYTES // (8 * op.N * op.K))
    for e0 in range(0, wl.E, per):
        es = np.arange(e0, min(wl.E, e0 + per), dtype=np.int32)
        sel = (np.repeat(es, op.N), np.tile(np.arange(op.N, dtype=np.int32), len(es)))
        ref = oracle.kgemm(a_h, b_h, off, sel=sel)
        cmp.add(dW[int(es[0]):int(es[-1]) + 1].reshape(-1, op.K).cpu().numpy(), ref)
    rec = cmp.finish()
    assert rec["elements"] == wl.E * op.N * op.K
    for e in np.flatnonzero(wl.counts == 0):
        assert bool((dW[int(e)] == 0).all()), f"expert {e} has no rows but dW[e] != 0"


def test_full_output_mx_kgemm(gpu_lib):
    import torch
    wl = W.ALL["a3b_mxfp8"]()
    op = wl.op("mx_wgrad_gw13")
    off = wl.offsets
    h = {k: wl.tensor(k) for k in (op.a, op.b, op.sa, op.sb)}
    d = {k: torch.from_numpy(v).cuda() for k, v in h.items()}
    doff = offsets_dev(off)
    dW = gpu_lib.kgemm_mxfp8(d[op.a], gpu_lib.mx_scales_blocked_k(d[op.sa], doff), d[op.b],
                             gpu_lib.mx_scales_blocked_k(d[op.sb], doff), doff)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp = FullCompare("fp32", "a3b_mxfp8/mx_wgrad_gw13/full")
    per = max(1, EXPERT_BYTES // (8 * op.N * op.K))
    for e0 in range(0, wl.E, per):
        es = np.arange(e0, min(wl.E, e0 + per), dtype=np.int32)
        sel = (np.repeat(es, op.N), np.tile(np.arange(op.N, dtype=np.int32), len(es)))
        ref = oracle.kgemm_mx(h[op.a], h[op.sa], h[op.b], h[op.sb], off, sel=sel)
        cmp.add(dW[int(es[0]):int(es[-1]) + 1].reshape(-1, op.K).cpu().numpy(), ref)
    rec = cmp.finish()
    assert rec["elements"] == wl.E * op.N * op.K


NESTED = [("lora_a3b", "lora_shrink"), ("lora_a3b", "lora_expand")]


@pytest.mark.parametrize("wname,opname", NESTED, ids=[f"{w}-{o}" for w, o in NESTED])
def test_full_output_nested(gpu_lib, wname, opname):
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    a_h, b_h = wl.tensor(op.a), wl.tensor(op.b)
    y = torch.full((wl.M, op.outer * op.N), 7.0, dtype=torch.bfloat16, device="cuda")  # sentinel
    gpu_lib.mgemm_nested(to_dev(a_h), to_dev(b_h), offsets_dev(off), transpose_B=op.transpose_B, out=y)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp = FullCompare("bf16", f"{wname}/{opname}/full")
    n = int(off[-1])
    for r0 in range(0, n, ROW_CHUNK):
        rows = np.arange(r0, min(n, r0 + ROW_CHUNK), dtype=np.int64)
        ref = oracle.mgemm_nested(a_h, b_h, off, transpose_B=op.transpose_B, rows=rows)
        cmp.add(to_host_bits(y[r0:r0 + len(rows)]), ref)
    rec = cmp.finish()
    assert rec["elements"] == n * op.outer * op.N
    if n < wl.M:
        assert bool((y[n:] == 7.0).all()), "rows past offsets[L] were written"


def test_full_output_mx_mgemm(gpu_lib):
    import torch
    wl = W.ALL["a3b_mxfp8"]()
    op = wl.op("mx_fwd_down")
    off = wl.offsets
    h = {k: wl.tensor(k) for k in (op.a, op.b, op.sa, op.sb)}
    d = {k: torch.from_numpy(v).cuda() for k, v in h.items()}
    doff = offsets_dev(off)
    sab = gpu_lib.mx_scales_blocked(d[op.sa], doff)
    sbb = gpu_lib.mx_scales_blocked(d[op.sb].view(-1, d[op.sb].shape[-1]), gpu_lib.mx_weight_offsets(wl.E, op.N))
    y = torch.full((wl.M, op.N), 7.0, dtype=torch.bfloat16, device="cuda")  # sentinel
    gpu_lib.mgemm_mxfp8(d[op.a], sab, d[op.b], sbb, doff, transpose_B=op.transpose_B, out=y)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp = FullCompare("bf16", "a3b_mxfp8/mx_fwd_down/full")
    n = int(off[-1])
    for r0 in range(0, n, ROW_CHUNK):
        rows = np.arange(r0, min(n, r0 + ROW_CHUNK), dtype=np.int64)
        ref = oracle.mgemm_mx(h[op.a], h[op.sa], h[op.b], h[op.sb], off, transpose_B=op.transpose_B, rows=rows)
        cmp.add(to_host_bits(y[r0:r0 + len(rows)]), ref)
    rec = cmp.finish()
    assert rec["elements"] == n * op.N
    if n < wl.M:
        assert bool((y[n:] == 7.0).all()), "rows past offsets[E] were written"


def test_full_output_swiglu_forward(gpu_lib):
    import torch
    wl = W.ALL["a3b_swiglu"]()
    op = wl.op("fwd_gate_up_swiglu")
    off = wl.offsets
    a_h, b_h = wl.tensor(op.a), wl.tensor(op.b)
    h, y13 = gpu_lib.mgemm_swiglu(to_dev(a_h), to_dev(b_h), offsets_dev(off), y13=True)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp_h = FullCompare("bf16", "a3b_swiglu/fwd_gate_up_swiglu/h/full")
    cmp_y = FullCompare("bf16", "a3b_swiglu/fwd_gate_up_swiglu/y13/full")
    n = int(off[-1])
    for r0 in range(0, n, ROW_CHUNK):
        rows = np.arange(r0, min(n, r0 + ROW_CHUNK), dtype=np.int64)
        y_ref = oracle.mgemm(a_h, b_h, off, rows=rows)
        cmp_y.add(to_host_bits(y13[r0:r0 + len(rows)]), y_ref)
        cmp_h.add(to_host_bits(h[r0:r0 + len(rows)]), oracle.swiglu(y_ref))
    assert cmp_y.finish()["elements"] == n * op.N
    assert cmp_h.finish()["elements"] == n * op.N // 2


def test_full_output_swiglu_input_gradient(gpu_lib):
    import torch
    wl = W.ALL["a3b_swiglu"]()
    op = wl.op("dgrad_down_swiglu")
    off = wl.offsets
    a_h, b_h, c_h = wl.tensor(op.a), wl.tensor(op.b), wl.tensor(op.c)
    dy13 = gpu_lib.mgemm_swiglu_dgrad(to_dev(a_h), to_dev(b_h), offsets_dev(off), to_dev(c_h))
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp = FullCompare("bf16", "a3b_swiglu/dgrad_down_swiglu/full")
    n = int(off[-1])
    for r0 in range(0, n, ROW_CHUNK):
        rows = np.arange(r0, min(n, r0 + ROW_CHUNK), dtype=np.int64)
        dh = oracle.mgemm(a_h, b_h, off, transpose_B=True, rows=rows)
        cmp.add(to_host_bits(dy13[r0:r0 + len(rows)]), oracle.swiglu_bwd(dh, W.bf16_bits_to_f32(c_h[rows])))
    assert cmp.finish()["elements"] == n * 2 * op.N


def test_full_output_kgemm_accumulate(gpu_lib):
    import torch
    wl = W.ALL["a3b_acc"]()
    op = wl.op("wgrad_gw2_acc")
    off = wl.offsets
    a_h, b_h = wl.tensor(op.a), wl.tensor(op.b)
    init = W.bf16_bits_to_f32(W.normal_bf16((wl.E, op.N, op.K), 1.0, wl.seed, 90))
    dW = torch.from_numpy(init).cuda()
    gpu_lib.kgemm(to_dev(a_h), to_dev(b_h), offsets_dev(off), out=dW, accumulate=True)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    cmp = FullCompare("fp32", "a3b_acc/wgrad_gw2_acc/full")
    per = max(1, EXPERT_BYTES // (8 * op.N * op.K))
    for e0 in range(0, wl.E, per):
        es = np.arange(e0, min(wl.E, e0 + per), dtype=np.int32)
        sel = (np.repeat(es, op.N), np.tile(np.arange(op.N, dtype=np.int32), len(es)))
        ref = oracle.kgemm(a_h, b_h, off, sel=sel) + init[e0:e0 + len(es)].reshape(-1, op.K).astype(np.float64)
        cmp.add(dW[int(es[0]):int(es[-1]) + 1].reshape(-1, op.K).cpu().numpy(), ref)
    assert cmp.finish()["elements"] == wl.E * op.N * op.K


def test_full_output_mx_scale_layouts(gpu_lib):
    """Every conversion of the MXFP8 step at its full size, bit for bit: the
    activation and weight scales of the four M-grouped GEMMs (blocked layout,
    groups along the rows) and the scales of the two weight gradients (groups
    along the contraction); nothing past the used blocks is written."""
    import torch
    wl = W.ALL["a3b_mxfp8"]()
    off = wl.offsets
    doff = offsets_dev(off)

    def rows_grouped(src, goff):
        R, KS = src.shape
        G = len(goff) - 1
        used = sum((int(goff[g + 1]) - int(goff[g]) + 127) // 128 for g in range(G)) * ((KS + 3) // 4) * 512
        out = torch.full((gpu_lib.mx_blocked_bytes(R, KS, G),), 0xEE, dtype=torch.uint8, device="cuda")
        gpu_lib.mx_scales_blocked(torch.from_numpy(src).cuda(), offsets_dev(goff), out=out)
        return out, used, oracle.mx_blocked(src, goff)

    def contraction_grouped(src, goff):
        R, KS = src.shape
        G = len(goff) - 1
        nq = sum((int(goff[g + 1]) - int(goff[g]) + 127) // 128 for g in range(G))
        used = ((R + 127) // 128) * nq * 512
        out = torch.full((gpu_lib.mx_blocked_k_bytes(R, KS, G),), 0xEE, dtype=torch.uint8, device="cuda")
        gpu_lib.mx_scales_blocked_k(torch.from_numpy(src).cuda(), doff, out=out)
        return out, used, oracle.mx_blocked_k(src, goff)

    checked = 0
    for op in wl.ops:
        if op.kind == "mx":
            sa = wl.tensor(op.sa)
            sb = wl.tensor(op.sb)
            cases = [rows_grouped(sa, off),
                     rows_grouped(sb.reshape(-1, sb.shape[-1]), np.arange(0, (wl.E + 1) * op.N, op.N, dtype=np.int32))]
        else:
            cases = [contraction_grouped(wl.tensor(op.sa), off), contraction_grouped(wl.tensor(op.sb), off)]
        for out, used, want in cases:
            torch.cuda.synchronize()
            assert gpu_lib.device_status() == 0
            got = out.cpu().numpy()
            np.testing.assert_array_equal(got[:used], want[:used], err_msg=op.name)
            assert (got[used:] == 0xEE).all(), f"{op.name}: bytes past the used blocks were written"
            checked += 1
    assert checked == 12
