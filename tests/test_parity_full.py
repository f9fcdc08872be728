"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times, on sampled outputs that the oracle computes one by one.

Sampled Mgemm rows: the first and last row of every non-empty expert (the
ragged tile edges) plus random rows; every column of each sampled row is
checked.  Sampled Kgemm rows of dW: for every expert, n = 0, 127, 128, N-1
and a random n (tile edges along N); every k of each row is checked.  Empty
experts must give dW[e] == 0 exactly (checked in full).
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads as W
from parity import check_bf16, check_fp32, offsets_dev, to_dev, to_host_bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

_HOST = {}


def host_tensor(wl, name):
    shape, std, stream = wl.tensors[name]
    key = (wl.seed, stream, tuple(shape), std)
    if key not in _HOST:
        _HOST[key] = W.normal_bf16(shape, std, wl.seed, stream)
    return _HOST[key]


_DEV = {}


def dev_tensor(wl, name):
    shape, std, stream = wl.tensors[name]
    key = (wl.seed, stream, tuple(shape), std)
    if key not in _DEV:
        _DEV[key] = to_dev(host_tensor(wl, name))
    return _DEV[key]


def sample_rows(off, rng, n_random=256):
    rows = []
    for e in range(len(off) - 1):
        if off[e + 1] > off[e]:
            rows += [int(off[e]), int(off[e + 1]) - 1]
    rows += list(rng.integers(0, int(off[-1]), size=n_random))
    return np.unique(np.array(rows, dtype=np.int64))


def sample_pairs(counts, N, rng):
    es, ns = [], []
    for e in range(len(counts)):
        if counts[e] == 0:
            continue
        for n in sorted({0, min(127, N - 1), min(128, N - 1), N - 1, int(rng.integers(0, N))}):
            es.append(e)
            ns.append(n)
    return np.array(es, dtype=np.int32), np.array(ns, dtype=np.int32)


MX = [("a3b_mxfp8", op) for op in ("mx_fwd_gate_up", "mx_fwd_down", "mx_dgrad_down", "mx_dgrad_gate_up",
                                    "mx_wgrad_gw2", "mx_wgrad_gw13")]


def dev_u8(wl, name):
    shape, kind, stream = wl.tensors[name]
    key = (wl.seed, stream, tuple(shape), str(kind))
    if key not in _DEV:
        import torch
        _DEV[key] = torch.from_numpy(host_u8(wl, name)).cuda()
    return _DEV[key]


def host_u8(wl, name):
    shape, kind, stream = wl.tensors[name]
    key = (wl.seed, stream, tuple(shape), str(kind))
    if key not in _HOST:
        _HOST[key] = wl.tensor(name)
    return _HOST[key]


@pytest.mark.parametrize("wname,opname", MX, ids=[f"{w}-{o}" for w, o in MX])
def test_full_size_sampled_mxfp8(gpu_lib, wname, opname):
    """Scale layout conversion and MXFP8 GEMM as the benchmark runs them."""
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    rng = np.random.default_rng(zlib.crc32(f"{wname}/{opname}".encode()))
    doff = offsets_dev(off)
    sa, sb = dev_u8(wl, op.sa), dev_u8(wl, op.sb)
    if op.kind == "mxk":
        dW = gpu_lib.kgemm_mxfp8(dev_u8(wl, op.a), gpu_lib.mx_scales_blocked_k(sa, doff), dev_u8(wl, op.b),
                                 gpu_lib.mx_scales_blocked_k(sb, doff), doff)
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        es, ns = sample_pairs(wl.counts, op.N, rng)
        got = dW[torch.from_numpy(es).long().cuda(), torch.from_numpy(ns).long().cuda()].cpu().numpy()
        ref = oracle.kgemm_mx(host_u8(wl, op.a), host_u8(wl, op.sa), host_u8(wl, op.b), host_u8(wl, op.sb), off,
                              sel=(es, ns))
        check_fp32(got, ref, f"{wname}/{opname}")
        return
    sab = gpu_lib.mx_scales_blocked(sa, doff)
    sbb = gpu_lib.mx_scales_blocked(sb.view(-1, sb.shape[-1]), gpu_lib.mx_weight_offsets(wl.E, op.N))
    y = gpu_lib.mgemm_mxfp8(dev_u8(wl, op.a), sab, dev_u8(wl, op.b), sbb, doff, transpose_B=op.transpose_B)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    rows = sample_rows(off, rng, n_random=32)
    got = to_host_bits(y[torch.from_numpy(rows).cuda()])
    ref = oracle.mgemm_mx(host_u8(wl, op.a), host_u8(wl, op.sa), host_u8(wl, op.b), host_u8(wl, op.sb), off,
                          transpose_B=op.transpose_B, rows=rows)
    check_bf16(got, ref, f"{wname}/{opname}")


NESTED = [("lora_a3b", "lora_shrink"), ("lora_a3b", "lora_expand")]


@pytest.mark.parametrize("wname,opname", NESTED, ids=[f"{w}-{o}" for w, o in NESTED])
def test_full_size_sampled_nested(gpu_lib, wname, opname):
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    rng = np.random.default_rng(zlib.crc32(f"{wname}/{opname}".encode()))
    a_h, b_h = host_tensor(wl, op.a), host_tensor(wl, op.b)
    y = gpu_lib.mgemm_nested(dev_tensor(wl, op.a), dev_tensor(wl, op.b), offsets_dev(off),
                             transpose_B=op.transpose_B)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    rows = sample_rows(off, rng)
    got = to_host_bits(y[torch.from_numpy(rows).cuda()])
    ref = oracle.mgemm_nested(a_h, b_h, off, transpose_B=op.transpose_B, rows=rows)
    check_bf16(got, ref, f"{wname}/{opname}")


CASES = [("uniform8", "fwd"), ("uniform16", "fwd")] + [
    (w, op) for w in ("a3b", "skewed", "skewed_tail")
    for op in ("fwd_gate_up", "fwd_down", "dgrad_down", "dgrad_gate_up", "wgrad_gw2", "wgrad_gw13")]


FUSED = [(w, op) for w in ("a3b_swiglu", "skewed_tail_swiglu")
         for op in ("fwd_gate_up_swiglu", "dgrad_down_swiglu")]


@pytest.mark.parametrize("wname,opname", FUSED, ids=[f"{w}-{o}" for w, o in FUSED])
def test_full_size_sampled_swiglu(gpu_lib, wname, opname):
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    rng = np.random.default_rng(zlib.crc32(f"{wname}/{opname}".encode()))
    a_h, b_h = host_tensor(wl, op.a), host_tensor(wl, op.b)
    a_d, b_d = dev_tensor(wl, op.a), dev_tensor(wl, op.b)
    doff = offsets_dev(off)
    rows = sample_rows(off, rng)
    sel = torch.from_numpy(rows).cuda()
    if op.fuse == "swiglu":
        h, y13 = gpu_lib.mgemm_swiglu(a_d, b_d, doff, y13=True)
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        y_ref = oracle.mgemm(a_h, b_h, off, rows=rows)
        check_bf16(to_host_bits(y13[sel]), y_ref, f"{wname}/{opname}/y13")
        check_bf16(to_host_bits(h[sel]), oracle.swiglu(y_ref), f"{wname}/{opname}/h")
    else:
        c_h, c_d = host_tensor(wl, op.c), dev_tensor(wl, op.c)
        dy13 = gpu_lib.mgemm_swiglu_dgrad(a_d, b_d, doff, c_d)
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        dh = oracle.mgemm(a_h, b_h, off, transpose_B=True, rows=rows)
        ref = oracle.swiglu_bwd(dh, W.bf16_bits_to_f32(c_h[rows]))
        check_bf16(to_host_bits(dy13[sel]), ref, f"{wname}/{opname}")


@pytest.mark.parametrize("wname,opname", CASES, ids=[f"{w}-{o}" for w, o in CASES])
def test_full_size_sampled(gpu_lib, wname, opname):
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    rng = np.random.default_rng(zlib.crc32(f"{wname}/{opname}".encode()))
    a_h, b_h = host_tensor(wl, op.a), host_tensor(wl, op.b)
    a_d, b_d = dev_tensor(wl, op.a), dev_tensor(wl, op.b)
    doff = offsets_dev(off)
    if op.kind == "mgemm":
        y = gpu_lib.mgemm(a_d, b_d, doff, transpose_B=op.transpose_B)
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        rows = sample_rows(off, rng)
        got = to_host_bits(y[torch.from_numpy(rows).cuda()])
        ref = oracle.mgemm(a_h, b_h, off, transpose_B=op.transpose_B, rows=rows)
        check_bf16(got, ref, f"{wname}/{opname}")
    else:
        dW = gpu_lib.kgemm(a_d, b_d, doff)
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        es, ns = sample_pairs(wl.counts, op.N, rng)
        got = dW[torch.from_numpy(es).long().cuda(), torch.from_numpy(ns).long().cuda()].cpu().numpy()
        ref = oracle.kgemm(a_h, b_h, off, sel=(es, ns))
        check_fp32(got, ref, f"{wname}/{opname}")
        for e in np.flatnonzero(wl.counts == 0):
            assert bool((dW[int(e)] == 0).all()), f"expert {e} has no rows but dW[e] != 0"
        del dW


ACC = [("a3b_acc", "wgrad_gw2_acc"), ("a3b_acc", "wgrad_gw13_acc")]


@pytest.mark.parametrize("wname,opname", ACC, ids=[f"{w}-{o}" for w, o in ACC])
def test_full_size_sampled_accumulate(gpu_lib, wname, opname):
    """Fused wgrad accumulation at full size: a seeded FP32 main grad plus the
    grouped weight gradient, on sampled dW rows."""
    import torch
    wl = W.ALL[wname]()
    op = wl.op(opname)
    off = wl.offsets
    rng = np.random.default_rng(zlib.crc32(f"{wname}/{opname}".encode()))
    a_h, b_h = host_tensor(wl, op.a), host_tensor(wl, op.b)
    init = W.bf16_bits_to_f32(W.normal_bf16((wl.E, op.N, op.K), 1.0, wl.seed, 90))
    dW = torch.from_numpy(init).cuda()
    gpu_lib.kgemm(dev_tensor(wl, op.a), dev_tensor(wl, op.b), offsets_dev(off), out=dW, accumulate=True)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    es, ns = sample_pairs(wl.counts, op.N, rng)
    got = dW[torch.from_numpy(es).long().cuda(), torch.from_numpy(ns).long().cuda()].cpu().numpy()
    ref = init[es, ns].astype(np.float64) + oracle.kgemm(a_h, b_h, off, sel=(es, ns))
    check_fp32(got, ref, f"{wname}/{opname}")
    del dW
