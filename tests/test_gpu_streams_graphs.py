"""Stream semantics of the C ABI: calls on different streams run
independently and give the same bits as one stream, and a sequence of calls
(no host synchronisation, no allocation inside the library) can be captured
in a CUDA graph and replayed with new inputs -- the workspace entry point's
flag clear included."""
import numpy as np
import pytest

import workloads as W
from parity import offsets_dev, to_dev

pytestmark = pytest.mark.gpu


def layer_inputs(seed):
    counts = [300, 0, 17, 513, 128]
    off = W.offsets_from_counts(counts)
    E, N, K = len(counts), 384, 256
    M = int(off[-1]) + 4
    return dict(off=off, x=W.normal_bf16((M, K), 1.0, seed, 0), w=W.normal_bf16((E, N, K), 0.06, seed, 1),
                g=W.normal_bf16((M, N), 1.0, seed, 2), E=E, N=N, K=K, M=M,
                # a contraction of 16: single-CTA one-stage tiles with 16-column operand boxes
                x16=W.normal_bf16((M, 16), 1.0, seed, 3), w16=W.normal_bf16((E, N, 16), 0.25, seed, 4))


def run_ops(rg, d, outs, stream=None):
    rg.mgemm(d["x"], d["w"], d["off"], out=outs["y"], stream=stream)
    rg.mgemm(d["g"], d["w"], d["off"], transpose_B=True, out=outs["dx"], stream=stream)
    rg.kgemm(d["g"], d["x"], d["off"], out=outs["dw"], stream=stream)
    rg.mgemm(d["x16"], d["w16"], d["off"], out=outs["y16"], stream=stream)


def device_inputs(p):
    return dict(off=offsets_dev(p["off"]), x=to_dev(p["x"]), w=to_dev(p["w"]), g=to_dev(p["g"]),
                x16=to_dev(p["x16"]), w16=to_dev(p["w16"]))


def empty_outputs(p):
    import torch
    return dict(y=torch.empty((p["M"], p["N"]), dtype=torch.bfloat16, device="cuda"),
                dx=torch.empty((p["M"], p["K"]), dtype=torch.bfloat16, device="cuda"),
                dw=torch.empty((p["E"], p["N"], p["K"]), dtype=torch.float32, device="cuda"),
                y16=torch.empty((p["M"], p["N"]), dtype=torch.bfloat16, device="cuda"))


def same_bits(a, b, rows):
    import torch
    for k in ("y", "dx", "y16"):
        assert torch.equal(a[k][:rows].view(torch.int16), b[k][:rows].view(torch.int16)), k
    assert torch.equal(a["dw"].view(torch.int32), b["dw"].view(torch.int32)), "dw"


def test_two_streams_match_one_stream(gpu_lib):
    import torch
    pa, pb = layer_inputs(41), layer_inputs(42)
    da, db = device_inputs(pa), device_inputs(pb)
    ref_a, ref_b = empty_outputs(pa), empty_outputs(pb)
    run_ops(gpu_lib, da, ref_a)
    run_ops(gpu_lib, db, ref_b)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    out_a, out_b = empty_outputs(pa), empty_outputs(pb)
    torch.cuda.synchronize()
    for _ in range(3):  # interleaved launches on both streams
        run_ops(gpu_lib, da, out_a, stream=sa)
        run_ops(gpu_lib, db, out_b, stream=sb)
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    same_bits(out_a, ref_a, int(pa["off"][-1]))
    same_bits(out_b, ref_b, int(pb["off"][-1]))


def test_graph_capture_and_replay(gpu_lib):
    import torch
    p0, p1 = layer_inputs(43), layer_inputs(44)
    static = device_inputs(p0)
    outs = empty_outputs(p0)
    run_ops(gpu_lib, static, outs)  # library state set up before the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_ops(gpu_lib, static, outs)
    for p in (p1, p0, p1):  # new inputs copied into the captured buffers
        src = device_inputs(p)
        for k in ("x", "w", "g", "off", "x16", "w16"):
            static[k].copy_(src[k])
        graph.replay()
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        ref = empty_outputs(p)
        run_ops(gpu_lib, src, ref)
        torch.cuda.synchronize()
        same_bits(outs, ref, int(p["off"][-1]))


def test_graph_capture_of_the_workspace_entry_point(gpu_lib):
    """rg_kgemm_ws in a captured graph: its flag clear (a memset node) and the
    chunk-major kernel (90 dW tiles per expert, experts of several chunks)
    replayed with new inputs give rg_kgemm's bits each time."""
    import torch
    counts = [5000, 0, 300, 9000, 37]
    off = W.offsets_from_counts(counts)
    E, N, K = len(counts), 2560, 2304
    M = int(off[-1]) + 2

    def inputs(seed):
        return dict(g=to_dev(W.normal_bf16((M, N), 1.0, seed, 0)), x=to_dev(W.normal_bf16((M, K), 1.0, seed, 1)))

    static = inputs(45)
    doff = offsets_dev(off)
    ws = torch.empty(gpu_lib.kgemm_workspace_bytes(E, N, K), dtype=torch.uint8, device="cuda")
    dw = torch.empty((E, N, K), dtype=torch.float32, device="cuda")
    gpu_lib.kgemm(static["g"], static["x"], doff, out=dw, workspace=ws)  # set-up before the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu_lib.kgemm(static["g"], static["x"], doff, out=dw, workspace=ws)
    for seed in (46, 45, 47):
        src = inputs(seed)
        static["g"].copy_(src["g"])
        static["x"].copy_(src["x"])
        dw.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert gpu_lib.device_status() == 0
        ref = gpu_lib.kgemm(src["g"], src["x"], doff)
        torch.cuda.synchronize()
        assert torch.equal(dw.view(torch.int32), ref.view(torch.int32))
