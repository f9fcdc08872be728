"""Host logic of bench.py that feeds the reported roofline, without a GPU:
the DRAM-traffic lookup keyed to kernel sources, the algorithmic byte counts
(against byte sizes of the tensors each op reads and writes), the peak
selection, and the kernel and byte mapping of every registered workload."""
import hashlib
import json
import os

import numpy as np
import pytest

import bench
import workloads as W


def fake_tree(tmp_path, source: bytes, entry: dict):
    csrc = tmp_path / "moe_grouped_gemm_device_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "kgemm.cu").write_bytes(source)
    for h in bench.KERNEL_SOURCES["kgemm_kernel"][1:]:  # the headers, as in the package
        (csrc / h).write_bytes(b"// header " + h.encode() + b"\n")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kgemm_kernel": entry}))


def test_traffic_only_for_the_captured_source_and_workload(tmp_path, monkeypatch):
    src = b"// kernel source as captured\n"
    h = hashlib.sha256(src + b"".join(b"// header " + n.encode() + b"\n"
                                      for n in bench.KERNEL_SOURCES["kgemm_kernel"][1:])).hexdigest()[:16]
    fake_tree(tmp_path, src, {"source_sha256_16": h,
                              "workloads": {"a3b": {"wgrad_gw2": 700, "wgrad_gw13": 1300},
                                            "skewed": {"wgrad_gw13": 5000}}})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2", "wgrad_gw13"], "a3b") == 1000
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw13"], "a3b") == 1300
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw13"], "skewed") == 5000
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2", "wgrad_gw13"], "skewed") is None  # gw2 not captured
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw13"], "uniform") is None  # workload not captured
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2", "other_op"], "a3b") is None  # an op not captured
    assert bench.traffic_for("kgemm_kernel", [], "a3b") is None
    assert bench.traffic_for("mx_kgemm_kernel", ["wgrad_gw2"], "a3b") is None  # no entry
    # the kernel changed since the capture: no traffic figure
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2"], "a3b") == 700
    (tmp_path / "moe_grouped_gemm_device_gb300" / "csrc" / "kgemm.cu").write_bytes(src + b"// edit\n")
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2"], "a3b") is None
    # or a header it includes changed
    (tmp_path / "moe_grouped_gemm_device_gb300" / "csrc" / "kgemm.cu").write_bytes(src)
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2"], "a3b") == 700
    (tmp_path / "moe_grouped_gemm_device_gb300" / "csrc" / "ptx.cuh").write_bytes(b"// edited\n")
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2"], "a3b") is None


def test_committed_traffic_entries_name_known_kernels_and_workloads():
    """Every record names a kernel the bench knows, a workload and ops of that
    workload which the bench maps to that kernel, and bytes within a plausible
    band of the op's algorithmic bytes (outputs still in L2 at the kernel's end
    lower them, re-reads raise them): a record keyed to the wrong op or kernel
    fails here."""
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    by_name = {W.ALL[n]().name: W.ALL[n]() for n in W.ALL}
    for k, ent in d.items():
        if k.startswith("_"):
            continue
        assert k in bench.KERNEL_SOURCES, k
        assert len(ent["source_sha256_16"]) == 16
        for wl, per_op in ent["workloads"].items():
            assert wl in by_name, wl
            ops = {op.name: op for op in by_name[wl].ops}
            for name, v in per_op.items():
                assert isinstance(v, int) and v > 0, (k, wl, name)
                assert name in ops, (k, wl, name)
                assert bench.kernel_of(ops[name]) == k, (k, wl, name)
                ratio = v / bench.algorithmic_bytes(ops[name], by_name[wl].counts)
                assert 0.4 <= ratio <= 2.5, (k, wl, name, ratio)


def test_peak_kind_follows_the_timed_region():
    capped = {"sm_mhz": 1600.0, "reasons": ["sw_power_cap"]}
    free = {"sm_mhz": 2070.0, "reasons": []}
    # a short region runs at burst clocks whatever the record says
    assert bench.peak_kind(0.03, capped) == "burst"
    assert bench.peak_kind(0.03, free) == "burst"
    assert bench.peak_kind(0.03, None) == "burst"
    # a long region is compared with the sustained figure only when it was power-capped
    assert bench.peak_kind(2.0, capped) == "sustained"
    assert bench.peak_kind(2.0, free) == "burst"
    assert bench.peak_kind(2.0, None) == "burst"
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    assert bench.tensor_peak("kgemm_kernel", peaks, "burst") == 1900.0
    assert bench.tensor_peak("kgemm_kernel", peaks, "sustained") == 1700.0


def test_both_arms_print_the_same_config():
    """The reference arm's config is the GPU arm's (config_of), and it holds
    nothing measured."""
    wl = W.ALL["a3b"]()
    c = bench.config_of(wl)
    assert c == bench.config_of(W.ALL["a3b"]())
    assert set(c) == {"workload", "flops_per_step", "l2"}
    assert c["flops_per_step"] == wl.flops()
    assert "larger than L2" in c["l2"]
    assert "flushed" in bench.config_of(W.ALL["uniform8"]())["l2"]


def test_reference_budget_keeps_the_run_short():
    for steps, warmup in ((20, 5), (1000, 20), (1, 0)):
        b = bench.reference_budget_s(steps, warmup)
        assert 0.05 <= b <= 2.0
        assert (steps + warmup) * b <= max(90.0, 0.05 * (steps + warmup)) + 1e-9


COUNTS = np.array([3, 0, 5, 9])  # one empty group


def nbytes(*arrays):
    return sum(a.nbytes for a in arrays)


def test_algorithmic_bytes_match_tensor_sizes():
    M, E, N, K = int(COUNTS.sum()), len(COUNTS), 24, 40
    bf16 = np.float16  # two bytes, as bf16
    x, y = np.empty((M, K), bf16), np.empty((M, N), bf16)
    w_used = np.empty((3, N, K), bf16)  # the empty group's weights are never read
    fwd = W.Op("fwd", "mgemm", "x", "w", N, K)
    assert bench.algorithmic_bytes(fwd, COUNTS) == nbytes(x, w_used, y)
    dgrad = W.Op("dgrad", "mgemm", "x", "w", N, K, transpose_B=True)
    assert bench.algorithmic_bytes(dgrad, COUNTS) == nbytes(x, w_used, y)
    g = np.empty((M, N), bf16)
    dW = np.empty((E, N, K), np.float32)  # every group's dW is written (zeros for the empty one)
    wgrad = W.Op("wgrad", "kgemm", "g", "x", N, K)
    assert bench.algorithmic_bytes(wgrad, COUNTS) == nbytes(g, x, dW)
    acc = W.Op("wgrad_acc", "kgemm", "g", "x", N, K, accumulate=True)
    assert bench.algorithmic_bytes(acc, COUNTS) == nbytes(g, x, dW, dW)  # dW read and written
    h, y13 = np.empty((M, N // 2), bf16), np.empty((M, N), bf16)
    swiglu = W.Op("swiglu", "mgemm", "x", "w", N, K, fuse="swiglu")
    assert bench.algorithmic_bytes(swiglu, COUNTS) == nbytes(x, w_used, h, y13)


def test_fp8_kernels_take_twice_the_bf16_peak():
    peaks = {"bf16_tflops": 1100.0, "bf16_tflops_sustained": 1000.0}
    for k in bench.FP8_KERNELS:
        assert bench.tensor_peak(k, peaks, "sustained") == 2000.0
        assert bench.tensor_peak(k, peaks, "burst") == 2200.0
    assert bench.tensor_peak("kgemm_kernel", peaks, "sustained") == 1000.0
    assert bench.tensor_peak("mgemm_kernel<true>", peaks, "burst") == 1100.0


@pytest.mark.parametrize("name", sorted(W.ALL))
def test_every_workload_maps_to_kernels_and_bytes(name):
    wl = W.ALL[name]()
    for op in wl.ops:
        k = bench.kernel_of(op)
        assert k in bench.KERNEL_SOURCES, (name, op.name, k)
        assert bench.algorithmic_bytes(op, wl.counts) > 0
    assert bench.working_set_bytes(wl) > 0
    assert bench.workload_desc(wl).startswith(wl.name + ":")


@pytest.mark.parametrize("name", ["a3b", "skewed", "a3b_acc", "a3b_swiglu", "lora_a3b"])
def test_step_buffers_have_the_outputs_types(name):
    """Output buffers of every op as bench.py makes them (on the host here):
    fp32 dW [E, N, K] for the weight gradients, bf16 elsewhere; a flag
    workspace only for weight gradients of workloads with an expert longer
    than one accumulation chunk."""
    torch = pytest.importorskip("torch")
    import moe_grouped_gemm_device_gb300 as rg
    wl = W.ALL[name]()
    outs, scratch = bench.make_buffers(wl, rg, "cpu")
    long_expert = int(np.max(wl.counts)) > bench.KGEMM_CHUNK_ROWS
    for op in wl.ops:
        out = outs[op.name]
        if op.kind == "kgemm":
            assert out.dtype == torch.float32 and tuple(out.shape) == (wl.E, op.N, op.K)
            assert (op.name + ":ws" in scratch) == long_expert
            if long_expert:
                assert scratch[op.name + ":ws"].numel() == rg.kgemm_workspace_bytes(wl.E, op.N, op.K)
        else:
            assert out.dtype == torch.bfloat16
