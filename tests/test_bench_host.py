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
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kgemm_kernel": entry}))


def test_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    src = b"// kernel source as captured\n"
    h = hashlib.sha256(src).hexdigest()[:16]
    fake_tree(tmp_path, src, {"source_sha256_16": h, "per_op": {"wgrad_gw2": 700, "wgrad_gw13": 1300}})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2", "wgrad_gw13"]) == 1000
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw13"]) == 1300
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2", "other_op"]) is None  # an op not captured
    assert bench.traffic_for("kgemm_kernel", []) is None
    assert bench.traffic_for("mx_kgemm_kernel", ["wgrad_gw2"]) is None  # no entry
    # the kernel changed since the capture: no traffic figure
    (tmp_path / "moe_grouped_gemm_device_gb300" / "csrc" / "kgemm.cu").write_bytes(src + b"// edit\n")
    assert bench.traffic_for("kgemm_kernel", ["wgrad_gw2"]) is None


def test_committed_traffic_entries_name_known_kernels():
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for k, ent in d.items():
        if k.startswith("_"):
            continue
        assert k in bench.KERNEL_SOURCES, k
        assert len(ent["source_sha256_16"]) == 16
        assert all(isinstance(v, int) and v > 0 for v in ent["per_op"].values())


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
    peaks = {"bf16_tflops_sustained": 1000.0}
    for k in bench.FP8_KERNELS:
        assert bench.tensor_peak(k, peaks) == 2000.0
    assert bench.tensor_peak("kgemm_kernel", peaks) == 1000.0
    assert bench.tensor_peak("mgemm_kernel<true>", peaks) == 1000.0


@pytest.mark.parametrize("name", sorted(W.ALL))
def test_every_workload_maps_to_kernels_and_bytes(name):
    wl = W.ALL[name]()
    for op in wl.ops:
        k = bench.kernel_of(op)
        assert k in bench.KERNEL_SOURCES, (name, op.name, k)
        assert bench.algorithmic_bytes(op, wl.counts) > 0
    assert bench.working_set_bytes(wl) > 0
    assert bench.workload_desc(wl).startswith(wl.name + ":")
