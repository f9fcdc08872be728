"""Benchmark of the MoE grouped GEMM path on GB300.

One step is one pass of the whole path over one batch: the six grouped GEMMs
of a 30B-A3B-shaped expert layer on one GPU (32 local experts, 32768 routed
rows with Dirichlet(2) counts, d_model 3072, expert FFN 1280):

    fwd  gate-up   y13 = x  . w13[e]^T     (M-grouped, N=2560, K=3072)
    fwd  down      y2  = h  . w2[e]^T      (M-grouped, N=3072, K=1280)
    dgrad down     dh  = dy2 . w2[e]       (M-grouped, transpose_B)
    dgrad gate-up  dx  = dy13 . w13[e]     (M-grouped, transpose_B)
    wgrad gw2      dW2[e]  = dy2[e]^T h[e]  (K-grouped, fp32)
    wgrad gw13     dW13[e] = dy13[e]^T x[e] (K-grouped, fp32)

Metric: grouped-GEMM TFLOP/s = sum over calls of 2*sum_e(M_e)*N*K / time.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

``--workload a3b_swiglu`` (or skewed_tail_swiglu) runs the same layer with
the SwiGLU activation fused into the gate-up forward and into the down
projection's input gradient.  ``--workload lora_a3b`` runs batched LoRA over
the same experts as nested grouped GEMMs (shrink, then the two-outer-group
expand).

prints one JSON line.  ``--impl reference`` times the CPU oracle on the same
workload (a bounded sample of it per step) on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

L2_BYTES = 129 * 2**20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_OF = {"mgemm": "mgemm_kernel<false>", "mgemm_t": "mgemm_kernel<true>", "kgemm": "kgemm_kernel",
             "swiglu": "mgemm_kernel<false,swiglu>", "swiglu_bwd": "mgemm_kernel<true,swiglu_bwd>",
             "mx": "mx_mgemm_kernel<false>", "mx_t": "mx_mgemm_kernel<true>", "mx_blocked": "mx_blocked_kernel",
             "mxk": "mx_kgemm_kernel", "mx_blocked_k": "mx_blocked_k_kernel"}
KERNEL_SOURCES = {"mgemm_kernel<false>": "mgemm.cu", "mgemm_kernel<true>": "mgemm.cu",
                  "mgemm_kernel<false,swiglu>": "mgemm.cu", "mgemm_kernel<true,swiglu_bwd>": "mgemm.cu",
                  "kgemm_kernel": "kgemm.cu", "mx_mgemm_kernel<false>": "mxgemm.cu",
                  "mx_mgemm_kernel<true>": "mxgemm.cu", "mx_blocked_kernel": "mxgemm.cu",
                  "mx_kgemm_kernel": "mxgemm.cu", "mx_blocked_k_kernel": "mxgemm.cu"}
FP8_KERNELS = ("mx_mgemm_kernel<false>", "mx_mgemm_kernel<true>", "mx_kgemm_kernel")
CONVERSION_KERNELS = ("mx_blocked_kernel", "mx_blocked_k_kernel")


def tensor_peak(kernel: str, peaks) -> float:
    """Sustained dense tensor peak of the kernel's input type: the measured
    bf16 figure, times the nominal dense FP8/BF16 ratio (4.5 / 2.25) for FP8."""
    return peaks["bf16_tflops_sustained"] * (2.0 if kernel in FP8_KERNELS else 1.0)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="a3b", choices=sorted(W.ALL))
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU baseline budget")
    p.add_argument("--ops", default="", help="comma-separated subset of the step's ops (profiling)")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_of(op) -> str:
    if op.kind == "mxk":
        return KERNEL_OF["mxk"]
    if op.kind == "mx":
        return KERNEL_OF["mx_t" if op.transpose_B else "mx"]
    if op.kind == "nested":
        return KERNEL_OF["mgemm_t" if op.transpose_B else "mgemm"]
    if op.fuse:
        return KERNEL_OF[op.fuse]
    if op.kind == "kgemm":
        return KERNEL_OF["kgemm"]
    return KERNEL_OF["mgemm_t" if op.transpose_B else "mgemm"]


def algorithmic_bytes(op, counts) -> int:
    M = int(np.sum(counts))
    E = len(counts)
    if op.kind == "kgemm":  # grad and X read, dW written (and read first when accumulating)
        return 2 * M * op.N + 2 * M * op.K + (8 if op.accumulate else 4) * E * op.N * op.K
    nonempty = int(np.count_nonzero(counts))
    if op.kind == "mxk":  # FP8 grad and X, their scales, fp32 dW
        return M * op.N + M * op.K + (op.N + op.K) * (M // 32) + 4 * E * op.N * op.K
    if op.kind == "mx":  # FP8 operands, their scales (1 byte per 32), bf16 y
        return M * op.K + op.N * op.K * nonempty + (M + op.N * nonempty) * (op.K // 32) + 2 * M * op.N
    if op.kind == "nested":  # x [M, O*K], w [O, L, N, K] (non-empty groups), y [M, O*N]
        return op.outer * (2 * M * op.K + 2 * op.N * op.K * nonempty + 2 * M * op.N)
    operands = 2 * M * op.K + 2 * op.N * op.K * nonempty
    if op.fuse == "swiglu":      # h [M, N/2] and y13 [M, N] written
        return operands + 2 * M * (op.N // 2) + 2 * M * op.N
    if op.fuse == "swiglu_bwd":  # y13 [M, 2N] read, dy13 [M, 2N] written
        return operands + 2 * 2 * M * (2 * op.N)
    return operands + 2 * M * op.N


def workload_desc(wl) -> str:
    ops = ", ".join(f"{o.name}(N={o.N},K={o.K})" for o in wl.ops)
    c = wl.counts
    return (f"{wl.name}: E={wl.E}, M={wl.M}, rows/expert min {int(c.min())} max {int(c.max())}; "
            f"one step = {ops}")


def working_set_bytes(wl) -> int:
    tot = 0
    for name, (shape, kind, _) in wl.tensors.items():
        tot += (1 if isinstance(kind, (str, tuple)) else 2) * int(np.prod(shape))
    for op in wl.ops:
        if op.kind in ("kgemm", "mxk"):
            tot += 4 * wl.E * op.N * op.K
        elif op.kind == "nested":
            tot += 2 * wl.M * op.outer * op.N
        elif op.fuse == "swiglu":
            tot += 2 * wl.M * (op.N // 2) + 2 * wl.M * op.N
        elif op.fuse == "swiglu_bwd":
            tot += 2 * wl.M * 2 * op.N
        else:
            tot += 2 * wl.M * op.N
    return tot


# --------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.4)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [s.strip() for s in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- CPU oracle


def oracle_sample_step(wl, tensors, budget_s: float, rng) -> tuple[float, float, str]:
    """Run the oracle on a sample of every op's outputs; return (flops, seconds,
    description).  Rows / (expert, n) pairs are drawn uniformly at random; the
    count per op is sized to the time budget from a one-row probe."""
    import oracle
    off = wl.offsets
    counts = wl.counts
    per_op = budget_s / len(wl.ops)
    flops = 0.0
    secs = 0.0
    desc = []
    for op in wl.ops:
        a, b = tensors[op.a], tensors[op.b]
        if op.kind == "mx":
            unit = 2.0 * op.N * op.K

            def run(n):
                rows = rng.integers(0, int(off[-1]), size=n)
                oracle.mgemm_mx(a, tensors[op.sa], b, tensors[op.sb], off, transpose_B=op.transpose_B, rows=rows)
                return n * unit
        elif op.kind == "mxk":
            nz = np.flatnonzero(counts)

            def run(n):
                es = rng.choice(nz, size=n)
                ns = rng.integers(0, op.N, size=n)
                oracle.kgemm_mx(a, tensors[op.sa], b, tensors[op.sb], off, sel=(es, ns))
                return float(np.sum(2.0 * counts[es] * op.K))
        elif op.kind == "nested":
            unit = 2.0 * op.outer * op.N * op.K

            def run(n):
                rows = rng.integers(0, int(off[-1]), size=n)
                oracle.mgemm_nested(a, b, off, transpose_B=op.transpose_B, rows=rows)
                return n * unit
        elif op.kind == "mgemm":
            unit = 2.0 * op.N * op.K

            def run(n):
                rows = rng.integers(0, int(off[-1]), size=n)
                y = oracle.mgemm(a, b, off, transpose_B=op.transpose_B, rows=rows)
                if op.fuse == "swiglu":
                    oracle.swiglu(y)
                elif op.fuse == "swiglu_bwd":
                    oracle.swiglu_bwd(y, W.bf16_bits_to_f32(tensors[op.c][rows]))
                return n * unit
        else:
            nz = np.flatnonzero(counts)

            def run(n):
                es = rng.choice(nz, size=n)
                ns = rng.integers(0, op.N, size=n)
                oracle.kgemm(a, b, off, sel=(es, ns))
                return float(np.sum(2.0 * counts[es] * op.K))
        t0 = time.perf_counter()
        f = run(max(1, oracle.num_threads()))
        dt = time.perf_counter() - t0
        n = max(1, int(oracle.num_threads() * per_op / max(dt, 1e-6)))
        t0 = time.perf_counter()
        f = run(n)
        dt = time.perf_counter() - t0
        flops += f
        secs += dt
        desc.append(f"{op.name}:{n}")
    return flops, secs, "random outputs per op (" + ", ".join(desc) + ")"


def cpu_baseline(wl, tensors, budget_s: float) -> dict:
    import oracle
    rng = np.random.default_rng(1234)
    flops, secs, desc = oracle_sample_step(wl, tensors, budget_s, rng)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{desc}; Mgemm ops: sampled rows x all N; Kgemm ops: sampled (expert, n) "
                      f"rows of dW x all K; {secs:.1f} s of FP64 CPU work"}


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    tensors = {k: wl.tensor(k) for k in wl.tensors}
    per_step = max(0.05, min(2.0, 90.0 / max(1, args.steps + args.warmup)))
    rng = np.random.default_rng(99)
    for _ in range(args.warmup):
        oracle_sample_step(wl, tensors, per_step, rng)
    tot_f, tot_s, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, s, desc = oracle_sample_step(wl, tensors, per_step, rng)
        tot_f += f
        tot_s += s
    import oracle
    value = tot_f / tot_s / 1e12
    line = {
        "impl": "reference", "metric": "grouped GEMM TFLOP/s (fwd/dgrad/wgrad), 1 GPU",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * wl.flops() / (value * 1e12),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(wl)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": f"each step: {desc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU path


def traffic_for(kernel: str, op_names):
    """Mean per-launch DRAM bytes of `kernel` over the given ops, from the
    committed ncu captures (profiles/traffic.json), if they were taken on the
    current source of that kernel and cover every op; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    ent = json.load(open(path)).get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, "moe_grouped_gemm_device_gb300", "csrc", KERNEL_SOURCES[kernel])
    if ent.get("source_sha256_16") != hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]:
        return None
    per_op = ent.get("per_op", {})
    if not op_names or any(o not in per_op for o in op_names):
        return None
    return sum(per_op[o] for o in op_names) // len(op_names)


def slowest_rank_ms(ms: float, dist, device) -> float:
    """The timed region's length on the slowest rank (max over ranks; the
    value itself with one process)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank runs the same per-GPU step (expert-shard
    replicas), so the job does world x the step's FLOPs per slowest step."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


class Unit:
    """One timed launch of the step: a grouped GEMM, or (MXFP8) the scale
    layout conversions that precede it."""

    def __init__(self, name, kernel, flops, nbytes, call, op=None):
        self.name, self.kernel, self.flops, self.bytes, self.call, self.op = name, kernel, flops, nbytes, call, op


def build_units(wl, rg, tensors, outs, off_ref, scratch):
    counts = wl.counts
    E, M = wl.E, wl.M
    units = []
    for op in wl.ops:
        if op.kind == "mx":
            KS = op.K // 32
            sa, sb = tensors[op.sa], tensors[op.sb]
            sab, sbb = scratch[op.name + ":sa"], scratch[op.name + ":sb"]
            woff = scratch["woff:" + str(op.N)]
            # the scale layout of both operands is converted every step (scales
            # change whenever activations or weights are re-quantized)
            conv_bytes = (M + E * op.N) * KS + sab.numel() + sbb.numel()

            def conv(op=op, sa=sa, sb=sb, sab=sab, sbb=sbb, woff=woff):
                rg.mx_scales_blocked(sa, off_ref[0], out=sab)
                rg.mx_scales_blocked(sb.view(-1, sb.shape[-1]), woff, out=sbb)
            units.append(Unit(op.name + ".scales", KERNEL_OF["mx_blocked"], 0, conv_bytes, conv))

            def gemm(op=op, sab=sab, sbb=sbb):
                rg.mgemm_mxfp8(tensors[op.a], sab, tensors[op.b], sbb, off_ref[0], transpose_B=op.transpose_B,
                               out=outs[op.name])
            units.append(Unit(op.name, kernel_of(op), op.flops(counts), algorithmic_bytes(op, counts), gemm, op))
            continue
        if op.kind == "mxk":
            sa, sb = tensors[op.sa], tensors[op.sb]
            sab, sbb = scratch[op.name + ":sa"], scratch[op.name + ":sb"]
            conv_bytes = (op.N + op.K) * (M // 32) + sab.numel() + sbb.numel()

            def conv(sa=sa, sb=sb, sab=sab, sbb=sbb):
                rg.mx_scales_blocked_k(sa, off_ref[0], out=sab)
                rg.mx_scales_blocked_k(sb, off_ref[0], out=sbb)
            units.append(Unit(op.name + ".scales", KERNEL_OF["mx_blocked_k"], 0, conv_bytes, conv))

            def wgrad(op=op, sab=sab, sbb=sbb):
                rg.kgemm_mxfp8(tensors[op.a], sab, tensors[op.b], sbb, off_ref[0], out=outs[op.name])
            units.append(Unit(op.name, kernel_of(op), op.flops(counts), algorithmic_bytes(op, counts), wgrad, op))
            continue

        def call(op=op):
            out = outs[op.name]
            if op.kind == "kgemm":
                rg.kgemm(tensors[op.a], tensors[op.b], off_ref[0], out=out, accumulate=op.accumulate)
            elif op.kind == "nested":
                rg.mgemm_nested(tensors[op.a], tensors[op.b], off_ref[0], transpose_B=op.transpose_B, out=out)
            elif op.fuse == "swiglu":
                rg.mgemm_swiglu(tensors[op.a], tensors[op.b], off_ref[0], out=out, y13=outs[op.name + ":y13"])
            elif op.fuse == "swiglu_bwd":
                rg.mgemm_swiglu_dgrad(tensors[op.a], tensors[op.b], off_ref[0], tensors[op.c], out=out)
            else:
                rg.mgemm(tensors[op.a], tensors[op.b], off_ref[0], transpose_B=op.transpose_B, out=out)
        units.append(Unit(op.name, kernel_of(op), op.flops(counts), algorithmic_bytes(op, counts), call, op))
    return units


def main():
    args = parse()
    wl = W.ALL[args.workload]()
    if args.ops:
        keep = args.ops.split(",")
        wl.ops = [o for o in wl.ops if o.name in keep]
        assert wl.ops, f"no op of {wl.name} matches {keep}"
        used = ({o.a for o in wl.ops} | {o.b for o in wl.ops} | {o.c for o in wl.ops if o.c}
                | {o.sa for o in wl.ops if o.sa} | {o.sb for o in wl.ops if o.sb})
        wl.tensors = {k: v for k, v in wl.tensors.items() if k in used}
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import moe_grouped_gemm_device_gb300 as rg
    sys.path.insert(0, os.path.join(ROOT, "tests"))

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rg.load()

    # ---- inputs: seeded on the host, then resident in HBM -------------------
    host = {k: wl.tensor(k) for k in wl.tensors}
    off_np = wl.offsets
    counts = wl.counts

    def as_torch(a):  # bf16 bit patterns (uint16) or FP8 / E8M0 codes (uint8)
        if a.dtype == np.uint8:
            return torch.from_numpy(a)
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)

    d = {k: as_torch(v).to(dev) for k, v in host.items()}
    off = torch.from_numpy(off_np).to(dev)
    is_mx = any(op.kind in ("mx", "mxk") for op in wl.ops)

    def make_buffers():
        """Output tensors of every op and the scale-layout buffers (MXFP8)."""
        outs, scratch = {}, {}
        for op in wl.ops:
            if op.kind in ("kgemm", "mxk"):
                # a main grad that steps accumulate into starts at zero
                alloc = torch.zeros if getattr(op, "accumulate", False) else torch.empty
                outs[op.name] = alloc((wl.E, op.N, op.K), dtype=torch.float32, device=dev)
            elif op.kind == "nested":
                outs[op.name] = torch.empty((wl.M, op.outer * op.N), dtype=torch.bfloat16, device=dev)
            elif op.fuse == "swiglu":
                outs[op.name] = torch.empty((wl.M, op.N // 2), dtype=torch.bfloat16, device=dev)
                outs[op.name + ":y13"] = torch.empty((wl.M, op.N), dtype=torch.bfloat16, device=dev)
            elif op.fuse == "swiglu_bwd":
                outs[op.name] = torch.empty((wl.M, 2 * op.N), dtype=torch.bfloat16, device=dev)
            else:
                outs[op.name] = torch.empty((wl.M, op.N), dtype=torch.bfloat16, device=dev)
            if op.kind == "mx":
                KS = op.K // 32
                scratch[op.name + ":sa"] = torch.empty((rg.mx_blocked_bytes(wl.M, KS, wl.E),), dtype=torch.uint8,
                                                       device=dev)
                scratch[op.name + ":sb"] = torch.empty((rg.mx_blocked_bytes(wl.E * op.N, KS, wl.E),),
                                                       dtype=torch.uint8, device=dev)
                scratch["woff:" + str(op.N)] = rg.mx_weight_offsets(wl.E, op.N, device=dev)
            if op.kind == "mxk":
                MS = wl.M // 32
                scratch[op.name + ":sa"] = torch.empty((rg.mx_blocked_k_bytes(op.N, MS, wl.E),),
                                                       dtype=torch.uint8, device=dev)
                scratch[op.name + ":sb"] = torch.empty((rg.mx_blocked_k_bytes(op.K, MS, wl.E),),
                                                       dtype=torch.uint8, device=dev)
        return outs, scratch

    outs, scratch = make_buffers()
    stream = torch.cuda.current_stream(dev)
    off_used = [off]
    units = build_units(wl, rg, d, outs, off_used, scratch)
    nu = len(units)

    def step(evs=None):
        for i, u in enumerate(units):
            if evs is not None:
                evs[i].record(stream)
            u.call()
        if evs is not None:
            evs[nu].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = rg.device_status()
    if status:
        raise SystemExit(f"device status {status:#x} after warm-up")

    # ---- timed region -------------------------------------------------------
    # Events around every launch, on the launching stream, give the per-kernel
    # durations of the timed steps themselves.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nu + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for s in range(args.steps):
        step(evs[s])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = evs[0][0].elapsed_time(evs[-1][nu])
    clocks = sampler.stop() if sampler else None
    status = rg.device_status()
    if status:
        raise SystemExit(f"device status {status:#x} after timed region")
    # [steps, units] launch durations; the mean feeds the throughput and the
    # roofline, the median and best decile (10th percentile of the duration)
    # describe the spread
    unit_ms = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(nu)] for e in evs])
    per_unit_ms = unit_ms.mean(axis=0)
    step_ms = unit_ms.sum(axis=1)
    ms = slowest_rank_ms(ms, dist, dev)
    ms_per_step = ms / args.steps
    flops_step = wl.flops()
    value = job_throughput(flops_step, ms_per_step, world)

    # ---- end to end through the public API with host buffers ---------------
    # Every step copies its inputs from pinned host memory, runs the ops and
    # copies every output back.  Consecutive steps are pipelined over two
    # device buffer sets: step i's host->device copies (one stream) overlap
    # step i-1's kernels (the compute stream) and step i-2's device->host
    # copies (a third stream); events order each buffer set's reuse.
    e2e = None
    if rank == 0 and args.e2e_steps > 0:
        pin = {k: as_torch(v).pin_memory() for k, v in host.items()}
        pin_off = torch.from_numpy(off_np).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in pin.values()) + pin_off.numel() * 4
        d1 = {k: torch.empty_like(v) for k, v in d.items()}
        off1 = [torch.empty_like(off)]
        outs1, scratch1 = make_buffers()
        sets = [(d, off_used, outs, units), (d1, off1, outs1, build_units(wl, rg, d1, outs1, off1, scratch1))]
        pin_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in o.items()} for _, _, o, _ in sets]
        d2h = sum(t.numel() * t.element_size() for t in pin_out[0].values())
        s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = [{n: torch.cuda.Event() for n in ("h2d", "comp", "d2h")} for _ in sets]
        started = [False, False]

        def e2e_step(i):
            b = i & 1
            dd, oo, outs_b, units_b = sets[b]
            e = ev[b]
            with torch.cuda.stream(s_h2d):
                if started[b]:
                    s_h2d.wait_event(e["comp"])  # step i-2's kernels are done with this input set
                for k, t in pin.items():
                    dd[k].copy_(t, non_blocking=True)
                oo[0].copy_(pin_off, non_blocking=True)
                e["h2d"].record(s_h2d)
            stream.wait_event(e["h2d"])
            if started[b]:
                stream.wait_event(e["d2h"])  # step i-2's outputs have left this set
            for u in units_b:
                u.call()
            e["comp"].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(e["comp"])
                for k, t in outs_b.items():
                    pin_out[b][k].copy_(t, non_blocking=True)
                e["d2h"].record(s_d2h)
            started[b] = True

        for i in range(2):  # warm both buffer sets
            e2e_step(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_h2d)
        for i in range(args.e2e_steps):
            e2e_step(i)
        stream.wait_stream(s_d2h)
        b.record(stream)
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(b) / args.e2e_steps
        e2e = {"value": flops_step / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms, "pipelined": "h2d / kernels / d2h of consecutive steps on three streams"}
        status = rg.device_status()
        if status:
            raise SystemExit(f"device status {status:#x} after the end-to-end steps")

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel ------------------------------------
    peaks, peak_src = load_peaks()
    per_kernel = {}
    per_op = {}
    for i, u in enumerate(units):
        ent = per_kernel.setdefault(u.kernel, {"ms": 0.0, "flops": 0, "bytes": 0, "launches": 0, "ops": []})
        ent["ms"] += per_unit_ms[i]
        ent["flops"] += u.flops
        ent["bytes"] += u.bytes
        ent["launches"] += 1
        ent["ops"].append(u.name)
        sec = per_unit_ms[i] * 1e-3
        med, p10 = float(np.median(unit_ms[:, i])), float(np.percentile(unit_ms[:, i], 10))
        rec = {"ms": round(float(per_unit_ms[i]), 4), "ms_median": round(med, 4), "ms_best_decile": round(p10, 4),
               "algorithmic_gbs": round(u.bytes / sec / 1e9, 1)}
        if u.flops:
            pk = tensor_peak(u.kernel, peaks)
            rec["tflops"] = round(u.flops / sec / 1e12, 1)
            rec["tflops_median"] = round(u.flops / (med * 1e-3) / 1e12, 1)
            rec["tflops_best_decile"] = round(u.flops / (p10 * 1e-3) / 1e12, 1)
            rec["pct_peak_sustained"] = round(100 * u.flops / sec / 1e12 / pk, 1)
        per_op[u.name] = rec
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms"])
    de = per_kernel[dom]
    traffic = traffic_for(dom, de["ops"])
    fp8 = dom in FP8_KERNELS
    peak = tensor_peak(dom, peaks)
    peak_name = ("measured bf16 sustained x 2 (nominal dense FP8/BF16 ratio 4.5/2.25; MEASURED_PEAKS.json)" if fp8
                 else "measured bf16 sustained (MEASURED_PEAKS.json)")
    # The kernel's bound: tensor cores when its arithmetic intensity is above
    # the ridge of the measured peaks, HBM below it (e.g. LoRA rank-16 GEMMs).
    ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if de["flops"] / de["bytes"] >= ridge:
        achieved = de["flops"] / (de["ms"] * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 4),
                    "peak_source": peak_name if peak_src == "measured" else "fallback 1.7 PFLOP/s sustained",
                    "frac_of_burst": round(achieved / (peaks["bf16_tflops"] * (2 if fp8 else 1)), 4)}
    else:
        achieved = de["bytes"] / (de["ms"] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_source": f"{peak_src} HBM copy (MEASURED_PEAKS.json)" if peak_src == "measured"
                    else "fallback 6.8 TB/s"}
    roofline.update({"traffic": traffic, "kernel": dom, "launches_per_step": de["launches"],
                     "algorithmic_flops_per_launch": de["flops"] // de["launches"],
                     "algorithmic_bytes_per_launch": de["bytes"] // de["launches"],
                     "share_of_step": round(de["ms"] / float(per_unit_ms.sum()), 3)})

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(wl, host, args.cpu_seconds)

    line = {
        "metric": "grouped GEMM TFLOP/s (fwd/dgrad/wgrad), 1 GPU",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "step_ms_median": round(float(np.median(step_ms)), 5),
        "step_ms_best_decile": round(float(np.percentile(step_ms, 10)), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 (MXFP8: E8M0 scale per 32)" if is_mx else "bf16",
        "data": "synthetic (seeded random E4M3 codes and E8M0 scales)" if is_mx
                else "synthetic (seeded normal inputs, random-init weights)",
        "config": {"workload": workload_desc(wl),
                   "flops_per_step": flops_step,
                   "l2": f"inputs larger than L2: step working set {working_set_bytes(wl) / 1e9:.2f} GB vs 129 MB L2",
                   "pct_of_peak_sustained": round(100 * value / world / peak, 1)},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": sum(2 if u.kernel in CONVERSION_KERNELS else 1 for u in units) * args.steps,
        "clocks": clocks,
        "per_op": per_op,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
