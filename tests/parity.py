"""Helpers shared by the GPU parity tests: moving seeded inputs to the device
and the tolerance checks.

Tolerances (from the specification of the grouped GEMM):
  * bf16 outputs: relative Frobenius error <= 4e-3 and, per element,
    |gpu - ref| <= 2e-2 * (|ref| + 1).  Rounding an exact result to bf16 alone
    gives a relative error <= 2^-9 per element (RMS about 1.1e-3).
  * fp32 dW: relative Frobenius error <= 1e-5 against the exact (FP64) result
    on the same bf16 inputs.  Products of bf16 values are exact in fp32, so the
    error is that of fp32 accumulation over at most one expert's rows.
"""
import json
import os

import numpy as np

import workloads as W

BF16_REL_FRO = 4e-3
BF16_ELEM = 2e-2
FP32_REL_FRO = 1e-5


def to_dev(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_host_bits(t) -> np.ndarray:
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def offsets_dev(off: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(off, dtype=np.int32)).to(device)


def rel_fro(g: np.ndarray, r: np.ndarray) -> float:
    nr = np.linalg.norm(r)
    ne = np.linalg.norm(g - r)
    return float(ne / nr) if nr > 0 else float(ne)


def _log(what: str, rec: dict) -> None:
    path = os.environ.get("RG_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": what, **rec}) + "\n")


def check_bf16(gpu_bits: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    g = W.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    fro = rel_fro(g, ref)
    err = np.abs(g - ref)
    worst = float(np.max(err / (np.abs(ref) + 1))) if err.size else 0.0
    _log(what, {"rel_fro": fro, "elem": worst, "tol_fro": BF16_REL_FRO, "tol_elem": BF16_ELEM})
    assert fro <= BF16_REL_FRO, f"{what}: relative Frobenius error {fro:.3e} > {BF16_REL_FRO}"
    assert worst <= BF16_ELEM, f"{what}: element error {worst:.3e}*(|ref|+1) > {BF16_ELEM}"
    return {"rel_fro": fro, "elem": worst}


def check_fp32(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> dict:
    g = np.asarray(gpu, dtype=np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    fro = rel_fro(g, ref)
    _log(what, {"rel_fro": fro, "tol_fro": FP32_REL_FRO})
    assert fro <= FP32_REL_FRO, f"{what}: relative Frobenius error {fro:.3e} > {FP32_REL_FRO}"
    return {"rel_fro": fro}


def bf16_round_exact(ref: np.ndarray) -> np.ndarray:
    """bf16 bits of exact values (round to nearest even) -- the result a
    correct fp32-accumulating kernel must produce when every partial sum is
    exactly representable."""
    return W.f32_to_bf16_bits(ref.astype(np.float32))


class FullCompare:
    """The checks of check_bf16 / check_fp32 over an output too large to hold
    twice in float64: fed chunk by chunk, it accumulates the squared error and
    reference norms (relative Frobenius error of the whole output) and, for
    bf16, the worst per-element error relative to |ref| + 1."""

    def __init__(self, kind: str, what: str):
        assert kind in ("bf16", "fp32")
        self.kind, self.what = kind, what
        self.err2 = 0.0
        self.ref2 = 0.0
        self.worst = 0.0
        self.count = 0

    def add(self, gpu: np.ndarray, ref: np.ndarray) -> None:
        g = (W.bf16_bits_to_f32(gpu) if self.kind == "bf16" else np.asarray(gpu)).astype(np.float64)
        assert g.shape == ref.shape, (g.shape, ref.shape)
        assert np.isfinite(g).all(), f"{self.what}: non-finite output"
        d = g - ref
        self.err2 += float(np.sum(d * d))
        self.ref2 += float(np.sum(ref * ref))
        if self.kind == "bf16" and d.size:
            self.worst = max(self.worst, float(np.max(np.abs(d) / (np.abs(ref) + 1))))
        self.count += d.size

    def finish(self) -> dict:
        fro = float(np.sqrt(self.err2 / self.ref2)) if self.ref2 > 0 else float(np.sqrt(self.err2))
        rec = {"rel_fro": fro, "elements": self.count}
        if self.kind == "bf16":
            rec["elem"] = self.worst
            _log(self.what, {**rec, "tol_fro": BF16_REL_FRO, "tol_elem": BF16_ELEM})
            assert fro <= BF16_REL_FRO, f"{self.what}: relative Frobenius error {fro:.3e} > {BF16_REL_FRO}"
            assert self.worst <= BF16_ELEM, f"{self.what}: element error {self.worst:.3e}*(|ref|+1) > {BF16_ELEM}"
        else:
            _log(self.what, {**rec, "tol_fro": FP32_REL_FRO})
            assert fro <= FP32_REL_FRO, f"{self.what}: relative Frobenius error {fro:.3e} > {FP32_REL_FRO}"
        return rec
