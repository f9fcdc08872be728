"""Seeded synthetic inputs for the MoE grouped GEMM workloads.

This module only draws numbers: per-expert row counts, the cumulative
row-offset vector built from them, and bf16 operand tensors.  It holds none
of the grouped-GEMM arithmetic, so both the CPU oracle (``oracle/``) and the
CUDA path (``moe_grouped_gemm_device_gb300``) can take their inputs from it
without sharing any of the method's code.

Conventions:

* Offsets are int32 ``[E+1]`` with a leading zero: expert ``e`` owns rows
  ``offsets[e] .. offsets[e+1]-1`` (RapidGEMM README, "Kernels": ``cnt`` is
  the cumulative row-offset tensor with a leading zero).
* ``N(0, v)`` in a workload description means variance ``v``: weights of a
  layer whose contraction length is ``K`` are drawn with std ``1/sqrt(K)``.
* Random numbers come from numpy's PCG64.  A tensor is filled in fixed-size
  chunks, chunk ``i`` from ``SeedSequence([seed, stream, i])``, so the values
  do not depend on how many threads generate them.  FP32 normals are rounded
  to bf16 with round-to-nearest-even.
* bf16 tensors are returned as ``np.uint16`` bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 22  # elements per independently seeded chunk

# --------------------------------------------------------------------------
# bf16 bit helpers (number representation only)
# --------------------------------------------------------------------------


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# Seeded tensor fills
# --------------------------------------------------------------------------

_POOL: ThreadPoolExecutor | None = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def normal_bf16(shape, std: float, seed: int, stream: int) -> np.ndarray:
    """bf16 bits of N(0, std^2) values of the given shape."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)
    std32 = np.float32(std)

    def fill(i: int) -> None:
        lo = i * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.default_rng(np.random.SeedSequence([seed, stream, i]))
        v = rng.standard_normal(hi - lo, dtype=np.float32)
        if std32 != np.float32(1.0):
            v *= std32
        out[lo:hi] = f32_to_bf16_bits(v)

    nchunks = (n + CHUNK - 1) // CHUNK
    if nchunks <= 1:
        if n:
            fill(0)
    else:
        list(_pool().map(fill, range(nchunks)))
    return out.reshape(shape)


def integer_bf16(shape, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    """bf16 bits of integers drawn uniformly from [lo, hi] (exact in bf16)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, stream]))
    v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(v)


def e4m3_codes(shape, seed: int, stream: int) -> np.ndarray:
    """Random FP8 E4M3 codes (uint8): sign, exponent field and mantissa field
    drawn uniformly (exponent field 4..15), the NaN code S.1111.111 redrawn as
    S.1111.110.  No value is rounded: the codes are the random draw."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint8)

    def fill(i: int) -> None:
        lo = i * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.default_rng(np.random.SeedSequence([seed, stream, i]))
        sign = rng.integers(0, 2, size=hi - lo, dtype=np.uint8) << np.uint8(7)
        expo = rng.integers(4, 16, size=hi - lo, dtype=np.uint8) << np.uint8(3)
        mant = rng.integers(0, 8, size=hi - lo, dtype=np.uint8)
        c = sign | expo | mant
        c[(c & np.uint8(0x7F)) == np.uint8(0x7F)] -= np.uint8(1)
        out[lo:hi] = c

    nchunks = (n + CHUNK - 1) // CHUNK
    if nchunks <= 1:
        if n:
            fill(0)
    else:
        list(_pool().map(fill, range(nchunks)))
    return out.reshape(shape)


def e8m0_codes(shape, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    """Random E8M0 scale codes (uint8) drawn uniformly from [lo, hi]."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, stream]))
    return rng.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.uint8)


# RMS of the values of e4m3_codes is about 119 (2^6.9): scale codes around
# 120 (2^-7) give activations of RMS ~1, and 120 - log2(sqrt(K)) weights of
# RMS ~1/sqrt(K), the magnitudes of the bf16 workloads.
MX_ACT_SCALES = (119, 121)


def mx_weight_scales(K: int) -> tuple:
    c = 120 - int(round(np.log2(np.sqrt(K))))
    return (c - 1, c + 1)


# --------------------------------------------------------------------------
# Row counts and offsets
# --------------------------------------------------------------------------


def offsets_from_counts(counts) -> np.ndarray:
    counts = np.asarray(counts, dtype=np.int64)
    assert (counts >= 0).all()
    off = np.zeros(len(counts) + 1, dtype=np.int64)
    np.cumsum(counts, out=off[1:])
    assert off[-1] < 2**31
    return off.astype(np.int32)


def counts_tiny(seed: int = 0) -> np.ndarray:
    """E=4, M=512: multinomial over experts 0, 1, 3 with expert 2 empty.

    A draw in which some count is a multiple of 128 is replaced by the next
    draw of the same generator, so every tile boundary is ragged.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0]))
    while True:
        c3 = rng.multinomial(512, [1 / 3] * 3)
        if all(c % 128 != 0 for c in c3):
            break
    return np.array([c3[0], c3[1], 0, c3[2]], dtype=np.int64)


def counts_dirichlet(E: int, M: int, alpha: float, seed: int) -> np.ndarray:
    """Dirichlet(alpha) shares rounded to integers that sum to M.

    floor(M*p), then one extra row to each of the largest fractional parts
    (ties to the lower expert index) until the sum is M.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0]))
    p = rng.dirichlet([alpha] * E)
    raw = M * p
    base = np.floor(raw).astype(np.int64)
    rem = int(M - base.sum())
    frac = raw - base
    order = np.lexsort((np.arange(E), -frac))
    base[order[:rem]] += 1
    assert base.sum() == M
    return base


def counts_zipf(E: int, M: int, s: float, seed: int, tail: bool = False) -> np.ndarray:
    """Truncated Zipf(s) over a seeded permutation of the experts.

    Rank r (1..E) has probability proportional to r**-s; expert perm[r-1]
    gets rank r; counts are a multinomial(M) draw.  With ``tail=True`` the 32
    lowest-probability ranks instead get Uniform{0..7} rows, the 4 lowest of
    them none at all, and rank 1 absorbs the difference so the sum stays M.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0]))
    perm = rng.permutation(E)
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p_rank = ranks ** (-s)
    p_rank /= p_rank.sum()
    c_rank = rng.multinomial(M, p_rank).astype(np.int64)
    if tail:
        trng = np.random.default_rng(np.random.SeedSequence([seed, 1]))
        ntail = min(32, E - 1)
        c_rank[E - ntail:] = trng.integers(0, 8, size=ntail)
        c_rank[E - min(4, ntail):] = 0
        c_rank[0] += M - c_rank.sum()
        assert c_rank[0] >= 0
    counts = np.zeros(E, dtype=np.int64)
    counts[perm] = c_rank
    assert counts.sum() == M
    return counts


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------


@dataclass
class Op:
    """One grouped-GEMM call.

    kind 'mgemm': y[M,N] from a=x[M,K] and b=w ([E,N,K], or [E,K,N] when
    transpose_B).  kind 'kgemm': dW[E,N,K] fp32 from a=grad[M,N], b=X[M,K].
    ``a`` and ``b`` name tensors of the owning workload.
    """

    name: str
    kind: str
    a: str
    b: str
    N: int
    K: int
    transpose_B: bool = False
    # "" (plain GEMM), "swiglu" (forward gate-up with SwiGLU in the epilogue:
    # writes h [M, N/2] and y13 [M, N]) or "swiglu_bwd" (input gradient of the
    # down projection followed by the SwiGLU backward; ``c`` names the saved
    # y13 [M, 2N] it reads, and it writes dy13 [M, 2N])
    fuse: str = ""
    c: str = ""
    # kind 'nested': O outer groups over the columns (a = x [M, O*K], b = w
    # [O, L, N, K], output [M, O*N])
    outer: int = 1
    # kind 'mx': MXFP8 Mgemm; a, b are E4M3 code tensors, sa [M, K/32] and sb
    # [E, N, K/32] their E8M0 scale tensors.  kind 'mxk': MXFP8 Kgemm; a =
    # grad [M, N], b = X [M, K] E4M3 codes, sa [N, M/32] and sb [K, M/32]
    sa: str = ""
    sb: str = ""
    # kind 'kgemm': add dW to the existing FP32 output (main grad) instead of
    # overwriting it
    accumulate: bool = False

    def flops(self, counts) -> int:
        return 2 * int(np.sum(counts)) * self.outer * self.N * self.K


@dataclass
class Workload:
    name: str
    seed: int
    E: int
    M: int
    counts: np.ndarray
    tensors: dict = field(default_factory=dict)  # name -> (shape, std, stream)
    ops: list = field(default_factory=list)

    @property
    def offsets(self) -> np.ndarray:
        return offsets_from_counts(self.counts)

    def tensor(self, name: str) -> np.ndarray:
        shape, std, stream = self.tensors[name]
        if std == "e4m3":
            return e4m3_codes(shape, self.seed, stream)
        if isinstance(std, tuple) and std[0] == "e8m0":
            return e8m0_codes(shape, std[1], std[2], self.seed, stream)
        return normal_bf16(shape, std, self.seed, stream)

    def op(self, name: str) -> Op:
        for o in self.ops:
            if o.name == name:
                return o
        raise KeyError(name)

    def flops(self) -> int:
        return sum(o.flops(self.counts) for o in self.ops)


def _layer(name, seed, E, M, counts, d_model, d_ffn2, d_ffn):
    """An MoE expert layer: gate-up [M,d_model]x[E,d_ffn2,d_model]^T, down
    [M,d_ffn]x[E,d_model,d_ffn]^T, their input gradients and FP32 weight
    gradients.  Activations and gradients ~N(0,1), weights ~N(0,1/K)."""
    w = Workload(name, seed, E, M, counts)
    w.tensors = {
        "x": ((M, d_model), 1.0, 1),
        "w13": ((E, d_ffn2, d_model), 1.0 / np.sqrt(d_model), 2),
        "h": ((M, d_ffn), 1.0, 3),
        "w2": ((E, d_model, d_ffn), 1.0 / np.sqrt(d_ffn), 4),
        "dy13": ((M, d_ffn2), 1.0, 5),
        "dy2": ((M, d_model), 1.0, 6),
    }
    w.ops = [
        Op("fwd_gate_up", "mgemm", "x", "w13", N=d_ffn2, K=d_model),
        Op("fwd_down", "mgemm", "h", "w2", N=d_model, K=d_ffn),
        Op("dgrad_down", "mgemm", "dy2", "w2", N=d_ffn, K=d_model, transpose_B=True),
        Op("dgrad_gate_up", "mgemm", "dy13", "w13", N=d_model, K=d_ffn2, transpose_B=True),
        Op("wgrad_gw2", "kgemm", "dy2", "h", N=d_model, K=d_ffn),
        Op("wgrad_gw13", "kgemm", "dy13", "x", N=d_ffn2, K=d_model),
    ]
    return w


def with_swiglu(w: Workload) -> Workload:
    """The same layer with the SwiGLU activation fused into its GEMMs: the
    gate-up forward also applies SwiGLU (h = SiLU(gate) * up), and the
    down projection's input gradient also applies the SwiGLU backward to a
    saved gate-up output y13 ~N(0,1).  GEMM shapes and FLOPs are unchanged."""
    import copy
    f = copy.deepcopy(w)
    f.name = w.name + "_swiglu"
    d_ffn2 = w.op("fwd_gate_up").N
    f.tensors["y13"] = ((w.M, d_ffn2), 1.0, 7)
    ops = []
    for o in w.ops:
        if o.name == "fwd_gate_up":
            o = Op("fwd_gate_up_swiglu", "mgemm", o.a, o.b, N=o.N, K=o.K, fuse="swiglu")
        elif o.name == "dgrad_down":
            o = Op("dgrad_down_swiglu", "mgemm", o.a, o.b, N=o.N, K=o.K, transpose_B=True,
                   fuse="swiglu_bwd", c="y13")
        ops.append(o)
    f.ops = ops
    return f


def with_wgrad_accumulation(w: Workload) -> Workload:
    """The same layer with both weight gradients added to an existing FP32
    main grad (fused wgrad accumulation) instead of overwriting dW."""
    import copy
    f = copy.deepcopy(w)
    f.name = w.name + "_acc"
    f.ops = [Op(o.name + "_acc", o.kind, o.a, o.b, N=o.N, K=o.K, accumulate=True) if o.kind == "kgemm" else o
             for o in w.ops]
    return f


def tiny() -> Workload:
    """E=4, K=256, N=128, M=512, expert 2 empty (seed 0)."""
    c = counts_tiny(0)
    w = Workload("tiny_E4_M512_N128_K256", 0, 4, 512, c)
    w.tensors = {
        "x": ((512, 256), 1.0, 1),
        "w": ((4, 128, 256), 1.0 / 16.0, 2),
        "grad": ((512, 128), 1.0, 3),
    }
    w.ops = [
        Op("fwd", "mgemm", "x", "w", N=128, K=256),
        Op("dgrad", "mgemm", "grad", "w", N=256, K=128, transpose_B=True),
        Op("wgrad", "kgemm", "grad", "x", N=128, K=256),
    ]
    return w


def uniform(g: int, m: int) -> Workload:
    """g groups of m rows each, n=768, k=2048, forward only (seed 2)."""
    c = np.full(g, m, dtype=np.int64)
    w = Workload(f"uniform_g{g}_m{m}_n768_k2048", 2, g, g * m, c)
    stream0 = 10 * g
    w.tensors = {
        "x": ((g * m, 2048), 1.0, stream0 + 1),
        "w": ((g, 768, 2048), 1.0 / np.sqrt(2048), stream0 + 2),
    }
    w.ops = [Op("fwd", "mgemm", "x", "w", N=768, K=2048)]
    return w


def a3b_layer() -> Workload:
    """30B-A3B expert layer on one GPU: 32 local experts, 32768 routed rows,
    Dirichlet(2) counts, d_model 3072, expert FFN 1280 (seed 3)."""
    c = counts_dirichlet(32, 32768, 2.0, 3)
    return _layer("a3b_E32_M32768", 3, 32, 32768, c, 3072, 2560, 1280)


def skewed(tail: bool = False) -> Workload:
    """128 experts, 65536 rows, Zipf(1.2) counts over a seeded permutation
    (seed 5); ``tail`` adds the tiny/empty-expert tail."""
    c = counts_zipf(128, 65536, 1.2, 5, tail=tail)
    name = "skewed_zipf_tail_E128_M65536" if tail else "skewed_zipf_E128_M65536"
    return _layer(name, 5, 128, 65536, c, 3072, 2560, 1280)


def a3b_mxfp8() -> Workload:
    """The 30B-A3B expert layer's six grouped GEMMs in MXFP8: E4M3 operands
    with one E8M0 scale per 32 elements along each contraction (seed 3,
    Dirichlet(2) shares over 32 experts, M = 32768, every expert a whole
    number of 32-row blocks so that the weight gradient's row-wise scale
    blocks never straddle two experts).  The weights carry one scale tensor per direction (row-wise
    for the forward, column-wise for the input gradient), as a training step
    that quantizes each weight once per GEMM direction would hold.  Codes and
    scales are random draws; scales put activations at RMS ~1 and weights at
    RMS ~1/sqrt(K), like the bf16 layer."""
    # expert row counts in whole 32-row scale blocks: Dirichlet(2) shares of
    # the 1024 blocks of 32 rows
    c = counts_dirichlet(32, 1024, 2.0, 3) * 32
    E, M, dm, d2, d1 = 32, 32768, 3072, 2560, 1280
    act = ("e8m0",) + MX_ACT_SCALES

    def wsc(K):
        return ("e8m0",) + mx_weight_scales(K)

    w = Workload("a3b_mxfp8_E32_M32768", 3, E, M, c)
    w.tensors = {
        "xq": ((M, dm), "e4m3", 21), "sx": ((M, dm // 32), act, 22),
        "w13q": ((E, d2, dm), "e4m3", 23), "sw13": ((E, d2, dm // 32), wsc(dm), 24),
        "hq": ((M, d1), "e4m3", 25), "sh": ((M, d1 // 32), act, 26),
        "w2q": ((E, dm, d1), "e4m3", 27), "sw2": ((E, dm, d1 // 32), wsc(d1), 28),
        "dy2q": ((M, dm), "e4m3", 29), "sdy2": ((M, dm // 32), act, 30),
        "sw2t": ((E, d1, dm // 32), wsc(dm), 31),
        "dy13q": ((M, d2), "e4m3", 32), "sdy13": ((M, d2 // 32), act, 33),
        "sw13t": ((E, dm, d2 // 32), wsc(d2), 34),
        # column-wise scales (one per column and 32-row block) for the wgrad
        "sdy2c": ((dm, M // 32), act, 35), "shc": ((d1, M // 32), act, 36),
        "sdy13c": ((d2, M // 32), act, 37), "sxc": ((dm, M // 32), act, 38),
    }
    w.ops = [
        Op("mx_fwd_gate_up", "mx", "xq", "w13q", N=d2, K=dm, sa="sx", sb="sw13"),
        Op("mx_fwd_down", "mx", "hq", "w2q", N=dm, K=d1, sa="sh", sb="sw2"),
        Op("mx_dgrad_down", "mx", "dy2q", "w2q", N=d1, K=dm, transpose_B=True, sa="sdy2", sb="sw2t"),
        Op("mx_dgrad_gate_up", "mx", "dy13q", "w13q", N=dm, K=d2, transpose_B=True, sa="sdy13", sb="sw13t"),
        Op("mx_wgrad_gw2", "mxk", "dy2q", "hq", N=dm, K=d1, sa="sdy2c", sb="shc"),
        Op("mx_wgrad_gw13", "mxk", "dy13q", "xq", N=d2, K=dm, sa="sdy13c", sb="sxc"),
    ]
    return w


def lora_a3b(adapters: int = 4, rank: int = 16) -> Workload:
    """Batched LoRA over the 30B-A3B expert layer's gate-up projection (the
    nested grouped GEMM of CUTLASS discussion #1452): the a3b routed rows
    (seed 3) are split over `adapters` LoRA adapters per expert (a seeded
    multinomial with equal shares) and ordered (adapter, expert), giving
    L = adapters * 32 inner row groups.

      lora_shrink  s = x . A[l]^T     x [M, 3072], A [1, L, 2r, 3072] (gate
                                      and up adapters' A stacked): N = 2r
      lora_expand  y[:, o*1280:] = s[:, o*r:] . B[o, l]^T for o = gate, up:
                                      s [M, 2r], B [2, L, 1280, r]: O = 2

    All values ~N(0,1) except weights ~N(0, 1/K)."""
    base = counts_dirichlet(32, 32768, 2.0, 3)
    rng = np.random.default_rng(np.random.SeedSequence([3, 2]))
    split = np.stack([rng.multinomial(int(c), [1.0 / adapters] * adapters) for c in base], axis=1)
    counts = split.reshape(-1).astype(np.int64)  # index = adapter * 32 + expert
    L, M, d_model, d_half = adapters * 32, 32768, 3072, 1280
    w = Workload(f"lora_a3b_A{adapters}_r{rank}_L{L}_M{M}", 3, L, M, counts)
    w.tensors = {
        "x": ((M, d_model), 1.0, 1),
        "lora_a": ((1, L, 2 * rank, d_model), 1.0 / np.sqrt(d_model), 11),
        "s": ((M, 2 * rank), 1.0, 12),
        "lora_b": ((2, L, d_half, rank), 1.0 / np.sqrt(rank), 13),
    }
    w.ops = [
        Op("lora_shrink", "nested", "x", "lora_a", N=2 * rank, K=d_model, outer=1),
        Op("lora_expand", "nested", "s", "lora_b", N=d_half, K=rank, outer=2),
    ]
    return w


ALL = {
    "tiny": tiny,
    "uniform8": lambda: uniform(8, 4096),
    "uniform16": lambda: uniform(16, 2048),
    "a3b": a3b_layer,
    "skewed": lambda: skewed(False),
    "skewed_tail": lambda: skewed(True),
    "a3b_swiglu": lambda: with_swiglu(a3b_layer()),
    "a3b_acc": lambda: with_wgrad_accumulation(a3b_layer()),
    "skewed_tail_swiglu": lambda: with_swiglu(skewed(True)),
    "lora_a3b": lora_a3b,
    "a3b_mxfp8": a3b_mxfp8,
}
