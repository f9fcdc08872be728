"""Run MXFP8 Mgemm cases through a library built with CTA pairs for the
block-scaled GEMM (RG_MX_PAIR=1, with the debug-bounds checks on) and check
them against the oracle: integer codes bit for bit (forward and input
gradient, experts whose last pair tile leaves the second CTA without rows or
with a few, an output-column tail and a contraction tail), random codes
within the bf16 tolerance, many small experts, and rows past offsets[E] left
untouched.

    python tests/mx_pair_cases.py PATH/TO/librg.so

Run in a process of its own: the binding loads one library per process.
"""
import os
import sys
import zlib

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as W  # noqa: E402
from parity import bf16_round_exact, check_bf16, offsets_dev, to_host_bits  # noqa: E402

SENTINEL_BF16 = 0x4640


def int_codes(shape, seed, stream):
    """E4M3 codes of integers in {-2..2}."""
    e4, _ = oracle.mx_decode_tables()
    table = np.array([int(np.flatnonzero(e4 == v)[0]) for v in (-2.0, -1.0, 0.0, 1.0, 2.0)], dtype=np.uint8)
    rng = np.random.default_rng(np.random.SeedSequence([seed, stream]))
    return table[rng.integers(0, 5, size=shape)]


def main(lib_path):
    import torch
    from moe_grouped_gemm_device_gb300 import _build
    _build.LIB = lib_path
    import moe_grouped_gemm_device_gb300 as rg
    rg.load()
    n_cases = 0

    def run(xq, sx, wq, sw, off, tB):
        E = len(off) - 1
        M = xq.shape[0]
        N = wq.shape[2] if tB else wq.shape[1]
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        sxb = rg.mx_scales_blocked(dev(sx), offsets_dev(off))
        swb = rg.mx_scales_blocked(dev(sw.reshape(E * N, -1)), rg.mx_weight_offsets(E, N))
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        y.view(torch.int16).fill_(SENTINEL_BF16)
        rg.mgemm_mxfp8(dev(xq), sxb, dev(wq), swb, offsets_dev(off), transpose_B=tB, out=y)
        torch.cuda.synchronize()
        st = rg.device_status()
        assert st == 0, f"device status {st:#x}"
        got = to_host_bits(y)
        valid = int(off[-1])
        assert (got[valid:] == SENTINEL_BF16).all(), "rows past offsets[E] were written"
        return got[:valid], oracle.mgemm_mx(xq, sx, wq, sw, off, transpose_B=tB)[:valid]

    # integer codes, scales 1/2..2: exact partial sums, bit-exact bf16
    for counts, N, K in [([600, 0, 300, 130, 1, 37], 512, 256), ([129, 256, 255, 3], 400, 320)]:
        off = W.offsets_from_counts(counts)
        E, M = len(counts), int(off[-1]) + 5
        for tB in (False, True):
            xq = int_codes((M, K), 81, 0)
            wq = int_codes((E, K, N) if tB else (E, N, K), 81, 1)
            sx = W.e8m0_codes((M, K // 32), 126, 128, 81, 2)
            sw = W.e8m0_codes((E, N, K // 32), 126, 128, 81, 3)
            got, ref = run(xq, sx, wq, sw, off, tB)
            bad = int((got != bf16_round_exact(ref)).sum())
            print(f"integer counts={counts} N={N} K={K} tB={tB}: {bad} mismatches", flush=True)
            assert bad == 0
            n_cases += 1
    # random codes at realistic scales
    for E, N, K, total in [(7, 640, 544, 3000), (2, 1296, 1024, 900), (3, 16, 32, 200), (300, 256, 128, 6000)]:
        rng = np.random.default_rng(zlib.crc32(f"mxpair/{E}/{N}/{K}".encode()))
        counts = rng.multinomial(total, [1 / E] * E)
        counts[0] = 0
        off = W.offsets_from_counts(counts)
        M = int(off[-1]) + 3
        s = int(rng.integers(1 << 20))
        for tB in (False, True):
            xq = W.e4m3_codes((M, K), s, 0)
            wq = W.e4m3_codes((E, K, N) if tB else (E, N, K), s, 1)
            sx = W.e8m0_codes((M, K // 32), *W.MX_ACT_SCALES, s, 2)
            sw = W.e8m0_codes((E, N, K // 32), *W.mx_weight_scales(K), s, 3)
            got, ref = run(xq, sx, wq, sw, off, tB)
            check_bf16(got, ref, f"mx pair E={E} N={N} K={K} tB={tB}")
            print(f"random E={E} N={N} K={K} tB={tB}: ok", flush=True)
            n_cases += 1
    print(f"ALL OK {n_cases} cases", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
