"""GPU parity at a large row count: M = 2^24 + 2^23 + 77 rows of 64 bf16
columns, so row offsets times the row pitch pass 2^31 bytes and every
address computation must be 64-bit.  The operands are zero except for a few
thousand seeded integer rows spread over the whole range (expert boundaries
and the last rows included); zero rows add nothing to either GEMM, so the
oracle runs on those rows alone, and integer inputs make the comparison
bit-exact."""
import numpy as np
import pytest

import oracle
import workloads as W
from parity import bf16_round_exact, offsets_dev, to_host_bits

pytestmark = pytest.mark.gpu

M = (1 << 24) + (1 << 23) + 77
K = 64
# three experts; the second one starts past 2^24 rows (2^31 bytes of x)
OFFSETS = np.array([0, (1 << 24) + 5, (1 << 24) + 300, M - 3], dtype=np.int32)


def sparse_rows(seed, n_random=3000):
    rng = np.random.default_rng(seed)
    picks = [rng.integers(0, M, size=n_random)]
    for b in OFFSETS:
        picks.append(np.arange(max(0, int(b) - 3), min(M, int(b) + 3)))
    picks.append(np.arange(M - 8, M))
    return np.unique(np.concatenate(picks))


def host_dev_sparse(rows, cols, seed, stream):
    """Device bf16 [M, cols] holding integer rows at `rows`, zeros elsewhere,
    and the host copy of those rows."""
    import torch
    vals = W.integer_bf16((len(rows), cols), -2, 2, seed, stream)
    d = torch.zeros((M, cols), dtype=torch.int16, device="cuda")
    d[torch.from_numpy(rows).cuda()] = torch.from_numpy(vals.view(np.int16)).cuda()
    return vals, d.view(torch.bfloat16)


def test_mgemm_large_m_bit_exact(gpu_lib):
    import torch
    E, N = len(OFFSETS) - 1, 256
    rows = sparse_rows(21)
    xv, x = host_dev_sparse(rows, K, 21, 0)
    w = W.integer_bf16((E, N, K), -2, 2, 21, 1)
    y = gpu_lib.mgemm(x, torch.from_numpy(w.view(np.int16)).cuda().view(torch.bfloat16),
                      offsets_dev(OFFSETS))
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    # the sampled rows inside some expert, compared with the oracle on the
    # same rows; a zero row of x gives a zero row of y
    inside = rows[rows < OFFSETS[-1]]
    got = to_host_bits(y[torch.from_numpy(inside).cuda()])
    x_rows = np.zeros((M, K), dtype=np.uint16)
    x_rows[rows] = xv
    ref = oracle.mgemm(x_rows, w, OFFSETS, rows=inside)
    np.testing.assert_array_equal(got, bf16_round_exact(ref))
    zero_row = int(np.setdiff1d(np.arange(M - 100000, M - 10), rows)[0])
    assert (W.bf16_bits_to_f32(to_host_bits(y[zero_row:zero_row + 1])) == 0).all()


def test_kgemm_large_m_bit_exact(gpu_lib):
    import torch
    E, N = len(OFFSETS) - 1, 64
    rows = sparse_rows(22)
    gv, g = host_dev_sparse(rows, N, 22, 0)
    xv, x = host_dev_sparse(rows, K, 22, 1)
    dW = gpu_lib.kgemm(g, x, offsets_dev(OFFSETS))
    torch.cuda.synchronize()
    assert gpu_lib.device_status() == 0
    # the same sums over the nonzero rows only: offsets counted in that subset
    keep = rows < OFFSETS[-1]
    sub_off = np.searchsorted(rows[keep], OFFSETS).astype(np.int32)
    ref = oracle.kgemm(gv[keep], xv[keep], sub_off)
    np.testing.assert_array_equal(dW.cpu().numpy().astype(np.float64), ref)
