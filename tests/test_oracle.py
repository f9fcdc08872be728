"""Pins for the CPU oracle (no GPU).

The oracle is trusted only because these tests tie it to things other than
itself: hand-worked values, an independent brute-force loop, ordinary GEMMs
from numpy, exact integer arithmetic and invariants of the definitions
(RapidGEMM README, "Kernels": Mgemm for forward / input gradient, Kgemm for
the FP32 weight gradient, both over a cumulative row-offset vector with a
leading zero).
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(a):
    """Exact bf16 bit patterns of small integers / bf16-representable values."""
    return W.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def rand_bits(rng, shape, scale=1.0):
    return W.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


def f64(b):
    return W.bf16_bits_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------- hand-worked


def test_golden_handworked_fwd():
    g = json.load(open(os.path.join(GOLDEN, "handworked_e3.json")))
    off = np.array(g["offsets"], dtype=np.int32)
    f = g["fwd"]
    y = oracle.mgemm(bits(f["x"]), bits(f["w"]), off)
    np.testing.assert_array_equal(y[:3], np.array(f["y_rows_0_to_2"], dtype=np.float64))
    assert np.isnan(y[3]).all()  # row 3 belongs to no expert


def test_golden_handworked_dgrad():
    g = json.load(open(os.path.join(GOLDEN, "handworked_e3.json")))
    off = np.array(g["offsets"], dtype=np.int32)
    d = g["dgrad"]
    y = oracle.mgemm(bits(d["x"]), bits(d["w"]), off, transpose_B=True)
    np.testing.assert_array_equal(y[:3], np.array(d["y_rows_0_to_2"], dtype=np.float64))


def test_golden_handworked_wgrad():
    g = json.load(open(os.path.join(GOLDEN, "handworked_e3.json")))
    off = np.array(g["offsets"], dtype=np.int32)
    d = g["wgrad"]
    dW = oracle.kgemm(bits(d["grad"]), bits(d["X"]), off)
    np.testing.assert_array_equal(dW, np.array(d["dW"], dtype=np.float64))


# ---------------------------------------------------------------- brute force


def brute_mgemm(x, w, offsets, transpose_B):
    """Independent pure-Python triple loop over plain lists."""
    M, K = len(x), len(x[0])
    E = len(offsets) - 1
    N = len(w[0][0]) if transpose_B else len(w[0])
    y = [[None] * N for _ in range(M)]
    for e in range(E):
        for r in range(offsets[e], offsets[e + 1]):
            for n in range(N):
                s = 0.0
                for k in range(K):
                    b = w[e][k][n] if transpose_B else w[e][n][k]
                    s += x[r][k] * b
                y[r][n] = s
    return y


def brute_kgemm(grad, X, offsets):
    N, K = len(grad[0]), len(X[0])
    E = len(offsets) - 1
    dW = [[[0.0] * K for _ in range(N)] for _ in range(E)]
    for e in range(E):
        for n in range(N):
            for k in range(K):
                s = 0.0
                for r in range(offsets[e], offsets[e + 1]):
                    s += grad[r][n] * X[r][k]
                dW[e][n][k] = s
    return dW


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("transpose_B", [False, True])
def test_mgemm_matches_brute_force(seed, transpose_B):
    rng = np.random.default_rng(seed)
    E = 3
    M = int(rng.integers(4, 13))
    N = int(rng.integers(1, 8))
    K = int(rng.integers(1, 8))
    counts = rng.multinomial(M - 2, [0.5, 0.0, 0.5])  # expert 1 empty, 2 rows past offsets[E]
    off = W.offsets_from_counts(counts)
    x = rand_bits(rng, (M, K))
    w = rand_bits(rng, (E, K, N) if transpose_B else (E, N, K))
    y = oracle.mgemm(x, w, off, transpose_B=transpose_B)
    ref = brute_mgemm(f64(x).tolist(), f64(w).tolist(), off.tolist(), transpose_B)
    for r in range(M):
        if ref[r][0] is None:
            assert np.isnan(y[r]).all()
        else:
            np.testing.assert_array_equal(y[r], np.array(ref[r]))


@pytest.mark.parametrize("seed", range(6))
def test_kgemm_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    E = 3
    M = int(rng.integers(4, 13))
    N = int(rng.integers(1, 8))
    K = int(rng.integers(1, 8))
    counts = rng.multinomial(M - 1, [0.3, 0.0, 0.7])
    off = W.offsets_from_counts(counts)
    grad = rand_bits(rng, (M, N))
    X = rand_bits(rng, (M, K))
    dW = oracle.kgemm(grad, X, off)
    ref = np.array(brute_kgemm(f64(grad).tolist(), f64(X).tolist(), off.tolist()))
    np.testing.assert_array_equal(dW, ref)


# ---------------------------------------------------------------- ordinary GEMMs


def test_single_group_is_ordinary_gemm():
    rng = np.random.default_rng(7)
    M, N, K = 37, 19, 53
    x = rand_bits(rng, (M, K))
    w = rand_bits(rng, (1, N, K))
    off = np.array([0, M], dtype=np.int32)
    y = oracle.mgemm(x, w, off)
    np.testing.assert_allclose(y, f64(x) @ f64(w[0]).T, rtol=1e-12, atol=1e-12)
    wt = rand_bits(rng, (1, K, N))
    yt = oracle.mgemm(x, wt, off, transpose_B=True)
    np.testing.assert_allclose(yt, f64(x) @ f64(wt[0]), rtol=1e-12, atol=1e-12)
    grad = rand_bits(rng, (M, N))
    dW = oracle.kgemm(grad, x, off)
    np.testing.assert_allclose(dW[0], f64(grad).T @ f64(x), rtol=1e-12, atol=1e-12)


def test_integer_inputs_are_exact():
    """Integers in {-2..2}: every partial sum is an exact integer, so the
    result must equal numpy's int64 GEMM per group exactly."""
    rng = np.random.default_rng(11)
    E, N, K = 4, 24, 300
    counts = np.array([130, 0, 1, 97])
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + 5
    xi = rng.integers(-2, 3, size=(M, K))
    wi = rng.integers(-2, 3, size=(E, N, K))
    gi = rng.integers(-2, 3, size=(M, N))
    y = oracle.mgemm(bits(xi), bits(wi), off)
    yt = oracle.mgemm(bits(xi), bits(wi.transpose(0, 2, 1).copy()), off, transpose_B=True)
    dW = oracle.kgemm(bits(gi), bits(xi), off)
    for e in range(E):
        a, b = off[e], off[e + 1]
        ref = xi[a:b] @ wi[e].T
        np.testing.assert_array_equal(y[a:b], ref.astype(np.float64))
        np.testing.assert_array_equal(yt[a:b], ref.astype(np.float64))
        np.testing.assert_array_equal(dW[e], (gi[a:b].T @ xi[a:b]).astype(np.float64))


# ---------------------------------------------------------------- invariants


def test_concatenating_groups_reproduces_grouped_result():
    rng = np.random.default_rng(3)
    E, N, K = 5, 11, 29
    counts = np.array([3, 0, 8, 1, 6])
    off = W.offsets_from_counts(counts)
    M = int(off[-1])
    x = rand_bits(rng, (M, K))
    w = rand_bits(rng, (E, N, K))
    y = oracle.mgemm(x, w, off)
    parts = []
    for e in range(E):
        a, b = off[e], off[e + 1]
        one = np.array([0, b - a], dtype=np.int32)
        parts.append(oracle.mgemm(x[a:b], w[e:e + 1], one))
    np.testing.assert_array_equal(y, np.concatenate(parts))


def test_dgrad_equals_forward_on_transposed_weights():
    rng = np.random.default_rng(4)
    E, N, K = 3, 13, 21
    off = W.offsets_from_counts([5, 7, 2])
    x = rand_bits(rng, (14, K))
    w_kn = rand_bits(rng, (E, K, N))
    a = oracle.mgemm(x, w_kn, off, transpose_B=True)
    b = oracle.mgemm(x, np.ascontiguousarray(w_kn.transpose(0, 2, 1)), off)
    np.testing.assert_array_equal(a, b)


def test_kgemm_empty_group_is_zero_and_rows_past_end_ignored():
    rng = np.random.default_rng(5)
    off = np.array([0, 4, 4, 9], dtype=np.int32)
    M, N, K = 12, 6, 10
    grad = rand_bits(rng, (M, N))
    X = rand_bits(rng, (M, K))
    dW = oracle.kgemm(grad, X, off)
    assert (dW[1] == 0).all()
    grad2 = grad.copy()
    grad2[9:] = bits(np.full((3, N), 1e30))  # rows past offsets[E] must not matter
    np.testing.assert_array_equal(oracle.kgemm(grad2, X, off), dW)


def test_kgemm_split_group_sums_to_whole():
    """Splitting a group into two consecutive groups and adding their dW gives
    the original (exact with integer inputs)."""
    rng = np.random.default_rng(6)
    M, N, K = 40, 9, 17
    gi = rng.integers(-2, 3, size=(M, N))
    xi = rng.integers(-2, 3, size=(M, K))
    whole = oracle.kgemm(bits(gi), bits(xi), np.array([0, 3, 40], dtype=np.int32))
    split = oracle.kgemm(bits(gi), bits(xi), np.array([0, 3, 25, 40], dtype=np.int32))
    np.testing.assert_array_equal(whole[0], split[0])
    np.testing.assert_array_equal(whole[1], split[1] + split[2])


def test_row_and_pair_subsets_match_full():
    rng = np.random.default_rng(8)
    off = W.offsets_from_counts([10, 0, 7, 15])
    M, N, K = 35, 12, 20
    x = rand_bits(rng, (M, K))
    w = rand_bits(rng, (4, N, K))
    y = oracle.mgemm(x, w, off)
    rows = np.array([31, 0, 16, 17, 9])
    np.testing.assert_array_equal(oracle.mgemm(x, w, off, rows=rows), y[rows])
    grad = rand_bits(rng, (M, N))
    dW = oracle.kgemm(grad, x, off)
    se, sn = np.array([3, 0, 1, 2]), np.array([11, 0, 5, 7])
    np.testing.assert_array_equal(oracle.kgemm(grad, x, off, sel=(se, sn)), dW[se, sn])


def test_bad_offsets_rejected():
    x = bits(np.ones((4, 8)))
    w = bits(np.ones((2, 8, 8)))
    for off in ([1, 2, 4], [0, 3, 2], [0, 2, 5]):
        with pytest.raises(ValueError):
            oracle.mgemm(x, w, np.array(off, dtype=np.int32))


def test_planted_index_mistake_is_caught():
    """A transposed weight index (w[e,k,n] read as w[e,n,k]) changes the
    result whenever N != K: the pins above must see it."""
    rng = np.random.default_rng(9)
    x = rand_bits(rng, (6, 5))
    w = rand_bits(rng, (1, 3, 5))
    off = np.array([0, 6], dtype=np.int32)
    right = oracle.mgemm(x, w, off)
    wrong = f64(x) @ f64(w[0]).reshape(5, 3)  # the mistake, planted on the CPU side only
    assert not np.allclose(right, wrong)


# ---------------------------------------------------------------- generator


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    v = rng.standard_normal(100000).astype(np.float32) * 3
    # add exact ties: values halfway between two bf16 numbers
    ties = (np.arange(1, 1001, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    v = np.concatenate([v, ties, -ties])
    ours = W.f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_workload_counts():
    t = W.tiny()
    assert t.counts.sum() == 512 and t.counts[2] == 0
    assert all(c % 128 for c in t.counts[[0, 1, 3]])
    a = W.a3b_layer()
    assert a.counts.sum() == 32768 and len(a.counts) == 32
    s = W.skewed()
    assert s.counts.sum() == 65536 and len(s.counts) == 128
    st = W.skewed(tail=True)
    assert st.counts.sum() == 65536 and (st.counts == 0).sum() >= 4
    assert (st.counts <= 7).sum() >= 32
    off = a.offsets
    assert off[0] == 0 and off[-1] == 32768 and (np.diff(off) >= 0).all()


# ---------------------------------------------------------------- SwiGLU


def test_swiglu_handworked_and_limits():
    e = np.e
    y = np.array([[0.0, 1.0, 5.0, 2.0],      # F=2: gate (0, 1), up (5, 2)
                  [-50.0, 40.0, 3.0, -1.0]])  # gate (-50, 40), up (3, -1)
    h = oracle.swiglu(y)
    # by hand: silu(0)*5 = 0;  silu(1)*2 = 2/(1+1/e);  silu(-50)*3 ~ -150*e^-50;  silu(40)*-1 ~ -40
    np.testing.assert_allclose(h[0], [0.0, 2.0 / (1.0 + 1.0 / e)], rtol=1e-15)
    assert abs(h[1, 0]) < 1e-18 and h[1, 0] <= 0.0
    np.testing.assert_allclose(h[1, 1], -40.0, rtol=1e-15)


def test_swiglu_matches_library_sigmoid_and_layout():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(21)
    y = rng.standard_normal((7, 10)) * 4
    h = oracle.swiglu(y)
    gate, up = y[:, :5], y[:, 5:]
    np.testing.assert_allclose(h, gate * scipy_special.expit(gate) * up, rtol=1e-13, atol=1e-300)
    # swapping the halves changes the result (the gate half is the first one)
    assert not np.allclose(h, oracle.swiglu(np.concatenate([up, gate], axis=1)))


def test_swiglu_bwd_is_the_gradient_of_swiglu():
    """Central differences of <dh, swiglu(y13)> reproduce swiglu_bwd."""
    rng = np.random.default_rng(22)
    y = rng.standard_normal((3, 8)) * 3
    dh = rng.standard_normal((3, 4))
    g = oracle.swiglu_bwd(dh, y)
    eps = 1e-6
    num = np.zeros_like(y)
    for i in range(y.shape[0]):
        for j in range(y.shape[1]):
            yp, ym = y.copy(), y.copy()
            yp[i, j] += eps
            ym[i, j] -= eps
            num[i, j] = (np.sum(dh * oracle.swiglu(yp)) - np.sum(dh * oracle.swiglu(ym))) / (2 * eps)
    np.testing.assert_allclose(g, num, rtol=1e-7, atol=1e-8)


def test_swiglu_bwd_matches_autograd_and_handworked():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(23)
    y = rng.standard_normal((5, 12)) * 4
    dh = rng.standard_normal((5, 6))
    yt = torch.tensor(y, requires_grad=True)
    h = torch.nn.functional.silu(yt[:, :6]) * yt[:, 6:]
    h.backward(torch.tensor(dh))
    np.testing.assert_allclose(oracle.swiglu_bwd(dh, y), yt.grad.numpy(), rtol=1e-12, atol=1e-14)
    # gate 0: s = 1/2, so d gate = dh*up/2 and d up = 0; a large gate passes dh through
    d = oracle.swiglu_bwd(np.array([[2.0, 1.0]]), np.array([[0.0, 60.0, 3.0, 5.0]]))
    np.testing.assert_allclose(d[0], [3.0, 5.0, 0.0, 60.0], rtol=1e-12, atol=1e-20)


# ------------------------------------------------ nested grouped GEMM (CUTLASS #1452)


@pytest.mark.parametrize("transpose_B", [False, True])
def test_nested_golden_handworked(transpose_B):
    g = json.load(open(os.path.join(GOLDEN, "handworked_nested.json")))
    off = np.array(g["offsets"], dtype=np.int32)
    y = oracle.mgemm_nested(bits(g["x"]), bits(g["w"]), off, transpose_B=transpose_B)
    want = g["dgrad" if transpose_B else "fwd"]["y_rows_0_to_1"]
    np.testing.assert_array_equal(y[:2], np.array(want, dtype=np.float64))
    assert np.isnan(y[2]).all()  # row 2 belongs to no inner group


def brute_nested(x, w, offsets, O, transpose_B):
    """Independent pure-Python loop: outer group, inner group, row, column, k."""
    M = len(x)
    K = len(w[0][0]) if transpose_B else len(w[0][0][0])
    N = len(w[0][0][0]) if transpose_B else len(w[0][0])
    L = len(offsets) - 1
    y = [[None] * (O * N) for _ in range(M)]
    for o in range(O):
        for l in range(L):
            for r in range(offsets[l], offsets[l + 1]):
                for n in range(N):
                    s = 0.0
                    for k in range(K):
                        b = w[o][l][k][n] if transpose_B else w[o][l][n][k]
                        s += x[r][o * K + k] * b
                    y[r][o * N + n] = s
    return y


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("transpose_B", [False, True])
def test_nested_matches_brute_force(seed, transpose_B):
    rng = np.random.default_rng(500 + seed)
    O = int(rng.integers(1, 4))
    L = 3
    M = int(rng.integers(4, 11))
    N = int(rng.integers(1, 6))
    K = int(rng.integers(1, 6))
    counts = rng.multinomial(M - 1, [0.5, 0.0, 0.5])  # inner group 1 empty, 1 row past offsets[L]
    off = W.offsets_from_counts(counts)
    x = rand_bits(rng, (M, O * K))
    w = rand_bits(rng, (O, L, K, N) if transpose_B else (O, L, N, K))
    y = oracle.mgemm_nested(x, w, off, transpose_B=transpose_B)
    ref = brute_nested(f64(x).tolist(), f64(w).tolist(), off.tolist(), O, transpose_B)
    for r in range(M):
        if ref[r][0] is None:
            assert np.isnan(y[r]).all()
        else:
            np.testing.assert_array_equal(y[r], np.array(ref[r]))


@pytest.mark.parametrize("transpose_B", [False, True])
def test_nested_blocks_are_ordinary_gemms_on_integers(transpose_B):
    """Every (outer, inner) block is an ordinary GEMM of a column slice of x
    with one weight matrix; integer inputs make both sides exact."""
    rng = np.random.default_rng(7)
    O, L, N, K = 3, 4, 5, 6
    counts = np.array([3, 0, 4, 2])
    off = W.offsets_from_counts(counts)
    M = int(off[-1]) + 2
    xi = rng.integers(-2, 3, size=(M, O * K))
    wi = rng.integers(-2, 3, size=(O, L, K, N) if transpose_B else (O, L, N, K))
    y = oracle.mgemm_nested(bits(xi), bits(wi), off, transpose_B=transpose_B)
    for o in range(O):
        for l in range(L):
            r0, r1 = int(off[l]), int(off[l + 1])
            b = wi[o, l] if transpose_B else wi[o, l].T
            np.testing.assert_array_equal(y[r0:r1, o * N:(o + 1) * N],
                                          (xi[r0:r1, o * K:(o + 1) * K] @ b).astype(np.float64))
    assert np.isnan(y[int(off[-1]):]).all()


@pytest.mark.parametrize("transpose_B", [False, True])
def test_nested_flattens_to_grouped_gemms(transpose_B):
    """Both flattenings of the discussion: (1) column block o equals the plain
    grouped GEMM of x's column slice o with the weight stack w[o]; (2) LoRA over
    MoE -- inner groups ordered (adapter, expert) with O = 1 -- equals one
    grouped GEMM per adapter over that adapter's rows and expert stack."""
    rng = np.random.default_rng(11)
    O, L, N, K = 2, 6, 7, 5
    counts = rng.multinomial(40, [1 / L] * L)
    counts[2] = 0
    off = W.offsets_from_counts(counts)
    M = int(off[-1])
    x = rand_bits(rng, (M, O * K))
    w = rand_bits(rng, (O, L, K, N) if transpose_B else (O, L, N, K))
    y = oracle.mgemm_nested(x, w, off, transpose_B=transpose_B)
    for o in range(O):
        xo = np.ascontiguousarray(x[:, o * K:(o + 1) * K])
        np.testing.assert_array_equal(y[:, o * N:(o + 1) * N],
                                      oracle.mgemm(xo, w[o], off, transpose_B=transpose_B))
    # (2): 2 adapters x 3 experts, inner group l = 3 * adapter + expert
    x1 = np.ascontiguousarray(x[:, :K])
    y1 = oracle.mgemm_nested(x1, np.ascontiguousarray(w[:1]), off, transpose_B=transpose_B)
    for a in range(2):
        r0, r1 = int(off[3 * a]), int(off[3 * a + 3])
        sub = (off[3 * a:3 * a + 4] - off[3 * a]).astype(np.int32)
        ya = oracle.mgemm(np.ascontiguousarray(x1[r0:r1]), np.ascontiguousarray(w[0, 3 * a:3 * a + 3]),
                          sub, transpose_B=transpose_B)
        np.testing.assert_array_equal(y1[r0:r1], ya)


def test_nested_row_subset_matches_full():
    rng = np.random.default_rng(12)
    off = W.offsets_from_counts(np.array([5, 0, 7]))
    x = rand_bits(rng, (14, 2 * 8))
    w = rand_bits(rng, (2, 3, 9, 8))
    full = oracle.mgemm_nested(x, w, off)
    rows = np.array([11, 0, 4, 5, 4])
    np.testing.assert_array_equal(oracle.mgemm_nested(x, w, off, rows=rows), full[rows])
    with pytest.raises(ValueError):
        oracle.mgemm_nested(x, w, off, rows=np.array([12]))  # past offsets[L]


def test_nested_planted_column_offset_mistake_is_caught():
    """Reading every outer group's contraction from x's first column block
    (a dropped o*K offset) must differ from the oracle whenever the blocks
    differ: the pins above must see it."""
    rng = np.random.default_rng(13)
    off = W.offsets_from_counts(np.array([3, 4]))
    x = rand_bits(rng, (7, 2 * 4))
    w = rand_bits(rng, (2, 2, 3, 4))
    right = oracle.mgemm_nested(x, w, off)
    wrong = np.concatenate(  # the mistake, planted on the CPU side only
        [np.concatenate([f64(x[r0:r1, :4]) @ f64(w[o, l]).T for l, (r0, r1) in enumerate([(0, 3), (3, 7)])])
         for o in range(2)], axis=1)
    assert not np.allclose(right, wrong)


# ------------------------------------------------ MXFP8 (E4M3 elements, E8M0 block scales)


def test_mx_decode_tables_match_closed_forms_and_torch():
    e4, e8 = oracle.mx_decode_tables()
    # closed forms of the OCP E4M3 / E8M0 encodings
    assert e4[0x00] == 0.0 and e4[0x80] == 0.0
    assert e4[0x01] == 2.0 ** -9 and e4[0x07] == 7 * 2.0 ** -9  # subnormals
    assert e4[0x08] == 2.0 ** -6 and e4[0x38] == 1.0 and e4[0x40] == 2.0
    assert e4[0x7E] == 448.0 and e4[0xFE] == -448.0 and e4[0xB8] == -1.0
    assert np.isnan(e4[0x7F]) and np.isnan(e4[0xFF])
    assert e8[127] == 1.0 and e8[0] == 2.0 ** -127 and e8[254] == 2.0 ** 127 and np.isnan(e8[255])
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    t4 = codes.view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(e4, t4)
    if hasattr(torch, "float8_e8m0fnu"):
        t8 = codes.view(torch.float8_e8m0fnu).double().numpy()
        np.testing.assert_array_equal(e8, t8)


def _mx_tiny(rng, E, M, N, K, transpose_B):
    xq = W.e4m3_codes((M, K), int(rng.integers(1 << 30)), 0)
    wq = W.e4m3_codes((E, K, N) if transpose_B else (E, N, K), int(rng.integers(1 << 30)), 1)
    sx = W.e8m0_codes((M, K // 32), 118, 130, int(rng.integers(1 << 30)), 2)
    sw = W.e8m0_codes((E, N, K // 32), 118, 130, int(rng.integers(1 << 30)), 3)
    return xq, sx, wq, sw


@pytest.mark.parametrize("transpose_B", [False, True])
def test_mx_mgemm_matches_brute_force(transpose_B):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    E, M, N, K = 3, 7, 3, 64
    off = W.offsets_from_counts([3, 0, 3])  # one row past offsets[E]
    xq, sx, wq, sw = _mx_tiny(rng, E, M, N, K, transpose_B)
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy().tolist()  # noqa: E731
    X, Wt, SX, SW = dec(xq), dec(wq), sx.tolist(), sw.tolist()
    y = oracle.mgemm_mx(xq, sx, wq, sw, off, transpose_B=transpose_B)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            for n in range(N):
                s = 0.0
                for k in range(K):
                    b = Wt[e][k][n] if transpose_B else Wt[e][n][k]
                    s += (X[r][k] * 2.0 ** (SX[r][k // 32] - 127)) * (b * 2.0 ** (SW[e][n][k // 32] - 127))
                assert y[r, n] == s
    assert np.isnan(y[6]).all()


@pytest.mark.parametrize("transpose_B", [False, True])
def test_mx_mgemm_equals_bf16_grouped_gemm_on_dequantized_inputs(transpose_B):
    """Every scaled E4M3 value (4 significant bits, moderate exponent) is a
    bf16 value: dequantizing both operands exactly and running the pinned
    bf16 grouped GEMM must give the identical FP64 result."""
    rng = np.random.default_rng(32)
    E, N, K = 4, 9, 96
    off = W.offsets_from_counts([5, 0, 11, 6])
    M = int(off[-1]) + 2
    xq, sx, wq, sw = _mx_tiny(rng, E, M, N, K, transpose_B)
    e4, e8 = oracle.mx_decode_tables()
    xv = e4[xq] * e8[np.repeat(sx, 32, axis=1)]
    swk = e8[np.repeat(sw, 32, axis=2)]  # scale of w element (n, k): [E, N, K]
    wv = e4[wq] * (np.transpose(swk, (0, 2, 1)) if transpose_B else swk)
    xb, wb = W.f32_to_bf16_bits(xv.astype(np.float32)), W.f32_to_bf16_bits(wv.astype(np.float32))
    assert (W.bf16_bits_to_f32(xb) == xv).all() and (W.bf16_bits_to_f32(wb) == wv).all()
    np.testing.assert_array_equal(oracle.mgemm_mx(xq, sx, wq, sw, off, transpose_B=transpose_B),
                                  oracle.mgemm(xb, wb, off, transpose_B=transpose_B))


def test_mx_mgemm_integer_codes_exact():
    """Integer elements and scales of 1/2, 1 and 2: the result is an exact
    small multiple of 1/4, equal to an int64 numpy GEMM per group."""
    e4, _ = oracle.mx_decode_tables()
    code_of = {v: int(np.flatnonzero(e4 == v)[0]) for v in (-2.0, -1.0, 0.0, 1.0, 2.0)}
    rng = np.random.default_rng(33)
    E, N, K = 2, 5, 64
    off = W.offsets_from_counts([4, 3])
    M = 7
    xi = rng.integers(-2, 3, size=(M, K))
    wi = rng.integers(-2, 3, size=(E, N, K))
    sxe = rng.integers(-1, 2, size=(M, K // 32))
    swe = rng.integers(-1, 2, size=(E, N, K // 32))
    enc = np.vectorize(lambda v: code_of[float(v)])
    y = oracle.mgemm_mx(enc(xi).astype(np.uint8), (127 + sxe).astype(np.uint8),
                        enc(wi).astype(np.uint8), (127 + swe).astype(np.uint8), off)
    xs = xi * 2.0 ** np.repeat(sxe, 32, axis=1)
    for e in range(E):
        ws = wi[e] * 2.0 ** np.repeat(swe[e], 32, axis=1)
        r0, r1 = off[e], off[e + 1]
        np.testing.assert_array_equal(y[r0:r1], xs[r0:r1] @ ws.T)


def test_mx_planted_scale_index_mistake_is_caught():
    """Indexing the scale with k % 32 instead of k // 32 must change the
    result: the pins above must see it."""
    rng = np.random.default_rng(34)
    off = W.offsets_from_counts([4])
    xq, sx, wq, sw = _mx_tiny(rng, 1, 4, 3, 64, False)
    e4, e8 = oracle.mx_decode_tables()
    right = oracle.mgemm_mx(xq, sx, wq, sw, off)
    k = np.arange(64)
    wrong = (e4[xq] * e8[sx[:, (k % 32) % 2]]) @ (e4[wq[0]] * e8[sw[0][:, k // 32]]).T  # planted on the CPU
    assert not np.allclose(right, wrong)


def test_mx_blocked_golden_handworked():
    g = json.load(open(os.path.join(GOLDEN, "mx_blocked_handworked.json")))
    for case in g["cases"]:
        R, KS = case["R"], case["KS"]
        r, c = np.meshgrid(np.arange(R), np.arange(KS), indexing="ij")
        src = eval(case["src"], {}, {"r": r, "c": c}).astype(np.uint8)
        dst = oracle.mx_blocked(src, np.array(case["offsets"], dtype=np.int32))
        for x in case["expect"]:
            assert int(dst[x["byte"]]) == x["value"], x["why"]


def test_mx_blocked_is_a_bijection_with_pad():
    """Every (row, scale column) lands on its own byte, read back by the
    inverse of the layout; every other byte of the used blocks is the pad."""
    rng = np.random.default_rng(35)
    counts = np.array([130, 0, 1, 255, 128, 7])
    off = W.offsets_from_counts(counts)
    R, KS = int(off[-1]) + 3, 7
    src = rng.integers(0, 256, size=(R, KS), dtype=np.int64).astype(np.uint8)
    dst = oracle.mx_blocked(src, off, fill=0xEE)
    nc = (KS + 3) // 4
    seen = np.zeros(dst.size, dtype=bool)
    blk = 0
    for g in range(len(counts)):
        for base in range(int(off[g]), int(off[g + 1]), 128):
            for i in range(128):
                for col in range(nc * 4):
                    pos = (blk * nc + col // 4) * 512 + 16 * (i % 32) + 4 * (i // 32) + col % 4
                    assert not seen[pos]
                    seen[pos] = True
                    rr = base + i
                    want = src[rr, col] if (rr < off[g + 1] and col < KS) else 0x7F
                    assert dst[pos] == want
            blk += 1
    assert (dst[~seen] == 0xEE).all() and seen[: blk * nc * 512].all()


def test_mx_blocked_full_blocks_are_a_reshape():
    """Groups of exactly 128 rows and KS a multiple of 4: each 512-byte block
    is the 128x4 tile reshaped (i//32, i%32, j) -> (i%32, i//32, j)."""
    rng = np.random.default_rng(36)
    G, KS = 3, 8
    src = rng.integers(0, 256, size=(128 * G, KS), dtype=np.int64).astype(np.uint8)
    dst = oracle.mx_blocked(src, W.offsets_from_counts([128] * G))
    want = src.reshape(G, 4, 32, KS // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    np.testing.assert_array_equal(dst[: want.size], want)


def test_mx_blocked_k_golden_handworked():
    g = json.load(open(os.path.join(GOLDEN, "mx_blocked_k_handworked.json")))
    r, c = np.meshgrid(np.arange(g["R"]), np.arange(g["KS"]), indexing="ij")
    src = eval(g["src"], {}, {"r": r, "c": c}).astype(np.uint8)
    dst = oracle.mx_blocked_k(src, np.array(g["offsets"], dtype=np.int32))
    for x in g["expect"]:
        assert int(dst[x["byte"]]) == x["value"], x["why"]


def test_mx_blocked_k_reduces_to_row_layout_for_whole_chunks():
    """Groups whose lengths are multiples of 128 (whole chunks): the chunks
    run through the scale columns in order, which is the row-grouped layout
    of the whole matrix taken as one group."""
    rng = np.random.default_rng(37)
    R, KS = 300, 16
    src = rng.integers(0, 256, size=(R, KS), dtype=np.int64).astype(np.uint8)
    off = np.array([0, 128, 128, 384, 512], dtype=np.int32)
    a = oracle.mx_blocked_k(src, off)
    b = oracle.mx_blocked(src, np.array([0, R], dtype=np.int32))
    n = ((R + 127) // 128) * (KS // 4) * 512
    np.testing.assert_array_equal(a[:n], b[:n])


def test_mx_blocked_k_is_a_bijection_with_pad():
    rng = np.random.default_rng(38)
    off = np.array([0, 64, 64, 96, 416], dtype=np.int32)
    R, KS = 200, 13
    src = rng.integers(0, 256, size=(R, KS), dtype=np.int64).astype(np.uint8)
    dst = oracle.mx_blocked_k(src, off, fill=0xEE)
    seen = np.zeros(dst.size, dtype=bool)
    chunks = [(g, cb) for g in range(4) for cb in range(off[g] // 32, off[g + 1] // 32, 4)]
    NQ = len(chunks)
    for rb in range((R + 127) // 128):
        for q, (g, cb) in enumerate(chunks):
            for i in range(128):
                for j in range(4):
                    pos = (rb * NQ + q) * 512 + 16 * (i % 32) + 4 * (i // 32) + j
                    assert not seen[pos]
                    seen[pos] = True
                    r, col = 128 * rb + i, cb + j
                    want = src[r, col] if (r < R and col < off[g + 1] // 32) else 0x7F
                    assert dst[pos] == want
    assert (dst[~seen] == 0xEE).all()


def _mxk_tiny(rng, M, N, K):
    s = int(rng.integers(1 << 30))
    gq, xq = W.e4m3_codes((M, N), s, 0), W.e4m3_codes((M, K), s, 1)
    sg = W.e8m0_codes((N, M // 32), 118, 130, s, 2)
    sx = W.e8m0_codes((K, M // 32), 118, 130, s, 3)
    return gq, sg, xq, sx


def test_mx_kgemm_matches_brute_force():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(39)
    M, N, K = 96, 3, 4
    off = np.array([0, 32, 32, 96], dtype=np.int32)
    gq, sg, xq, sx = _mxk_tiny(rng, M, N, K)
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy().tolist()  # noqa: E731
    G, X, SG, SX = dec(gq), dec(xq), sg.tolist(), sx.tolist()
    dW = oracle.kgemm_mx(gq, sg, xq, sx, off)
    for e in range(3):
        for n in range(N):
            for k in range(K):
                s = 0.0
                for r in range(off[e], off[e + 1]):
                    s += (G[r][n] * 2.0 ** (SG[n][r // 32] - 127)) * (X[r][k] * 2.0 ** (SX[k][r // 32] - 127))
                assert dW[e, n, k] == s
    assert (dW[1] == 0).all()


def test_mx_kgemm_equals_bf16_kgemm_on_dequantized_inputs():
    rng = np.random.default_rng(40)
    M, N, K = 192, 9, 11
    off = np.array([0, 64, 64, 160, 192], dtype=np.int32)
    gq, sg, xq, sx = _mxk_tiny(rng, M, N, K)
    e4, e8 = oracle.mx_decode_tables()
    gv = e4[gq] * e8[np.repeat(sg, 32, axis=1).T]
    xv = e4[xq] * e8[np.repeat(sx, 32, axis=1).T]
    gb, xb = W.f32_to_bf16_bits(gv.astype(np.float32)), W.f32_to_bf16_bits(xv.astype(np.float32))
    assert (W.bf16_bits_to_f32(gb) == gv).all() and (W.bf16_bits_to_f32(xb) == xv).all()
    np.testing.assert_array_equal(oracle.kgemm_mx(gq, sg, xq, sx, off), oracle.kgemm(gb, xb, off))


def test_mx_kgemm_rejects_unaligned_groups():
    rng = np.random.default_rng(41)
    gq, sg, xq, sx = _mxk_tiny(rng, 64, 2, 2)
    with pytest.raises(ValueError):
        oracle.kgemm_mx(gq, sg, xq, sx, np.array([0, 40, 64], dtype=np.int32))
