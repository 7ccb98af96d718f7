"""Pins of the CPU oracle to things other than itself.

* The worked examples printed on the MatMul, Gemm and QLinearMatMul pages
  (fixtures in tests/golden/, each citing its page and example).
* GroupedMatMul: the page prints inputs only; the expected outputs below are
  derived by hand in comments (unit-vector rows select weight rows, small
  integer sums), so they are exact in every float type.
* Closed forms: integer wrap-around, int32 accumulator wrap, ties-to-even.
* Independent brute force: pure-Python loops with explicit index arithmetic
  (no numpy broadcasting or matmul) on tiny random inputs.
* Identities: (A B)^T = B^T A^T through transA/transB; GroupedMatMul with one
  group and one selection equals Gemm with a (1, N) bias; identity and
  permutation weights.
* The error-bound denominators (the *_abs_scale functions) by hand values
  with negative entries, a negative alpha and a broadcast C.

Every pin runs against both oracles: the numpy one (``oracle``) and the plain
C++ loops (``oracle.native``), which share no code with each other.
"""

import itertools
import json
import math
import pathlib

import numpy as np
import pytest

import oracle
import oracle.native

GOLDEN = pathlib.Path(__file__).parent / "golden"

# The oracle under test; the fixture below runs every pin once per oracle.
ORC = oracle


@pytest.fixture(autouse=True, params=["numpy", "cpp"])
def _which_oracle(request):
    global ORC
    ORC = oracle if request.param == "numpy" else oracle.native
    yield
    ORC = oracle


def _load(name):
    with open(GOLDEN / name) as f:
        return json.load(f)["examples"]


def _arr(spec):
    return np.array(spec["values"], dtype=spec["dtype"]).reshape(spec["shape"])


MATMUL_EX = _load("matmul_examples.json")
GEMM_EX = _load("gemm_examples.json")
QLINEAR_EX = _load("qlinearmatmul_examples.json")

# Printed float32 results carry ~8 significant digits and were themselves
# computed in float32: allow 1e-6 of the term magnitude plus of the value.
PRINT_TOL = 1e-6


@pytest.mark.parametrize("ex", MATMUL_EX, ids=[e["name"] for e in MATMUL_EX])
def test_matmul_page_examples(ex):
    A, B = _arr(ex["inputs"]["A"]), _arr(ex["inputs"]["B"])
    want = _arr(ex["outputs"]["Y"]).astype(np.float64)
    got = ORC.matmul(A, B)
    assert got.shape == want.shape
    scale = ORC.matmul_abs_scale(A, B)
    assert np.all(np.abs(got - want) <= PRINT_TOL * (scale + np.abs(want)))


@pytest.mark.parametrize("ex", GEMM_EX, ids=[e["name"] for e in GEMM_EX])
def test_gemm_page_examples(ex):
    at = ex["attributes"]
    kw = dict(alpha=at.get("alpha", 1.0), beta=at.get("beta", 1.0),
              transA=at.get("transA", 0), transB=at.get("transB", 0))
    A, B = _arr(ex["inputs"]["A"]), _arr(ex["inputs"]["B"])
    C = _arr(ex["inputs"]["C"]) if "C" in ex["inputs"] else None
    want = _arr(ex["outputs"]["Y"]).astype(np.float64)
    got = ORC.gemm(A, B, C, **kw)
    assert got.shape == want.shape
    scale = ORC.gemm_abs_scale(A, B, C, **kw)
    assert np.all(np.abs(got - want) <= PRINT_TOL * (scale + np.abs(want)))


@pytest.mark.parametrize("ex", QLINEAR_EX, ids=[e["name"] for e in QLINEAR_EX])
def test_qlinear_page_examples_bit_exact(ex):
    i = ex["inputs"]
    args = [_arr(i[k]) for k in ("a", "a_scale", "a_zero_point", "b", "b_scale",
                                 "b_zero_point", "y_scale", "y_zero_point")]
    want = _arr(ex["outputs"]["y"])
    got = ORC.qlinear_matmul(*args)
    assert got.dtype == want.dtype and got.shape == want.shape
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- QLinear closed forms

def _ql(a, b, sa=1.0, za=0, sb=1.0, zb=0, ys=1.0, yz=0, t_in=np.int8, t_out=np.int8):
    return ORC.qlinear_matmul(np.asarray(a, t_in), np.float32(sa), t_in(za),
                                 np.asarray(b, t_in), np.float32(sb), t_in(zb),
                                 np.float32(ys), t_out(yz))


def test_qlinear_ties_round_to_even():
    # acc = 1, 3, 5, -1, -3 with unit scales and y_scale = 2 gives quotients
    # 0.5, 1.5, 2.5, -0.5, -1.5; ties-to-even rounds them to 0, 2, 2, 0, -2.
    y = _ql([[1], [3], [5], [-1], [-3]], [[1]], ys=2.0)
    assert y.ravel().tolist() == [0, 2, 2, 0, -2]


def test_qlinear_saturation_and_zero_point_after_rounding():
    # 100*100 / 0.5 = 20000 saturates to 127; the zero point is added after
    # rounding: 7/2 = 3.5 -> 4, + 3 = 7 (adding before rounding would give 6.5 -> 6).
    assert _ql([[100]], [[100]], ys=0.5).item() == 127
    assert _ql([[7]], [[1]], ys=2.0, yz=3).item() == 7
    assert _ql([[0]], [[100]], t_in=np.uint8, t_out=np.uint8, za=100).item() == 0


def test_qlinear_per_row_and_per_column_parameters():
    # a = [[1,2],[3,4]], per-row za = [0,1], per-row sa = [1,2];
    # b = I, per-column zb = [0,0], sb = [1, 0.5]; y_scale 1, y_zp 0.
    # acc = (a - za) @ b = [[1,2],[2,3]];  s[m,n] = sa[m]*sb[n] = [[1,.5],[2,1]]
    # y = acc * s = [[1,1],[4,3]].
    a = np.array([[1, 2], [3, 4]], np.int8)
    b = np.array([[1, 0], [0, 1]], np.int8)
    for shape_a, shape_b in (((2,), (2,)), ((2, 1), (1, 2))):
        y = ORC.qlinear_matmul(
            a, np.array([1.0, 2.0], np.float32).reshape(shape_a), np.array([0, 1], np.int8).reshape(shape_a),
            b, np.array([1.0, 0.5], np.float32).reshape(shape_b), np.array([0, 0], np.int8).reshape(shape_b),
            np.float32(1.0), np.int8(0))
        assert y.tolist() == [[1, 1], [4, 3]]


def test_qlinear_accumulator_wraps_in_32_bits():
    # (255-0)*(255-0) = 65025 per k; K = 33026 gives 2147515650 > 2**31 - 1,
    # which wraps to 2147515650 - 2**32 = -2147451646.  With y_scale = 2**24
    # the quotient is about -128.0 (wrapped) instead of +128.0 (unwrapped).
    K = 33026
    a = np.full((1, K), 255, np.uint8)
    b = np.full((K, 1), 255, np.uint8)
    y = ORC.qlinear_matmul(a, np.float32(1), np.uint8(0), b, np.float32(1), np.uint8(0),
                              np.float32(2.0 ** 24), np.int8(0))
    assert y.item() == -128


def test_requantize_is_float32_sequence():
    # 49.90-style value: acc 1000, s = 0.0066*0.00705 (float32), y_scale 0.0107.
    s = np.float32(0.0066) * np.float32(0.00705)
    v = np.float32(1000) * s
    q = v / np.float32(0.0107)
    assert ORC.requantize(np.int32(1000), np.float32(0.0066), np.float32(0.00705),
                             np.float32(0.0107), np.int8(0), np.int8) == np.int8(round(float(q)))


# ---------------------------------------------------------------- integer closed forms

@pytest.mark.parametrize("dt,bits", [(np.int32, 32), (np.uint32, 32), (np.int64, 64), (np.uint64, 64)])
def test_integer_matmul_wraps_modulo_2n(dt, bits):
    # [2^(n-2), 2^(n-2)] @ [2, 2]^T = 2^n = 0 modulo 2^n; and 3 * x for a row
    # of x = 2^(n-1) gives 2^(n-1) (mod 2^n).
    h = 1 << (bits - 2)
    A = np.array([[h, h]], dtype=np.uint64).astype(dt)
    B = np.array([[2], [2]], dtype=dt)
    assert ORC.matmul(A, B).item() == 0
    A2 = np.array([[1 << (bits - 1)]], dtype=np.uint64).astype(dt)
    B2 = np.array([[3]], dtype=dt)
    want = np.array([1 << (bits - 1)], dtype=np.uint64).astype(dt).item()
    assert ORC.matmul(A2, B2).item() == want


def test_signed_integer_matmul_negative_values():
    A = np.array([[-3, 4]], np.int32)
    B = np.array([[5], [-6]], np.int32)
    assert ORC.matmul(A, B).item() == -39


# ---------------------------------------------------------------- brute force

def _bf_matmul(A, B):
    """numpy.matmul by explicit index arithmetic with Python numbers."""
    A = np.asarray(A)
    B = np.asarray(B)
    a_shape, b_shape = list(A.shape), list(B.shape)
    a1, b1 = len(a_shape) == 1, len(b_shape) == 1
    if a1:
        a_shape = [1] + a_shape
    if b1:
        b_shape = b_shape + [1]
    M, K = a_shape[-2], a_shape[-1]
    N = b_shape[-1]
    assert b_shape[-2] == K
    nb = max(len(a_shape), len(b_shape)) - 2
    pa = [1] * (nb - (len(a_shape) - 2)) + a_shape[:-2]
    pb = [1] * (nb - (len(b_shape) - 2)) + b_shape[:-2]
    batch = [max(x, y) if min(x, y) == 1 else x for x, y in zip(pa, pb)]
    af = [x.item() if hasattr(x, "item") else x for x in A.reshape(-1)]
    bf = [x.item() if hasattr(x, "item") else x for x in B.reshape(-1)]

    def flat(shape, idx):
        o = 0
        for s, i in zip(shape, idx):
            o = o * s + i
        return o
    out = {}
    for bidx in itertools.product(*[range(d) for d in batch]):
        ia = [i if d != 1 else 0 for i, d in zip(bidx, pa)]
        ib = [i if d != 1 else 0 for i, d in zip(bidx, pb)]
        for m in range(M):
            for n in range(N):
                s = 0
                for k in range(K):
                    s += af[flat(pa + [M, K], ia + [m, k])] * bf[flat(pb + [K, N], ib + [k, n])]
                out[bidx + (m, n)] = s
    shape = batch + ([] if a1 else [M]) + ([] if b1 else [N])
    res = np.zeros(shape, dtype=object)
    for key, v in out.items():
        bk, m, n = key[:nb], key[nb], key[nb + 1]
        k2 = bk + (() if a1 else (m,)) + (() if b1 else (n,))
        res[k2] = v
    return res


MATMUL_SHAPES = [((3,), (3,)), ((4,), (2, 4, 3)), ((2, 3, 4, 5), (5,)), ((2, 1, 3, 2), (4, 2, 5)),
                 ((3, 1, 2), (1, 2, 4)), ((5, 3), (3, 4)), ((1, 2, 3), (3, 2)), ((2, 0), (0, 3)),
                 ((0, 2, 3), (3, 2))]


@pytest.mark.parametrize("sa,sb", MATMUL_SHAPES)
def test_matmul_brute_force_float(sa, sb):
    rng = np.random.default_rng(7)
    A = rng.integers(-9, 10, size=sa).astype(np.float32) / 4
    B = rng.integers(-9, 10, size=sb).astype(np.float32) / 8
    got = ORC.matmul(A, B)
    want = _bf_matmul(A.astype(np.float64), B.astype(np.float64)).astype(np.float64)
    assert got.shape == want.shape
    assert np.array_equal(got, want)  # small dyadic values: every sum is exact


@pytest.mark.parametrize("dt", [np.int32, np.int64, np.uint32, np.uint64])
def test_matmul_brute_force_integer(dt):
    rng = np.random.default_rng(11)
    info = np.iinfo(dt)
    for sa, sb in MATMUL_SHAPES[:6]:
        A = rng.integers(info.min, info.max, size=sa, dtype=dt, endpoint=True)
        B = rng.integers(info.min, info.max, size=sb, dtype=dt, endpoint=True)
        got = ORC.matmul(A, B)
        bf = _bf_matmul(A.astype(object), B.astype(object))
        mod = 1 << (8 * np.dtype(dt).itemsize)
        want = [int(v) % mod for v in np.asarray(bf, dtype=object).reshape(-1)]
        have = [int(v) % mod for v in np.asarray(got).reshape(-1).tolist()]
        assert got.dtype == np.dtype(dt) and got.shape == bf.shape and have == want


def _bf_rne(q):
    f = math.floor(q)
    d = q - f
    if d > 0.5:
        return f + 1
    if d < 0.5:
        return f
    return f if f % 2 == 0 else f + 1


def _bf_qlinear_2d(a, za, sa, b, zb, sb, ys, yz, lo, hi):
    """Per element: exact int sum, wrap to int32, float32 steps one at a time, RNE by hand."""
    M, K = len(a), len(a[0])
    N = len(b[0])
    f32 = np.float32
    y = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = sum((a[m][k] - za[m]) * (b[k][n] - zb[n]) for k in range(K))
            acc = (acc + 2 ** 31) % 2 ** 32 - 2 ** 31
            s = f32(sa[m]) * f32(sb[n])
            v = f32(acc) * s
            q = float(v / f32(ys))
            t = float(f32(_bf_rne(q)) + f32(yz))
            y[m][n] = int(min(max(t, lo), hi))
    return y


@pytest.mark.parametrize("t_in,t_out", [(np.int8, np.int8), (np.uint8, np.uint8),
                                        (np.int8, np.uint8), (np.uint8, np.int8)])
def test_qlinear_brute_force(t_in, t_out):
    rng = np.random.default_rng(3)
    lo_in, hi_in = np.iinfo(t_in).min, np.iinfo(t_in).max
    lo, hi = float(np.iinfo(t_out).min), float(np.iinfo(t_out).max)
    M, K, N = 5, 9, 4
    a = rng.integers(lo_in, hi_in, size=(M, K), endpoint=True).astype(t_in)
    b = rng.integers(lo_in, hi_in, size=(K, N), endpoint=True).astype(t_in)
    za = rng.integers(lo_in, hi_in, size=(M,), endpoint=True).astype(t_in)
    zb = rng.integers(lo_in, hi_in, size=(N,), endpoint=True).astype(t_in)
    sa = rng.uniform(0.003, 0.01, size=(M,)).astype(np.float32)
    sb = rng.uniform(0.003, 0.01, size=(N,)).astype(np.float32)
    ys = np.float32(0.05)
    yz = t_out(rng.integers(np.iinfo(t_out).min, np.iinfo(t_out).max))
    got = ORC.qlinear_matmul(a, sa, za, b, sb, zb, ys, yz)
    want = _bf_qlinear_2d(a.astype(int).tolist(), za.astype(int).tolist(), sa.tolist(),
                          b.astype(int).tolist(), zb.astype(int).tolist(), sb.tolist(),
                          ys, int(yz), lo, hi)
    assert got.tolist() == want


def test_qlinear_batched_per_row_column_brute_force():
    # N-D: a [2, 3, 4] with per-row params [2, 3, 1]; b [2, 4, 5] with per-column [2, 1, 5].
    rng = np.random.default_rng(5)
    a = rng.integers(-128, 127, size=(2, 3, 4), endpoint=True).astype(np.int8)
    b = rng.integers(-128, 127, size=(2, 4, 5), endpoint=True).astype(np.int8)
    za = rng.integers(-20, 20, size=(2, 3, 1), endpoint=True).astype(np.int8)
    zb = rng.integers(-20, 20, size=(2, 1, 5), endpoint=True).astype(np.int8)
    sa = rng.uniform(0.003, 0.01, size=(2, 3, 1)).astype(np.float32)
    sb = rng.uniform(0.003, 0.01, size=(2, 1, 5)).astype(np.float32)
    got = ORC.qlinear_matmul(a, sa, za, b, sb, zb, np.float32(0.02), np.int8(-9))
    for d in range(2):
        want = _bf_qlinear_2d(a[d].astype(int).tolist(), za[d, :, 0].astype(int).tolist(),
                              sa[d, :, 0].tolist(), b[d].astype(int).tolist(),
                              zb[d, 0].astype(int).tolist(), sb[d, 0].tolist(),
                              np.float32(0.02), -9, -128.0, 127.0)
        assert got[d].tolist() == want


def _bf_gemm(A, B, C, alpha, beta, tA, tB):
    A = np.asarray(A).tolist()
    B = np.asarray(B).tolist()
    M = len(A[0]) if tA else len(A)
    K = len(A) if tA else len(A[0])
    N = len(B) if tB else len(B[0])
    Cn = None if C is None else np.asarray(C, dtype=np.float64)
    Y = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                a = A[k][i] if tA else A[i][k]
                b = B[j][k] if tB else B[k][j]
                s += a * b
            c = 0.0
            if Cn is not None:
                if Cn.ndim == 0:
                    c = float(Cn)
                elif Cn.ndim == 1:
                    c = float(Cn[0 if Cn.shape[0] == 1 else j])
                else:
                    c = float(Cn[0 if Cn.shape[0] == 1 else i, 0 if Cn.shape[1] == 1 else j])
            Y[i][j] = alpha * s + beta * c
    return np.array(Y, dtype=np.float64)


@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("c_shape", [None, (), (1,), (4,), (1, 4), (3, 1), (3, 4)])
def test_gemm_brute_force(tA, tB, c_shape):
    rng = np.random.default_rng(9)
    M, K, N = 3, 5, 4
    A = rng.integers(-8, 9, size=(K, M) if tA else (M, K)).astype(np.float32) / 2
    B = rng.integers(-8, 9, size=(N, K) if tB else (K, N)).astype(np.float32) / 4
    C = None if c_shape is None else (rng.integers(-8, 9, size=c_shape).astype(np.float32) / 8)
    got = ORC.gemm(A, B, C, alpha=0.5, beta=-2.0, transA=tA, transB=tB)
    want = _bf_gemm(A.astype(np.float64), B.astype(np.float64), C, 0.5, -2.0, tA, tB)
    assert np.array_equal(got, want)


def test_gemm_integer_exact():
    A = np.array([[2 ** 31 - 1, 2]], np.int32)
    B = np.array([[1], [1]], np.int32)
    C = np.array([[5]], np.int32)
    # A @ B = 2^31 + 1, which wraps to the int32 -2^31 + 1; then
    # 3 * (2^31 + 1) + (-1) * 5 = 3 * 2^31 - 2, which is 2^31 - 2 modulo 2^32:
    # the int32 2147483646 (alpha taken as 1 would give 2^31 - 4).
    got = ORC.gemm(A, B, C, alpha=3.0, beta=-1.0)
    want = ((3 * (2 ** 31 + 1) - 5) + 2 ** 31) % 2 ** 32 - 2 ** 31
    assert want == 2 ** 31 - 2
    assert got.item() == want
    # uint32, alpha 5, beta 7: 5 * (2^32 - 1) + 7 * 3 = 16 (mod 2^32)
    U = np.array([[2 ** 32 - 1]], np.uint32)
    got = ORC.gemm(U, np.array([[1]], np.uint32), np.array([[3]], np.uint32), alpha=5.0, beta=7.0)
    assert got.item() == 16


def test_gemm_integer_non_integral_alpha_beta():
    # The accumulator wraps in T first: A @ B = 2^31 is the int32 -2^31, so
    # 0.5 * acc + (-1) * 5 = -2^30 - 5.
    A = np.array([[2 ** 31 - 1, 1]], np.int32)
    B = np.array([[1], [1]], np.int32)
    C = np.array([[5]], np.int32)
    assert ORC.gemm(A, B, C, alpha=0.5, beta=-1.0).item() == -(2 ** 30) - 5
    # truncation toward zero: acc = +-3, alpha 0.5 -> +-1.5; with beta 0.25 and C = +-7 -> +-3.25
    A2 = np.array([[1, 2], [-1, -2]], np.int32)
    B2 = np.array([[1], [1]], np.int32)
    assert ORC.gemm(A2, B2, None, alpha=0.5).ravel().tolist() == [1, -1]
    C2 = np.array([[7], [-7]], np.int32)
    assert ORC.gemm(A2, B2, C2, alpha=0.5, beta=0.25).ravel().tolist() == [3, -3]
    # unsigned: 5 * float32(0.3) = 1.50000006 -> 1
    U = np.array([[5]], np.uint32)
    assert ORC.gemm(U, np.array([[1]], np.uint32), None, alpha=0.3).item() == 1
    # int64: the accumulator is rounded to float64 first: 2^54 + 3 -> 2^54 + 4, times 0.5
    L = np.array([[2 ** 54 + 3]], np.int64)
    assert ORC.gemm(L, np.array([[1]], np.int64), None, alpha=0.5).item() == 2 ** 53 + 2
    # results outside T's range are undefined: rejected
    with pytest.raises(ValueError):
        ORC.gemm(np.array([[2 ** 31 - 1]], np.int32), np.array([[1]], np.int32), None, alpha=1.5)


def test_gemm_transpose_identity():
    # (A B)^T = B^T A^T, expressed through the transA / transB attributes.
    rng = np.random.default_rng(1)
    A = rng.standard_normal((6, 5))
    B = rng.standard_normal((5, 7))
    Y = ORC.gemm(A, B)
    Yt = ORC.gemm(B, A, transA=1, transB=1)
    assert np.allclose(Y.T, Yt, rtol=0, atol=1e-12)
    Ai = rng.integers(-100, 100, size=(6, 5)).astype(np.int64)
    Bi = rng.integers(-100, 100, size=(5, 7)).astype(np.int64)
    assert np.array_equal(ORC.gemm(Ai, Bi).T, ORC.gemm(Bi, Ai, transA=1, transB=1))


def test_gemm_empty_k_and_column_broadcast():
    # K = 0: the product is empty, so Y = beta * C stretched; C of shape (M, 1)
    # is stretched along the columns.
    A = np.zeros((3, 0), np.float32)
    B = np.zeros((0, 4), np.float32)
    C = np.array([[1.0], [2.0], [3.0]], np.float32)
    Y = ORC.gemm(A, B, C, beta=2.0)
    assert np.array_equal(Y, np.repeat(np.array([[2.0], [4.0], [6.0]]), 4, axis=1))
    with pytest.raises(ValueError):
        ORC.gemm(A, B, np.zeros((2, 4), np.float32))


def test_matmul_shape_errors():
    with pytest.raises(ValueError):
        ORC.matmul(np.zeros((2, 3)), np.zeros((4, 2)))
    with pytest.raises(ValueError):
        ORC.matmul(np.zeros((2, 2, 3)), np.zeros((3, 3, 2)))
    with pytest.raises(ValueError):
        ORC.matmul(np.zeros(()), np.zeros((3,)))


# ---------------------------------------------------------------- GroupedMatMul
# Inputs are those of the examples on the GroupedMatMul - 29 page (section
# "Examples"); the page does not print outputs.

def _grouped_examples():
    f = np.float32
    return {
        # Row 0 of input is e0-weighted: [1,2] @ I = [1,2] (+[0.5,1]); [1,2] @ swap = [2,1] (+[1.5,2]);
        # [3,4] @ swap = [4,3] (+[1.5,2]); [3,4] @ I (+[0.5,1]).
        "_additional_types": (np.array([[1, 2], [3, 4]], f),
                              np.array([[[1, 0], [0, 1]], [[0, 1], [1, 0]]], f),
                              np.array([[0, 1], [1, 0]], np.int32),
                              np.array([[0.5, 1], [1.5, 2]], f),
                              [[[1.5, 3], [3.5, 3]], [[5.5, 5], [3.5, 5]]]),
        # [1,0,-1] @ W0 = [1,0] - [-1,0] = [2,0]; [0,1,2] @ W1 = [1,0] + 2*[0,1] = [1,2];
        # [1,1,0] @ W0 = [1,1]; [0,0,1] @ W1 = [0,1].
        "default": (np.array([[1, 0, -1], [0, 1, 2], [1, 1, 0], [0, 0, 1]], f),
                    np.array([[[1, 0], [0, 1], [-1, 0]], [[0, 1], [1, 0], [0, 1]]], f),
                    np.array([[0], [1], [0], [1]], np.int64), None,
                    [[[2, 0]], [[1, 2]], [[1, 1]], [[0, 1]]]),
        # Unit-vector rows select one weight row each, then the bias row is added.
        "_with_bias": (np.array([[1, 0], [0, 1]], f),
                       np.array([[[1, 0], [0, 1]], [[0, 1], [1, 0]], [[1, 1], [0, 0]]], f),
                       np.array([[0, 1], [2, 0]], np.int64),
                       np.array([[0.1, 0.2], [0.3, 0.0], [0.5, 0.5]], f),
                       [[[1.1, 0.2], [0.3, 1.0]], [[0.5, 0.5], [0.1, 1.2]]]),
        # W = 0..11 as [3,2,2]: W0 = [[0,1],[2,3]], W2 = [[8,9],[10,11]].
        # [1,2]@W0 = [4,7]; [3,4]@W0 = [8,15]; [5,6]@W2 = [100,111]; [7,8]@W2 = [136,151].
        "_with_unused_group": (np.array([[1, 2], [3, 4], [5, 6], [7, 8]], f),
                               np.arange(12, dtype=f).reshape(3, 2, 2),
                               np.array([[0], [0], [2], [2]], np.int64), None,
                               [[[4, 7]], [[8, 15]], [[100, 111]], [[136, 151]]]),
        # W0 = [[1,2,3],[4,5,6]]: [1,2] -> [9,12,15]; [3,4] -> [19,26,33]; [5,6] -> [29,40,51].
        "_single_group": (np.array([[1, 2], [3, 4], [5, 6]], f),
                          np.array([[[1, 2, 3], [4, 5, 6]]], f),
                          np.zeros((3, 1), np.int64), None,
                          [[[9, 12, 15]], [[19, 26, 33]], [[29, 40, 51]]]),
    }


@pytest.mark.parametrize("name", list(_grouped_examples()))
@pytest.mark.parametrize("dtype", [np.float16, np.float32, np.float64])
def test_grouped_page_examples_hand_derived(name, dtype):
    x, w, gi, bias, want = _grouped_examples()[name]
    b = None if bias is None else bias.astype(dtype)
    got = ORC.grouped_matmul(x.astype(dtype), w.astype(dtype), gi, b)
    want = np.array(want, np.float64)
    # Every term is a small integer; the only inexact values are the bias
    # entries, which are exact as the float of type `dtype` widened to float64.
    tol = 0 if bias is None else 1e-3 if dtype == np.float16 else 1e-7
    assert got.shape == want.shape and np.max(np.abs(got - want)) <= tol


def test_grouped_empty_shapes_and_invalid_index():
    x = np.arange(6, dtype=np.float32).reshape(2, 3)
    w = np.arange(24, dtype=np.float32).reshape(2, 3, 4)
    assert ORC.grouped_matmul(x, w, np.empty((2, 0), np.int64)).shape == (2, 0, 4)
    assert ORC.grouped_matmul(np.empty((0, 3), np.float32), w, np.empty((0, 2), np.int64)).shape == (0, 2, 4)
    for bad in (-1, 2):
        with pytest.raises(IndexError):
            ORC.grouped_matmul(x, w, np.array([[0], [bad]], np.int64))


def test_grouped_one_group_equals_gemm_with_bias():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 5))
    w = rng.standard_normal((1, 5, 6))
    bias = rng.standard_normal((1, 6))
    got = ORC.grouped_matmul(x, w, np.zeros((7, 1), np.int32), bias)[:, 0, :]
    want = ORC.gemm(x, w[0], bias)
    assert np.allclose(got, want, rtol=0, atol=1e-12)


def test_grouped_identity_and_permutation_weights():
    rng = np.random.default_rng(4)
    M, K, G, S = 6, 4, 3, 2
    x = rng.integers(-5, 6, size=(M, K)).astype(np.float32)
    perms = [np.eye(K)[list(p)] for p in ((0, 1, 2, 3), (3, 2, 1, 0), (1, 0, 3, 2))]
    w = np.stack(perms).astype(np.float32)   # weights[g] is a permutation matrix
    gi = rng.integers(0, G, size=(M, S)).astype(np.int64)
    out = ORC.grouped_matmul(x, w, gi)
    for m in range(M):
        for i in range(S):
            assert np.array_equal(out[m, i], x[m] @ perms[gi[m, i]])
            # a permutation matrix only reorders: the multiset of values is kept
            assert sorted(out[m, i].tolist()) == sorted(x[m].tolist())


def test_grouped_brute_force():
    rng = np.random.default_rng(6)
    M, K, N, G, S = 5, 3, 4, 3, 2
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    w = rng.integers(-4, 5, size=(G, K, N)).astype(np.float32)
    bias = rng.integers(-4, 5, size=(G, N)).astype(np.float32)
    gi = rng.integers(0, G, size=(M, S)).astype(np.int32)
    got = ORC.grouped_matmul(x, w, gi, bias)
    for m in range(M):
        for i in range(S):
            g = int(gi[m, i])
            for n in range(N):
                s = float(bias[g, n])
                for k in range(K):
                    s += float(x[m, k]) * float(w[g, k, n])
                assert got[m, i, n] == s


# ------------------------------------------------------------------ weight-only quantized experts
# ("GroupedMatMul - 29", Summary: DequantizeLinear of the weights, then GroupedMatMul)

def test_dequantize_worked_values():
    # (q - zp) * scale by hand: (-128 - 3) * 0.5 = -65.5, (127 + 1) * 1.5 = 192,
    # (5 - 3) * 0.5 = 1, (-5 + 1) * 1.5 = -6; all exact in bfloat16.
    q = np.array([[[-128, 127], [5, -5]]], dtype=np.int8)
    zp = np.array([[[3, -1]]], dtype=np.int8)
    scale = np.array([[[0.5, 1.5]]])
    got = ORC.dequantize_linear(q, scale, zp, None, "bf16")
    assert got.tolist() == [[[-65.5, 192.0], [1.0, -6.0]]]
    # uint8 with the default zero point 0
    qu = np.array([[[0, 255]]], dtype=np.uint8)
    assert ORC.dequantize_linear(qu, np.array([[[2.0, 0.25]]]), None, 1, "f16").tolist() == [[[0.0, 63.75]]]


def test_unpack_4bit_layout():
    # Two values per byte, the even element in the low nibble: 0x7F holds
    # (15, 7), 0x80 holds (0, 8), 0x0F holds (15, 0); as int4, nibbles of 8
    # and above are negative (15 -> -1, 8 -> -8).
    b = np.array([[0x7F, 0x80, 0x0F]], dtype=np.uint8)
    assert oracle.unpack_4bit(b, False).tolist() == [[15, 7, 0, 8, 15, 0]]
    assert oracle.unpack_4bit(b, True).tolist() == [[-1, 7, 0, -8, -1, 0]]
    assert oracle.unpack_4bit(b, True).dtype == np.int8 and oracle.unpack_4bit(b, False).dtype == np.uint8


def test_dequantize_4bit_worked_values():
    # int4 [-8, 7] and uint4 [0, 15] by hand: (-8 - 3) * 0.5 = -5.5,
    # (7 + 1) * 1.25 = 10, (15 - 9) * 0.75 = 4.5, (0 - 9) * 0.75 = -6.75.
    q = oracle.unpack_4bit(np.array([[[0x78]]], dtype=np.uint8), True)      # [[[-8, 7]]]
    zp = oracle.unpack_4bit(np.array([[[0xF3]]], dtype=np.uint8), True)     # [[[3, -1]]]
    assert ORC.dequantize_linear(q, np.array([[[0.5, 1.25]]]), zp, None, "bf16").tolist() == [[[-5.5, 10.0]]]
    qu = oracle.unpack_4bit(np.array([[[0x0F]]], dtype=np.uint8), False)    # [[[15, 0]]]
    zu = oracle.unpack_4bit(np.array([[[0x99]]], dtype=np.uint8), False)    # [[[9, 9]]]
    assert ORC.dequantize_linear(qu, np.array([[[0.75, 0.75]]]), zu, None, "f16").tolist() == [[[4.5, -6.75]]]


def test_dequantize_rounds_once_to_the_scale_type():
    # 255 * 1.5 = 382.5: bfloat16 spacing is 2 in [256, 512), so 382; exact in float16.
    q = np.array([[[127]]], dtype=np.int8)
    zp = np.array([[[-128]]], dtype=np.int8)
    s = np.array([[[1.5]]])
    assert ORC.dequantize_linear(q, s, zp, None, "bf16").item() == 382.0
    assert ORC.dequantize_linear(q, s, zp, None, "f16").item() == 382.5
    # ties go to the even neighbour: 174 * 1.5 = 261 -> 260, 178 * 1.5 = 267 -> 268
    for diff, want in ((174, 260.0), (178, 268.0), (-174, -260.0)):
        qq = np.array([[[diff - 128 if diff > 0 else diff + 127]]], dtype=np.int8)
        zz = np.array([[[-128 if diff > 0 else 127]]], dtype=np.int8)
        assert ORC.dequantize_linear(qq, s, zz, None, "bf16").item() == want


def test_bf16_rounding_matches_torch_conversion():
    # The bfloat16 rounding written out in the oracle against torch's float32 ->
    # bfloat16 conversion (round to nearest even), over every (q - zp) in
    # [-255, 255] and a set of bfloat16 scales.
    torch = pytest.importorskip("torch")
    diffs = np.arange(-255, 256, dtype=np.float64)
    scales = torch.tensor(np.random.default_rng(40).uniform(-3, 3, 64), dtype=torch.float32).to(torch.bfloat16)
    scales = scales.double().numpy()
    prod = np.multiply.outer(diffs, scales)            # exact in float32 (<= 17 significant bits)
    ours = ORC.round_to_bf16(prod)
    ref = torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, ref)


def test_dequantize_blocks_brute_force():
    rng = np.random.default_rng(41)
    G, K, N, block = 2, 7, 3, 3                        # Kb = 3, last block partial
    q = rng.integers(-128, 128, size=(G, K, N)).astype(np.int8)
    zp = rng.integers(-20, 21, size=(G, 3, N)).astype(np.int8)
    scale = rng.integers(1, 9, size=(G, 3, N)) / 8.0   # exact, products exact in every type
    got = ORC.dequantize_linear(q, scale, zp, block, "f32")
    for g in range(G):
        for k in range(K):
            for n in range(N):
                b = k // block
                assert got[g, k, n] == (int(q[g, k, n]) - int(zp[g, b, n])) * float(scale[g, b, n])


def test_grouped_qweights_reduces_to_grouped_matmul():
    # block = K, unit scales and zero points 0: the weights are the integers themselves.
    rng = np.random.default_rng(42)
    M, K, N, G, S = 6, 5, 4, 3, 2
    x = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    q = rng.integers(-128, 128, size=(G, K, N)).astype(np.int8)
    gi = rng.integers(0, G, size=(M, S)).astype(np.int32)
    bias = rng.integers(-4, 5, size=(G, N)).astype(np.float32)
    got = ORC.grouped_matmul_qweights(x, q, np.ones((G, 1, N)), None, K, gi, bias, "bf16")
    assert np.array_equal(got, ORC.grouped_matmul(x, q.astype(np.float32), gi, bias))
    # a per-column scale of 2**-3 scales every output of that column (bias excluded)
    s = np.ones((G, 1, N))
    s[:, :, 1] = 0.125
    got2 = ORC.grouped_matmul_qweights(x, q, s, None, K, gi, None, "bf16")
    ref2 = ORC.grouped_matmul(x, q.astype(np.float32), gi, None)
    assert np.array_equal(got2[:, :, 1], ref2[:, :, 1] * 0.125)
    assert np.array_equal(got2[:, :, 0], ref2[:, :, 0])


def test_grouped_qweights_uses_each_groups_parameters():
    # two groups with the same quantized weights but different zero points:
    # outputs differ by (zp1 - zp0) * scale * sum(x) for every column
    x = np.array([[1.0, 2.0, 3.0]])
    q = np.zeros((2, 3, 2), dtype=np.int8)
    zp = np.array([[[1, 1]], [[4, 4]]], dtype=np.int8)
    s = np.full((2, 1, 2), 0.5)
    gi = np.array([[0, 1]], dtype=np.int64)
    out = ORC.grouped_matmul_qweights(x, q, s, zp, None, gi, None, "f16")
    assert out[0, 0].tolist() == [-3.0, -3.0]          # (0 - 1) * 0.5 * 6
    assert out[0, 1].tolist() == [-12.0, -12.0]        # (0 - 4) * 0.5 * 6


def test_dequantize_rejects_bad_shapes():
    q = np.zeros((1, 4, 2), dtype=np.int8)
    with pytest.raises(ValueError):
        ORC.dequantize_linear(q, np.ones((1, 1, 2)), None, 2, "bf16")      # needs [1, 2, 2]
    with pytest.raises(TypeError):
        ORC.dequantize_linear(q, np.ones((1, 1, 2)), np.zeros((1, 1, 2), dtype=np.uint8), None, "bf16")
    with pytest.raises(TypeError):
        ORC.dequantize_linear(q.astype(np.int16), np.ones((1, 1, 2)), None, None, "bf16")


# ------------------------------------------------------------------ error-bound denominators
# Hand values chosen so that each plausible slip changes the result: a
# negative alpha (|alpha| dropped -> negative values), a row whose terms
# cancel (|A @ B| instead of |A| @ |B| -> 0 there), and a broadcast C with
# negative entries (the |beta * C| term dropped or taken without abs).

def test_gemm_abs_scale_hand_values():
    A = np.array([[1.0, -2.0], [3.0, -4.0]])
    B = np.array([[-1.0, 2.0], [-0.5, -3.0]])
    # |A| @ |B| = [[2, 8], [5, 18]] while A @ B = [[0, 8], [-1, 18]].
    # |alpha| = 0.5, |beta| = 2, C = [[1, -1]] stretched over the rows:
    want = np.array([[3.0, 6.0], [4.5, 11.0]])
    C = np.array([[1.0, -1.0]])
    got = ORC.gemm_abs_scale(A, B, C, alpha=-0.5, beta=-2.0)
    assert np.array_equal(got, want)
    # the same through the transposition attributes
    assert np.array_equal(ORC.gemm_abs_scale(A.T.copy(), B.T.copy(), C, alpha=-0.5, beta=-2.0, transA=1, transB=1),
                          want)
    # C of shape (M, 1) stretched along the columns: + 2 * [[1], [3]]
    got = ORC.gemm_abs_scale(A, B, np.array([[1.0], [-3.0]]), alpha=-0.5, beta=-2.0)
    assert np.array_equal(got, np.array([[3.0, 6.0], [8.5, 15.0]]))
    # C absent: the product term alone
    assert np.array_equal(ORC.gemm_abs_scale(A, B, None, alpha=-0.5), np.array([[1.0, 4.0], [2.5, 9.0]]))
    # and the value itself has the cancellation: Y[0, 0] = -0.5 * 0 - 2 * 1
    assert ORC.gemm(A, B, C, alpha=-0.5, beta=-2.0)[0, 0] == -2.0


def test_matmul_abs_scale_hand_values():
    # A [2, 1, 2] against B [2, 1] (1-D promotion of neither; batch of A only):
    # batch 0: |1|*|-1| + |-2|*|-0.5| = 2 (the product is -1 + 1 = 0);
    # batch 1: |-3|*|-1| + |4|*|-0.5| = 5 (the product is 3 - 2 = 1).
    A = np.array([[[1.0, -2.0]], [[-3.0, 4.0]]])
    B = np.array([[-1.0], [-0.5]])
    assert np.array_equal(ORC.matmul_abs_scale(A, B), np.array([[[2.0]], [[5.0]]]))
    assert np.array_equal(ORC.matmul(A, B), np.array([[[0.0]], [[1.0]]]))
    # 1-D operands: |[1, -2]| . |[-1, -0.5]| = 2 with the promoted dims removed
    assert ORC.matmul_abs_scale(np.array([1.0, -2.0]), np.array([-1.0, -0.5])).shape == ()
    assert float(ORC.matmul_abs_scale(np.array([1.0, -2.0]), np.array([-1.0, -0.5]))) == 2.0


def test_grouped_abs_scale_hand_values():
    # x = [1, -1]; W0 = [[2], [3]], W1 = [[-1], [1]]; bias = [-0.5, 0.25].
    # (m=0, i=0) picks group 0: |1*2| + |-1*3| + |-0.5| = 5.5 (the value is -1.5);
    # (m=0, i=1) picks group 1: |1*-1| + |-1*1| + |0.25| = 2.25 (the value is -1.75).
    x = np.array([[1.0, -1.0]])
    w = np.array([[[2.0], [3.0]], [[-1.0], [1.0]]])
    gi = np.array([[0, 1]], np.int64)
    bias = np.array([[-0.5], [0.25]])
    assert np.array_equal(ORC.grouped_abs_scale(x, w, gi, bias), np.array([[[5.5], [2.25]]]))
    assert np.array_equal(ORC.grouped_matmul(x, w, gi, bias), np.array([[[-1.5], [-1.75]]]))
    assert np.array_equal(ORC.grouped_abs_scale(x, w, gi), np.array([[[5.0], [2.0]]]))
