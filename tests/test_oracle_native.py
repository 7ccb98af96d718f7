"""The C++ oracle (oracle.native) against the numpy oracle on random inputs.

Both restate the pages independently (plain double-precision loops in C++;
numpy's float64 contraction in Python) and both are pinned by
tests/test_oracle_pins.py.  Here they must agree on random cases of every
operator and type: bit for bit for integers, QLinearMatMul and the
type roundings of DequantizeLinear; for floats within 1e-13 of the
error-bound denominator (both are float64 sums of the same exact products,
in different orders).
"""

import numpy as np
import pytest

import oracle
import oracle.native as nv

FTOL = 1e-13


def _close(a, b, scale):
    assert a.shape == b.shape
    assert np.all(np.abs(a - b) <= FTOL * (scale + 1e-300))


@pytest.mark.parametrize("sa,sb", [((7,), (7,)), ((9,), (3, 9, 5)), ((2, 3, 6, 5), (5,)), ((4, 1, 6, 3), (5, 3, 2)),
                                   ((33, 17), (17, 40)), ((1, 3, 8), (2, 1, 8, 4)), ((0, 4), (4, 3)), ((3, 0), (0, 2))])
def test_matmul_float_agrees(sa, sb):
    rng = np.random.default_rng(sum(sa) + 7 * sum(sb))
    A = rng.standard_normal(sa).astype(np.float32)
    B = rng.standard_normal(sb).astype(np.float32)
    scale = oracle.matmul_abs_scale(A, B)
    _close(nv.matmul(A, B), oracle.matmul(A, B), scale)
    _close(nv.matmul_abs_scale(A, B), scale, scale)


@pytest.mark.parametrize("dt", [np.int32, np.int64, np.uint32, np.uint64])
def test_matmul_integer_agrees(dt):
    rng = np.random.default_rng(3)
    info = np.iinfo(dt)
    for sa, sb in (((5, 9), (9, 4)), ((2, 3, 4), (4, 6)), ((6,), (2, 6, 3))):
        A = rng.integers(info.min, info.max, size=sa, dtype=dt, endpoint=True)
        B = rng.integers(info.min, info.max, size=sb, dtype=dt, endpoint=True)
        got, want = nv.matmul(A, B), oracle.matmul(A, B)
        assert got.dtype == want.dtype and np.array_equal(got, want)


@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("c_shape", [None, (), (1,), (23,), (1, 23), (19, 1), (19, 23)])
def test_gemm_float_agrees(tA, tB, c_shape):
    rng = np.random.default_rng(11 + 2 * tA + tB)
    M, K, N = 19, 37, 23
    A = rng.standard_normal((K, M) if tA else (M, K))
    B = rng.standard_normal((N, K) if tB else (K, N)).astype(np.float16)
    C = None if c_shape is None else rng.standard_normal(c_shape).astype(np.float32)
    kw = dict(alpha=-0.75, beta=1.5, transA=tA, transB=tB)
    scale = oracle.gemm_abs_scale(A, B, C, **kw)
    _close(nv.gemm(A, B, C, **kw), oracle.gemm(A, B, C, **kw), scale)
    _close(nv.gemm_abs_scale(A, B, C, **kw), scale, scale)


@pytest.mark.parametrize("dt", [np.int32, np.int64, np.uint32, np.uint64])
@pytest.mark.parametrize("alpha,beta", [(1.0, 1.0), (3.0, -2.0), (-7.0, 0.0)])
def test_gemm_integer_agrees(dt, alpha, beta):
    rng = np.random.default_rng(5)
    info = np.iinfo(dt)
    A = rng.integers(info.min, info.max, size=(6, 8), dtype=dt, endpoint=True)
    B = rng.integers(info.min, info.max, size=(5, 8), dtype=dt, endpoint=True)
    C = rng.integers(info.min, info.max, size=(1, 5), dtype=dt, endpoint=True)
    got = nv.gemm(A, B, C, alpha=alpha, beta=beta, transB=1)
    assert np.array_equal(got, oracle.gemm(A, B, C, alpha=alpha, beta=beta, transB=1))


@pytest.mark.parametrize("dt", [np.int32, np.int64, np.uint32])
def test_gemm_integer_non_integral_alpha_agrees(dt):
    rng = np.random.default_rng(8)
    A = rng.integers(0, 50, size=(7, 5)).astype(dt)
    B = rng.integers(0, 50, size=(5, 3)).astype(dt)
    C = rng.integers(0, 50, size=(7, 1)).astype(dt)
    got = nv.gemm(A, B, C, alpha=0.37, beta=1.25)
    assert np.array_equal(got, oracle.gemm(A, B, C, alpha=0.37, beta=1.25))


@pytest.mark.parametrize("t_a,t_b,t_y", [(np.int8, np.int8, np.int8), (np.uint8, np.uint8, np.uint8),
                                         (np.uint8, np.int8, np.int8), (np.int8, np.uint8, np.uint8)])
@pytest.mark.parametrize("gran", ["tensor", "row_col", "nd"])
def test_qlinear_agrees_bit_exact(t_a, t_b, t_y, gran):
    rng = np.random.default_rng(17)
    M, K, N = 21, 45, 13

    def q(t, shape):
        i = np.iinfo(t)
        return rng.integers(i.min, i.max, size=shape, endpoint=True).astype(t)
    if gran == "nd":
        a, b = q(t_a, (3, M, K)), q(t_b, (3, K, N))
        pa, pb = (3, M, 1), (3, 1, N)
    else:
        a, b = q(t_a, (M, K)), q(t_b, (K, N))
        pa, pb = ((), ()) if gran == "tensor" else ((M, 1), (1, N))
    sa = rng.uniform(0.003, 0.01, pa).astype(np.float32)
    sb = rng.uniform(0.003, 0.01, pb).astype(np.float16)
    za = rng.integers(-20, 21, pa).astype(t_a) if t_a == np.int8 else rng.integers(100, 150, pa).astype(t_a)
    zb = rng.integers(-20, 21, pb).astype(t_b) if t_b == np.int8 else rng.integers(100, 150, pb).astype(t_b)
    args = (a, sa, za, b, sb, zb, np.float32(0.05), t_y(3))
    got, want = nv.qlinear_matmul(*args), oracle.qlinear_matmul(*args)
    assert got.dtype == want.dtype and np.array_equal(got, want)
    # both saturate somewhere and not everywhere, so clamping is exercised
    info = np.iinfo(t_y)
    sat = np.mean((want == info.min) | (want == info.max))
    assert 0 < sat < 1


def test_requantize_agrees_on_near_ties():
    rng = np.random.default_rng(23)
    acc = rng.integers(-2 ** 31, 2 ** 31, size=4096, dtype=np.int64).astype(np.int32)
    acc[:64] = np.arange(-32, 32) * 2 + 1                         # odd values / 2: exact ties
    sa = rng.uniform(0.5, 2, 4096).astype(np.float32)
    sa[:64] = 1
    sb = np.ones(4096, np.float32)
    for ys, yz, t in ((2.0, 0, np.int8), (1.0e7, -9, np.int8), (3.3e6, 17, np.uint8)):
        got = nv.requantize(acc, sa, sb, np.float32(ys), t(yz), t)
        assert np.array_equal(got, oracle.requantize(acc, sa, sb, np.float32(ys), t(yz), t))


@pytest.mark.parametrize("with_bias", [False, True])
def test_grouped_agrees(with_bias):
    rng = np.random.default_rng(29)
    M, K, N, G, S = 17, 24, 11, 5, 3
    x = rng.standard_normal((M, K)).astype(np.float16)
    w = rng.standard_normal((G, K, N)).astype(np.float32)
    gi = rng.integers(0, G, (M, S)).astype(np.int32)
    bias = rng.standard_normal((G, N)) if with_bias else None
    scale = oracle.grouped_abs_scale(x, w, gi, bias)
    _close(nv.grouped_matmul(x, w, gi, bias), oracle.grouped_matmul(x, w, gi, bias), scale)
    _close(nv.grouped_abs_scale(x, w, gi, bias), scale, scale)
    with pytest.raises(IndexError):
        nv.grouped_matmul(x, w, np.full((M, S), G, np.int64))


@pytest.mark.parametrize("t", ["bf16", "f16", "f32", "f64"])
@pytest.mark.parametrize("block", [None, 4])
def test_dequantize_agrees_bit_exact(t, block):
    rng = np.random.default_rng(31)
    G, K, N = 3, 10, 7
    kb = 1 if block is None else -(-K // block)
    q = rng.integers(-128, 128, (G, K, N)).astype(np.int8)
    zp = rng.integers(-8, 9, (G, kb, N)).astype(np.int8)
    # scales that are values of T (bfloat16 ones have 8 significant bits)
    s = oracle.round_to(rng.uniform(-3, 3, (G, kb, N)).astype(np.float32).astype(np.float64), t)
    assert np.array_equal(nv.dequantize_linear(q, s, zp, block, t), oracle.dequantize_linear(q, s, zp, block, t))


@pytest.mark.parametrize("t", ["bf16", "f16"])
def test_type_rounding_agrees_over_the_whole_range(t):
    # float32 values (exact inputs for the numpy bfloat16 rounding) from far
    # below the smallest subnormal of T to beyond its largest finite value,
    # plus the exact midpoints between neighbouring values of T.
    rng = np.random.default_rng(37)
    lo, hi = (-140, 128) if t == "bf16" else (-27, 17)
    x = (rng.uniform(1, 2, 20000) * 2.0 ** rng.integers(lo, hi, 20000)).astype(np.float32)
    x[::2] *= -1
    with np.errstate(over="ignore"):
        v = oracle.round_to(x.astype(np.float64), t)
    fin = np.isfinite(v) & (v != 0)
    mids = ((v[fin][:-1] + v[fin][1:]) / 2).astype(np.float32)      # some are exact ties
    xs = np.concatenate([x, mids, np.array([0.0, -0.0, np.inf, -np.inf], np.float32)]).astype(np.float64)
    with np.errstate(over="ignore"):
        want = oracle.round_to(xs, t)
    assert np.array_equal(nv.round_to(xs, t), want)
