"""Gemm oracle (test infrastructure only).

Follows the Gemm operator page (onnx-light, ai.onnx Gemm since version 13),
its definition paragraph and its Inputs / Outputs sections:

* A' is A transposed when the attribute transA is non-zero, else A; likewise B'
  with transB.  A has shape (M, K), or (K, M) when transposed; B has shape
  (K, N), or (N, K) when transposed; Y has shape (M, N).
* Y = alpha * A' * B' + beta * C.
* C is optional; when it is absent the computation is done as if C were the
  scalar 0.  When present, C is unidirectionally broadcastable to (M, N).

Readings of points the page leaves open:

* Defaults are alpha = 1.0, beta = 1.0, transA = transB = 0; they are not
  printed, but the examples test_cc_gemm_default, test_cc_gemm_alpha,
  test_cc_gemm_beta and test_cc_gemm_default_scalar_bias only match with them.
* "Unidirectional broadcast" is read as numpy broadcasting in which only C may
  be stretched: C has at most two dimensions, right-aligned against (M, N),
  each equal to the target or 1.  This admits (), (1,), (N,), (1, N), (M, 1)
  and (M, N).
* Float types: the contraction is done in float64 and Y is returned unrounded.
  alpha and beta are float32 attributes, widened exactly.
* Integer types with integral alpha and beta: Y is computed exactly modulo
  2**n of T.  With a non-integral alpha or beta (the page does not say how a
  real-valued result becomes a T): the product A' @ B' is taken modulo 2**n
  as a T value, then r = alpha * acc + beta * C is evaluated in float64 (each
  product rounded, then the sum) and truncated toward zero.  Results outside
  T's range are undefined; the oracle raises ValueError for them.
"""

import numpy as np

from ._numeric import from_u64, is_integer_dtype, to_f64, to_u64


def gemm_output_shape(a_shape, b_shape, transA=0, transB=0):
    """(M, N) of Gemm, after checking the operand shapes against each other."""
    if len(a_shape) != 2 or len(b_shape) != 2:
        raise ValueError("Gemm operands A and B must be 2-D")
    M, K = (a_shape[1], a_shape[0]) if transA else (a_shape[0], a_shape[1])
    K2, N = (b_shape[1], b_shape[0]) if transB else (b_shape[0], b_shape[1])
    if K != K2:
        raise ValueError("contraction sizes differ: %d vs %d" % (K, K2))
    return (M, N)


def _broadcast_c(C, M, N):
    """C stretched to (M, N) under the unidirectional rule, or an error."""
    C = np.asarray(C)
    if C.ndim > 2:
        raise ValueError("C has more dimensions than Y")
    target = (M, N)[2 - C.ndim:]
    for dc, dt in zip(C.shape, target):
        if dc != dt and dc != 1:
            raise ValueError("C of shape %s is not unidirectionally broadcastable to %s"
                             % (C.shape, (M, N)))
    return np.broadcast_to(C.reshape((1,) * (2 - C.ndim) + C.shape), (M, N))


def _is_integral(x):
    xf = float(np.float32(x))
    return np.isfinite(xf) and xf == np.floor(xf)


def _integer_gemm_real(P, A_dtype, C, alpha, beta, M, N):
    """trunc(alpha * acc + beta * C) in float64 for an integer T (non-integral alpha/beta)."""
    acc = from_u64(P, A_dtype).astype(np.float64)          # the wrapped T value, rounded to float64
    r = np.float64(np.float32(alpha)) * acc
    if C is not None:
        r = r + np.float64(np.float32(beta)) * np.asarray(_broadcast_c(C, M, N)).astype(np.float64)
    t = np.trunc(r)
    bits = np.dtype(A_dtype).itemsize * 8
    lo, hi = (-(2.0 ** (bits - 1)), 2.0 ** (bits - 1)) if np.issubdtype(A_dtype, np.signedinteger) else (0.0, 2.0 ** bits)
    if not np.all((t >= lo) & (t < hi)):
        raise ValueError("integer Gemm result outside the range of %s is undefined" % np.dtype(A_dtype))
    if np.issubdtype(A_dtype, np.signedinteger):
        return t.astype(np.int64).astype(A_dtype)
    return np.array([int(v) for v in t.ravel()], dtype=np.uint64).reshape(t.shape).astype(A_dtype)


def gemm(A, B, C=None, alpha=1.0, beta=1.0, transA=0, transB=0):
    """Y = alpha * A' @ B' + beta * C  (float64 for float T, exact mod 2**n for integer T)."""
    A = np.asarray(A)
    B = np.asarray(B)
    M, N = gemm_output_shape(A.shape, B.shape, transA, transB)
    Ap = A.T if transA else A
    Bp = B.T if transB else B
    if is_integer_dtype(A.dtype):
        if B.dtype != A.dtype or (C is not None and np.asarray(C).dtype != A.dtype):
            raise TypeError("Gemm operands must share one type T")
        P = np.matmul(to_u64(Ap), to_u64(Bp))  # uint64: wraps modulo 2**64
        if not (_is_integral(alpha) and _is_integral(beta)):
            return _integer_gemm_real(P, A.dtype, C, alpha, beta, M, N)
        a_int = np.uint64(int(np.float32(alpha)) % (1 << 64))
        b_int = np.uint64(int(np.float32(beta)) % (1 << 64))
        Y = a_int * P
        if C is not None:
            Y = Y + b_int * to_u64(_broadcast_c(C, M, N))
        return from_u64(Y, A.dtype)
    P = np.matmul(to_f64(Ap), to_f64(Bp))
    Y = np.float64(np.float32(alpha)) * P
    if C is not None:
        Y = Y + np.float64(np.float32(beta)) * to_f64(_broadcast_c(C, M, N))
    return Y


def gemm_abs_scale(A, B, C=None, alpha=1.0, beta=1.0, transA=0, transB=0):
    """|alpha| * sum_k |A'[i,k]| |B'[k,j]| + |beta * C[i,j]| in float64.

    Denominator of the per-element float error bound for Gemm.
    """
    A = np.abs(to_f64(np.asarray(A)))
    B = np.abs(to_f64(np.asarray(B)))
    M, N = gemm_output_shape(A.shape, B.shape, transA, transB)
    Ap = A.T if transA else A
    Bp = B.T if transB else B
    S = abs(float(np.float32(alpha))) * np.matmul(Ap, Bp)
    if C is not None:
        S = S + abs(float(np.float32(beta))) * np.abs(to_f64(_broadcast_c(C, M, N)))
    return S
