"""MatMul oracle (test infrastructure only).

Follows the MatMul operator page (onnx-light, ai.onnx MatMul since version 13):
its summary defines the operator as the matrix product with the behaviour of
numpy.matmul, the output having the input type T; the type-constraint section lists
T in {bfloat16, double, float, float16, int32, int64, uint32, uint64}.  The
numpy.matmul rules that the page's worked examples exercise are written out
here step by step:

1. A 1-D first operand of length K is promoted to a [1, K] matrix and the
   promoted dimension is removed from the result (examples test_cc_matmul_1d_1d,
   test_cc_matmul_1d_3d, test_cc_matmul_vector_matrix).
2. A 1-D second operand of length K is promoted to a [K, 1] matrix and the
   promoted dimension is removed (test_cc_matmul_1d_1d, test_cc_matmul_4d_1d).
3. All dimensions but the last two are batch dimensions; they are aligned from
   the right, a missing dimension counts as 1, and each pair must be equal or
   contain a 1, which is stretched (test_cc_matmul_batch_broadcast,
   test_cc_matmul_bcast, test_cc_matmul_4d).
4. For every batch index b:  Y[b, i, j] = sum_k A[b, i, k] * B[b, k, j].

Float inputs are contracted in float64 and returned unrounded; integer inputs
are contracted exactly modulo 2**n of their type (see ``_numeric``).
"""

import itertools

import numpy as np

from ._numeric import from_u64, is_integer_dtype, to_f64, to_u64


def _broadcast_batch(sa, sb):
    """Right-aligned broadcast of two batch shapes (numpy rule, step 3).

    Returns the broadcast shape and both shapes left-padded with 1s.
    """
    n = max(len(sa), len(sb))
    sa = (1,) * (n - len(sa)) + tuple(sa)
    sb = (1,) * (n - len(sb)) + tuple(sb)
    out = []
    for da, db in zip(sa, sb):
        if da == db or db == 1:
            out.append(da)
        elif da == 1:
            out.append(db)
        else:
            raise ValueError("batch dimensions %s and %s do not broadcast" % (sa, sb))
    return tuple(out), sa, sb


def matmul_output_shape(a_shape, b_shape):
    """Shape of numpy.matmul(A, B) for operand shapes ``a_shape``, ``b_shape``."""
    a_shape, b_shape = tuple(a_shape), tuple(b_shape)
    if len(a_shape) == 0 or len(b_shape) == 0:
        raise ValueError("MatMul operands must have at least one dimension")
    pa = (1,) + a_shape if len(a_shape) == 1 else a_shape
    pb = b_shape + (1,) if len(b_shape) == 1 else b_shape
    if pa[-1] != pb[-2]:
        raise ValueError("contraction sizes differ: %d vs %d" % (pa[-1], pb[-2]))
    batch, _, _ = _broadcast_batch(pa[:-2], pb[:-2])
    out = batch
    if len(a_shape) > 1:
        out = out + (pa[-2],)
    if len(b_shape) > 1:
        out = out + (pb[-1],)
    return out


def _matmul_impl(A, B, contract2d, result_dtype):
    A = np.asarray(A)
    B = np.asarray(B)
    out_shape = matmul_output_shape(A.shape, B.shape)
    # Steps 1-2: promote 1-D operands.
    A2 = A.reshape((1,) + A.shape) if A.ndim == 1 else A
    B2 = B.reshape(B.shape + (1,)) if B.ndim == 1 else B
    # Step 3: broadcast the batch dimensions.
    batch, ba, bb = _broadcast_batch(A2.shape[:-2], B2.shape[:-2])
    A3 = np.broadcast_to(A2.reshape(ba + A2.shape[-2:]), batch + A2.shape[-2:])
    B3 = np.broadcast_to(B2.reshape(bb + B2.shape[-2:]), batch + B2.shape[-2:])
    M = A3.shape[-2]
    N = B3.shape[-1]
    # Step 4: one 2-D product per batch index (none if the batch is empty).
    Y = np.zeros(batch + (M, N), dtype=result_dtype)
    for idx in itertools.product(*[range(d) for d in batch]):
        Y[idx] = contract2d(A3[idx], B3[idx])
    return Y.reshape(out_shape)


def _contract_f64(a, b):
    return np.matmul(to_f64(a), to_f64(b))


def _contract_u64(a, b):
    return np.matmul(to_u64(a), to_u64(b))  # uint64 matmul wraps modulo 2**64


def matmul(A, B):
    """Y = A @ B with numpy.matmul semantics.

    Float operands (float16/float32/float64 arrays; bfloat16 data must be passed
    widened to float64 by the caller, which is exact) give a float64 result.
    Integer operands (int32/int64/uint32/uint64, both of the same type) give a
    result of that type, exact modulo 2**n.
    """
    A = np.asarray(A)
    B = np.asarray(B)
    if is_integer_dtype(A.dtype) or is_integer_dtype(B.dtype):
        if A.dtype != B.dtype:
            raise TypeError("MatMul operands must share one type T")
        Y = _matmul_impl(A, B, _contract_u64, np.uint64)
        return from_u64(Y, A.dtype)
    return _matmul_impl(A, B, _contract_f64, np.float64)


def matmul_abs_scale(A, B):
    """sum_k |A[b,i,k]| * |B[b,k,j]| in float64, shaped like ``matmul(A, B)``.

    This is the denominator of the per-element float error bound: the
    magnitude of the terms whose rounded sum the output is.
    """
    return _matmul_impl(np.abs(to_f64(np.asarray(A))), np.abs(to_f64(np.asarray(B))),
                        _contract_f64, np.float64)
