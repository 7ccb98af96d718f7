"""QLinearMatMul oracle (test infrastructure only).

Follows the page "QLinearMatMul - version 10" (onnx-light operator page
source): its summary paragraph (numpy.matmul behaviour; the quantization
formula; round to nearest with ties to even; scale / zero-point shapes; the
overflow sentence), its Inputs section and its Type Constraints section.

What is computed, in the order the page gives it:

1. The real-valued product of the dequantised operands is
   x = sum_k a_scale * (a - a_zero_point) * b_scale * (b - b_zero_point),
   with the integer part accumulated first:
   acc = sum_k (a[.., m, k] - a_zp) * (b[.., k, n] - b_zp).
   The page says that no single product overflows and that the accumulation
   may overflow only in 32 bits: acc is therefore the exact integer sum
   reduced modulo 2**32 (two's complement int32).
2. y = saturate(round(x / y_scale) + y_zero_point), where round is
   round-to-nearest with ties to even and saturate clamps to the range of the
   output type T3 (int8: [-128, 127], uint8: [0, 255]).

Readings of points the page leaves open:

* x is evaluated in IEEE float32 as  s = a_scale * b_scale;  v = float(acc) * s;
  q = v / y_scale;  r = rint(q);  t = r + float(y_zero_point);
  y = min(max(t, qmin), qmax)  -- each step one correctly rounded float32
  operation, in this order.  This reproduces all twelve printed examples.
  min/max follow IEEE fmin/fmax, so a NaN quotient saturates to qmin.
* Scales printed as float16 on the page's examples are widened exactly to
  float32 first (the v10 text says tensor(float)).
* Per-row scales of a have M elements: shape [M] (a is 2-D) or
  a.shape[:-1] + (1,) for N-D a.  Per-column scales of b have N elements:
  shape [N] (b is 2-D) or b.shape[:-2] + (1, N) for N-D b.  The page's text
  gives the per-column vector K elements, which cannot index the columns of
  the [M, N] result; N elements is the reading that can.
  A scale and its zero point have the same shape; a one-element scale is per
  tensor.
"""

import numpy as np

from ._numeric import from_u64, to_u64
from .matmul import matmul, matmul_output_shape

_RANGE = {np.dtype(np.int8): (-128.0, 127.0), np.dtype(np.uint8): (0.0, 255.0)}


def _quant_param(p, operand_shape, per_row):
    """Broadcastable view of a scale or zero point of operand a (per_row) or b."""
    p = np.asarray(p)
    if p.size == 1:
        return p.reshape(())
    nd = len(operand_shape)
    if per_row:
        M = operand_shape[-2] if nd >= 2 else 1
        if p.ndim == 1 and nd == 2 and p.shape[0] == M:
            return p.reshape(M, 1)
        if p.ndim == nd and nd >= 2 and p.shape[-1] == 1 and p.shape[:-1] == tuple(operand_shape[:-1]):
            return p
        raise ValueError("per-row parameter of shape %s does not fit a of shape %s"
                         % (p.shape, tuple(operand_shape)))
    N = operand_shape[-1] if nd >= 2 else 1
    if p.ndim == 1 and nd == 2 and p.shape[0] == N:
        return p.reshape(1, N)
    if (p.ndim == nd and nd >= 2 and p.shape[-2] == 1 and p.shape[-1] == N
            and p.shape[:-2] == tuple(operand_shape[:-2])):
        return p
    raise ValueError("per-column parameter of shape %s does not fit b of shape %s"
                     % (p.shape, tuple(operand_shape)))


def requantize(acc, scale_a, scale_b, y_scale, y_zero_point, out_dtype):
    """Step 2 on int32 accumulators, as a fixed sequence of float32 operations."""
    out_dtype = np.dtype(out_dtype)
    qmin, qmax = _RANGE[out_dtype]
    f32 = np.float32
    acc = np.asarray(acc)
    if acc.dtype != np.int32:
        raise TypeError("the accumulator must already be int32 (wrapped modulo 2**32)")
    s = np.asarray(scale_a).astype(f32) * np.asarray(scale_b).astype(f32)
    v = acc.astype(f32) * s
    q = v / f32(np.asarray(y_scale).astype(f32).reshape(()))
    r = np.rint(q)                      # round half to even
    t = r + f32(np.asarray(y_zero_point).reshape(()))
    t = np.fmin(np.fmax(t, f32(qmin)), f32(qmax))
    return t.astype(out_dtype)


def qlinear_matmul(a, a_scale, a_zero_point, b, b_scale, b_zero_point, y_scale, y_zero_point):
    """Quantized numpy.matmul of int8/uint8 operands; returns y of y_zero_point's type."""
    a = np.asarray(a)
    b = np.asarray(b)
    for x, zp, name in ((a, a_zero_point, "a"), (b, b_zero_point, "b")):
        if x.dtype not in _RANGE:
            raise TypeError("%s must be int8 or uint8" % name)
        if np.asarray(zp).dtype != x.dtype:
            raise TypeError("%s and its zero point must share a type" % name)
    y_dtype = np.asarray(y_zero_point).dtype
    if y_dtype not in _RANGE:
        raise TypeError("y_zero_point must be int8 or uint8")
    if np.asarray(a_scale).shape != np.asarray(a_zero_point).shape or \
            np.asarray(b_scale).shape != np.asarray(b_zero_point).shape:
        raise ValueError("a scale and its zero point must have the same shape")
    if np.asarray(y_scale).size != 1 or np.asarray(y_zero_point).size != 1:
        raise ValueError("y_scale and y_zero_point are per tensor")
    out_shape = matmul_output_shape(a.shape, b.shape)

    # numpy.matmul promotion of 1-D operands (their parameters are per tensor).
    a2 = a.reshape((1,) + a.shape) if a.ndim == 1 else a
    b2 = b.reshape(b.shape + (1,)) if b.ndim == 1 else b
    za = _quant_param(a_zero_point, a.shape, True)
    zb = _quant_param(b_zero_point, b.shape, False)
    sa = _quant_param(a_scale, a.shape, True)
    sb = _quant_param(b_scale, b.shape, False)

    # Step 1: exact integer accumulation of the zero-point-shifted operands.
    ac = a2.astype(np.int64) - za.astype(np.int64)
    bc = b2.astype(np.int64) - zb.astype(np.int64)
    acc = from_u64(to_u64(matmul(ac, bc)), np.int32)   # exact, then modulo 2**32

    # Step 2: per-element scale product, broadcast like the operands' batch.
    scale_a = np.broadcast_to(sa, a2.shape[:-1] + (1,))
    scale_b = np.broadcast_to(sb, b2.shape[:-2] + (1, b2.shape[-1]))
    y = requantize(acc, scale_a, scale_b, y_scale, y_zero_point, y_dtype)
    return y.reshape(out_shape)

