"""Weight-only quantized experts for GroupedMatMul (test infrastructure only).

"GroupedMatMul - 29" (onnx.ai), Summary, last paragraph: weight-only quantized
experts are expressed by applying DequantizeLinear, with the weights' scales
and zero points, to the quantized weights and passing the result to
GroupedMatMul; a runtime may fuse the two so that the dequantized [G, K, N]
weights are never formed.  The pages name DequantizeLinear without defining
it.  The reading used here (the plainest one):

* weights_q [G, K, N] of int8 or uint8, or of DequantizeLinear's 4-bit
  types int4 / uint4 (values in [-8, 7] / [0, 15]).  4-bit tensors are stored
  packed two per byte along their last axis, the even element in the low
  nibble (``unpack_4bit`` states the layout; the formula below sees the
  unpacked values).  scale and zero_point share one shape
  [G, Kb, N], Kb = ceil(K / block): element (g, k, n) uses entry
  (g, k // block, n), i.e. blocks of `block` consecutive k for each group and
  output column; block = K (Kb = 1) is one scale per group and column.
* W[g, k, n] = (weights_q[g, k, n] - zero_point[g, k // block, n])
               * scale[g, k // block, n],
  the difference an exact integer, the product rounded once (to nearest,
  ties to even) to T, the type of scale: bfloat16, float16, float or double.
  zero_point is optional (0) and has the type of weights_q.

Then output = GroupedMatMul(input, W, group_indices, bias) as in
``grouped_matmul``.  Values of type T are passed as float64 arrays holding
exactly representable values, with the type named by ``t``.
"""

import numpy as np

from .grouped_matmul import grouped_matmul, grouped_abs_scale

T_NAMES = ("bf16", "f16", "f32", "f64")


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even), as float64.

    Inputs must be exact in float32 (true of every (q - zp) * scale with a
    bfloat16 scale: at most 9 + 8 significant bits).  bfloat16 is the upper
    half of the float32 bit pattern; rounding adds 0x7FFF plus the lowest kept
    bit to the pattern and clears the lower half.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    if not np.array_equal(f.astype(np.float64), np.asarray(x, dtype=np.float64), equal_nan=True):
        raise ValueError("round_to_bf16 expects values exact in float32")
    bits = f.view(np.uint32).astype(np.uint64)
    finite = np.isfinite(f)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    out = np.where(finite, rounded.view(np.float32), f)
    return out.astype(np.float64)


def round_to(x, t):
    """Round float64 values once to type t (nearest, ties to even), returned as float64."""
    if t == "bf16":
        return round_to_bf16(x)
    if t == "f16":
        return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)
    if t == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if t == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError("t must be one of %s" % (T_NAMES,))


def unpack_4bit(packed, signed):
    """The 4-bit values stored in ``packed`` (uint8 [..., N/2]) as an int8
    (signed: int4, [-8, 7]) or uint8 (uint4, [0, 15]) array [..., N]: element
    2j of a row is the low nibble of byte j, element 2j + 1 its high nibble."""
    b = np.asarray(packed)
    if b.dtype != np.uint8:
        raise TypeError("packed 4-bit values arrive as uint8 bytes")
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int16)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    if signed:
        out = np.where(out >= 8, out - 16, out)
        return out.astype(np.int8)
    return out.astype(np.uint8)


def dequantize_linear(weights_q, scale, zero_point=None, block=None, t="bf16"):
    """W[g, k, n] = T((weights_q[g, k, n] - zero_point[g, k//block, n]) * scale[g, k//block, n])."""
    q = np.asarray(weights_q)
    if q.ndim != 3 or q.dtype not in (np.dtype(np.int8), np.dtype(np.uint8)):
        raise TypeError("weights_q must be an int8 or uint8 array [G, K, N]")
    G, K, N = q.shape
    block = K if block is None or block == 0 else int(block)
    if block < 1:
        raise ValueError("block must be positive")
    kb = -(-K // block)
    s = np.asarray(scale, dtype=np.float64)
    if s.shape != (G, kb, N):
        raise ValueError("scale must have shape [G, ceil(K/block), N] = %s" % ((G, kb, N),))
    if zero_point is None:
        z = np.zeros((G, kb, N), dtype=np.int64)
    else:
        z = np.asarray(zero_point)
        if z.dtype != q.dtype or z.shape != s.shape:
            raise TypeError("zero_point must have the type of weights_q and the shape of scale")
        z = z.astype(np.int64)
    kblk = np.arange(K) // block                       # quantization block of each k
    diff = q.astype(np.int64) - z[:, kblk, :]          # exact integers in [-255, 255]
    # The product of a 9-bit integer and a float64 value is exact in float64
    # for every T but double; round_to then rounds once.
    return round_to(diff.astype(np.float64) * s[:, kblk, :], t)


def grouped_matmul_qweights(input, weights_q, scale, zero_point, block, group_indices, bias=None, t="bf16"):
    """GroupedMatMul(input, DequantizeLinear(weights_q, scale, zero_point), group_indices, bias)."""
    w = dequantize_linear(weights_q, scale, zero_point, block, t)
    return grouped_matmul(input, w, group_indices, bias)


def grouped_qweights_abs_scale(input, weights_q, scale, zero_point, block, group_indices, bias=None, t="bf16"):
    """The float error-bound denominator of grouped_matmul_qweights: |input| @ |W| + |bias|."""
    w = dequantize_linear(weights_q, scale, zero_point, block, t)
    return grouped_abs_scale(input, w, group_indices, bias)
