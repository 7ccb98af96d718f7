"""Number-type helpers shared by the oracle modules (test infrastructure only).

Integer arithmetic follows numpy's wrap-around: a value of an n-bit integer
type is an element of Z / 2**n.  The oracle widens every integer operand to
uint64 (two's-complement bit pattern), does all sums and products in uint64,
where numpy wraps modulo 2**64 without error, and finally keeps the low n bits.
Because reduction modulo 2**n commutes with + and *, this gives the exact
result of the operation in the n-bit type, independent of summation order.
"""

import numpy as np

INT_TYPES = (np.int32, np.int64, np.uint32, np.uint64)
FLOAT_TYPES = (np.float16, np.float32, np.float64)


def is_integer_dtype(dt):
    return np.issubdtype(np.dtype(dt), np.integer)


def to_u64(x):
    """Two's-complement bit pattern of an integer array, widened to uint64."""
    x = np.asarray(x)
    if np.issubdtype(x.dtype, np.signedinteger):
        return x.astype(np.int64).view(np.uint64)
    return x.astype(np.uint64)


def from_u64(x, dtype):
    """Low bits of a uint64 array reinterpreted as ``dtype`` (wrap-around)."""
    dtype = np.dtype(dtype)
    x = np.asarray(x, dtype=np.uint64)
    bits = dtype.itemsize * 8
    if bits < 64:
        x = x & np.uint64((1 << bits) - 1)
    unsigned = np.dtype("u%d" % dtype.itemsize)
    return x.astype(unsigned).view(dtype)


def to_f64(x):
    """Exact widening of a float array (float16/float32/float64) to float64."""
    x = np.asarray(x)
    if not np.issubdtype(x.dtype, np.floating):
        raise TypeError("expected a floating-point array, got %s" % x.dtype)
    return x.astype(np.float64)
