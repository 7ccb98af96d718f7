"""Binding of the C++ oracle (TEST INFRASTRUCTURE ONLY).

``oracle/csrc/oracle.cpp`` restates the operator pages as plain C++ loops
(double accumulation, each sum taken over k in increasing order with no fused
multiply-add; exact integers modulo 2**n; float32 requantisation); this module
compiles it with g++ into ``oracle/csrc/liboracle.so`` and calls it through
ctypes.  The functions here only convert arrays (floats widened exactly to
float64, integers to 64-bit two's-complement patterns, 8-bit values and zero
points to int32), allocate the result, and turn the library's error codes into
the exceptions the numpy oracle raises.  Their names, arguments and results
match the numpy oracle's, so every pin runs against both.

Like the numpy oracle, this shares no code with the CUDA library; only
``tests/``, ``__graft_entry__`` and ``bench.py``'s CPU-baseline and reference
legs use it.  The thread count is ORACLE_THREADS if set, else every core
OpenMP reports; results do not depend on it.
"""

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "oracle.cpp")
LIB = os.path.join(HERE, "csrc", "liboracle.so")
# -ffp-contract=off: every product and sum is rounded separately (GCC fuses
# a*b+c by default on AArch64 otherwise).
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib_handle = None
_openmp = None

_ERRORS = {1: (ValueError, "shapes violate the operator's rules"),
           2: (TypeError, "element types violate the operator's type constraints"),
           3: (IndexError, "a group index lies outside [0, G)"),
           4: (ValueError, "integer Gemm result outside the range of T is undefined"),
           5: (ValueError, "invalid argument")}


def build(force=False):
    """Compile the C++ oracle (with OpenMP where the compiler has it); returns the library path."""
    global _openmp
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("no C++ compiler found to build the oracle")
    tmp = "%s.%d.tmp" % (LIB, os.getpid())
    err = ""
    for extra in (["-fopenmp"], []):
        r = subprocess.run([cxx, *CXXFLAGS, *extra, SRC, "-o", tmp], capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, LIB)
            _openmp = bool(extra)
            return LIB
        err = r.stderr
    raise RuntimeError("building the C++ oracle failed:\n" + err)


def _lib():
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            build()
            lib = ctypes.CDLL(LIB)
            I, L, P = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            D, F = ctypes.c_double, ctypes.c_float
            sigs = {
                "orc_num_threads": [I],
                "orc_matmul_shape": [I, P, I, P, P, P],
                "orc_matmul_f64": [I, P, P, I, P, P, P, I, I],
                "orc_matmul_u64": [I, P, P, I, P, P, P, I, I],
                "orc_gemm_shape": [L, L, L, L, I, I, I, P, P, P],
                "orc_gemm_f64": [L, L, P, L, L, P, I, P, P, D, D, I, I, P, I, I],
                "orc_gemm_u64": [L, L, P, L, L, P, I, P, P, D, D, I, I, P, I, I, I],
                "orc_requantize": [L, P, P, P, F, ctypes.c_int32, I, P],
                "orc_qlinear_matmul": [I, P, P, I, I, P, P, I, P, P, I,
                                       I, P, P, I, I, P, P, I, P, P, I,
                                       L, P, L, P, I, P, I],
                "orc_grouped_shape": [I, P, I, P, I, P, I, I, P, P],
                "orc_grouped_matmul_f64": [L, L, L, L, L, P, P, P, P, P, I, I],
                "orc_dequantize_linear": [I, P, P, I, I, P, P, I, P, P, I, L, I, P],
                "orc_round_to_type": [L, P, I, P],
            }
            for name, args in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = I
            _lib_handle = lib
    return _lib_handle


def num_threads():
    """Threads the oracle's loops use (ORACLE_THREADS, else every core OpenMP reports)."""
    return _lib().orc_num_threads(_threads())


def _threads():
    try:
        return int(os.environ.get("ORACLE_THREADS", "0"))
    except ValueError:
        return 0


def _check(status):
    if status != 0:
        exc, msg = _ERRORS.get(status, (RuntimeError, "oracle error %d" % status))
        raise exc(msg)


def _shape(x):
    return np.asarray(x.shape, dtype=np.int64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(x):
    x = np.asarray(x)
    if x.dtype.kind != "f":
        raise TypeError("expected a floating-point array, got %s" % x.dtype)
    return np.ascontiguousarray(x, dtype=np.float64)     # exact widening


def _u64(x):
    x = np.asarray(x)
    if x.dtype.kind == "i":
        return np.ascontiguousarray(x.astype(np.int64).view(np.uint64))
    return np.ascontiguousarray(x.astype(np.uint64))


def _from_u64(y, dtype):
    dtype = np.dtype(dtype)
    return y.astype(np.dtype("u%d" % dtype.itemsize)).view(dtype)


def _is_int(x):
    return np.asarray(x).dtype.kind in "iu"


# ------------------------------------------------------------------ MatMul

def matmul_output_shape(a_shape, b_shape):
    a_shape = np.asarray(a_shape, dtype=np.int64)
    b_shape = np.asarray(b_shape, dtype=np.int64)
    nd = ctypes.c_int()
    out = np.zeros(20, dtype=np.int64)
    _check(_lib().orc_matmul_shape(len(a_shape), _ptr(a_shape), len(b_shape), _ptr(b_shape), ctypes.byref(nd),
                                   _ptr(out)))
    return tuple(int(v) for v in out[:nd.value])


def _matmul(A, B, absval):
    A = np.asarray(A)
    B = np.asarray(B)
    if _is_int(A) or _is_int(B):
        if A.dtype != B.dtype:
            raise TypeError("MatMul operands must share one type T")
        if absval:
            raise TypeError("the error-bound denominator is defined for float operands")
        shape = matmul_output_shape(A.shape, B.shape)
        a, b = _u64(A), _u64(B)
        Y = np.zeros(shape, dtype=np.uint64)
        sa, sb = _shape(A), _shape(B)
        _check(_lib().orc_matmul_u64(A.ndim, _ptr(sa), _ptr(a), B.ndim, _ptr(sb), _ptr(b), _ptr(Y),
                                     8 * A.dtype.itemsize, _threads()))
        return _from_u64(Y, A.dtype)
    a, b = _f64(A), _f64(B)
    shape = matmul_output_shape(A.shape, B.shape)
    Y = np.zeros(shape, dtype=np.float64)
    sa, sb = _shape(A), _shape(B)
    _check(_lib().orc_matmul_f64(A.ndim, _ptr(sa), _ptr(a), B.ndim, _ptr(sb), _ptr(b), _ptr(Y), int(absval),
                                 _threads()))
    return Y


def matmul(A, B):
    """Y = A @ B with numpy.matmul semantics (float64 for floats, exact modulo 2**n for integers)."""
    return _matmul(A, B, False)


def matmul_abs_scale(A, B):
    """sum_k |A[b,i,k]| |B[b,k,j]| in float64: the per-element float error-bound denominator."""
    return _matmul(A, B, True)


# ------------------------------------------------------------------ Gemm

def _gemm_dims(A, B, C, transA, transB):
    if A.ndim != 2 or B.ndim != 2:
        raise ValueError("Gemm operands A and B must be 2-D")
    M, N = ctypes.c_int64(), ctypes.c_int64()
    cs = _shape(C) if C is not None else np.zeros(0, np.int64)
    _check(_lib().orc_gemm_shape(A.shape[0], A.shape[1], B.shape[0], B.shape[1], int(bool(transA)),
                                 int(bool(transB)), C.ndim if C is not None else -1, _ptr(cs),
                                 ctypes.byref(M), ctypes.byref(N)))
    return M.value, N.value, cs


def gemm_output_shape(a_shape, b_shape, transA=0, transB=0):
    if len(a_shape) != 2 or len(b_shape) != 2:
        raise ValueError("Gemm operands A and B must be 2-D")
    M, N = ctypes.c_int64(), ctypes.c_int64()
    _check(_lib().orc_gemm_shape(a_shape[0], a_shape[1], b_shape[0], b_shape[1], int(bool(transA)),
                                 int(bool(transB)), -1, None, ctypes.byref(M), ctypes.byref(N)))
    return (M.value, N.value)


def _gemm(A, B, C, alpha, beta, transA, transB, absval):
    A = np.asarray(A)
    B = np.asarray(B)
    C = None if C is None else np.asarray(C)
    M, N, cs = _gemm_dims(A, B, C, transA, transB)
    cnd = C.ndim if C is not None else -1
    if _is_int(A):
        if B.dtype != A.dtype or (C is not None and C.dtype != A.dtype):
            raise TypeError("Gemm operands must share one type T")
        if absval:
            raise TypeError("the error-bound denominator is defined for float operands")
        Y = np.zeros((M, N), dtype=np.uint64)
        a, b = _u64(A), _u64(B)
        c = None if C is None else _u64(C)
        _check(_lib().orc_gemm_u64(A.shape[0], A.shape[1], _ptr(a), B.shape[0], B.shape[1], _ptr(b), cnd,
                                   _ptr(cs), _ptr(c), float(alpha), float(beta), int(bool(transA)),
                                   int(bool(transB)), _ptr(Y), 8 * A.dtype.itemsize, int(A.dtype.kind == "i"),
                                   _threads()))
        return _from_u64(Y, A.dtype)
    a, b = _f64(A), _f64(B)
    c = None if C is None else _f64(C)
    Y = np.zeros((M, N), dtype=np.float64)
    _check(_lib().orc_gemm_f64(A.shape[0], A.shape[1], _ptr(a), B.shape[0], B.shape[1], _ptr(b), cnd, _ptr(cs),
                               _ptr(c), float(alpha), float(beta), int(bool(transA)), int(bool(transB)), _ptr(Y),
                               int(absval), _threads()))
    return Y


def gemm(A, B, C=None, alpha=1.0, beta=1.0, transA=0, transB=0):
    """Y = alpha * A' @ B' + beta * C  (float64 for float T, exact mod 2**n for integer T)."""
    return _gemm(A, B, C, alpha, beta, transA, transB, False)


def gemm_abs_scale(A, B, C=None, alpha=1.0, beta=1.0, transA=0, transB=0):
    """|alpha| * sum_k |A'[i,k]| |B'[k,j]| + |beta * C[i,j]|: the Gemm error-bound denominator."""
    return _gemm(A, B, C, alpha, beta, transA, transB, True)


# ------------------------------------------------------------------ QLinearMatMul

def _q8_code(x):
    dt = np.asarray(x).dtype
    return 0 if dt == np.int8 else 1 if dt == np.uint8 else -1


def _i32(x):
    return np.ascontiguousarray(np.asarray(x).astype(np.int32))


def _f32(x):
    return np.ascontiguousarray(np.asarray(x).astype(np.float32))


def requantize(acc, scale_a, scale_b, y_scale, y_zero_point, out_dtype):
    """The requantisation step on int32 accumulators, element by element (broadcast like numpy)."""
    acc = np.asarray(acc)
    if acc.dtype != np.int32:
        raise TypeError("the accumulator must already be int32 (wrapped modulo 2**32)")
    out_dtype = np.dtype(out_dtype)
    if out_dtype not in (np.dtype(np.int8), np.dtype(np.uint8)):
        raise TypeError("the output type must be int8 or uint8")
    acc_b, sa_b, sb_b = np.broadcast_arrays(acc, np.asarray(scale_a), np.asarray(scale_b))
    shape = acc_b.shape
    a, sa, sb = _i32(acc_b), _f32(sa_b), _f32(sb_b)
    y = np.zeros(shape, dtype=np.int32)
    _check(_lib().orc_requantize(a.size, _ptr(a), _ptr(sa), _ptr(sb),
                                 float(np.asarray(y_scale).astype(np.float32).reshape(())),
                                 int(np.asarray(y_zero_point).reshape(())), int(out_dtype == np.uint8), _ptr(y)))
    return y.astype(out_dtype)


def qlinear_matmul(a, a_scale, a_zero_point, b, b_scale, b_zero_point, y_scale, y_zero_point):
    """Quantized numpy.matmul of int8/uint8 operands; returns y of y_zero_point's type."""
    arrs = [np.asarray(x) for x in (a, a_scale, a_zero_point, b, b_scale, b_zero_point, y_scale, y_zero_point)]
    a, sa, za, b, sb, zb, ys, yz = arrs
    codes = [_q8_code(x) for x in (a, za, b, zb, yz)]
    shape = matmul_output_shape(a.shape, b.shape) if a.ndim and b.ndim else None
    if min(codes) < 0:
        raise TypeError("a, b, their zero points and y_zero_point must be int8 or uint8")
    if shape is None:
        raise ValueError("QLinearMatMul operands must have at least one dimension")
    y = np.zeros(shape, dtype=np.int32)
    conv = [_i32(a), _f32(sa), _i32(za), _i32(b), _f32(sb), _i32(zb), _f32(ys), _i32(yz)]
    shapes = [_shape(x) for x in arrs]
    _check(_lib().orc_qlinear_matmul(
        a.ndim, _ptr(shapes[0]), _ptr(conv[0]), codes[0],
        sa.ndim, _ptr(shapes[1]), _ptr(conv[1]),
        za.ndim, _ptr(shapes[2]), _ptr(conv[2]), codes[1],
        b.ndim, _ptr(shapes[3]), _ptr(conv[3]), codes[2],
        sb.ndim, _ptr(shapes[4]), _ptr(conv[4]),
        zb.ndim, _ptr(shapes[5]), _ptr(conv[5]), codes[3],
        ys.size, _ptr(conv[6]), yz.size, _ptr(conv[7]), codes[4], _ptr(y), _threads()))
    return y.astype(yz.dtype)


# ------------------------------------------------------------------ GroupedMatMul

def _grouped(input, weights, group_indices, bias, absval):
    x = np.asarray(input)
    w = np.asarray(weights)
    gi = np.asarray(group_indices)
    bias = None if bias is None else np.asarray(bias)
    ind = 0 if gi.dtype == np.int32 else 1 if gi.dtype == np.int64 else -1
    dims = np.zeros(5, dtype=np.int64)
    bs = _shape(bias) if bias is not None else np.zeros(0, np.int64)
    xs, ws, gs = _shape(x), _shape(w), _shape(gi)
    _check(_lib().orc_grouped_shape(x.ndim, _ptr(xs), w.ndim, _ptr(ws), gi.ndim, _ptr(gs), ind,
                                    bias.ndim if bias is not None else -1, _ptr(bs), _ptr(dims)))
    M, K, G, N, S = (int(v) for v in dims)
    xf, wf = _f64(x), _f64(w)
    bf = None if bias is None else _f64(bias)
    g64 = np.ascontiguousarray(gi.astype(np.int64))
    out = np.zeros((M, S, N), dtype=np.float64)
    _check(_lib().orc_grouped_matmul_f64(M, K, G, N, S, _ptr(xf), _ptr(wf), _ptr(g64), _ptr(bf), _ptr(out),
                                         int(absval), _threads()))
    return out


def grouped_matmul(input, weights, group_indices, bias=None):
    """output[m, i, :] = input[m, :] @ weights[g, :, :] (+ bias[g, :]),  g = group_indices[m, i]."""
    return _grouped(input, weights, group_indices, bias, False)


def grouped_abs_scale(input, weights, group_indices, bias=None):
    """|input[m]| @ |weights[g]| + |bias[g]| in float64: the float error-bound denominator."""
    return _grouped(input, weights, group_indices, bias, True)


# ------------------------------------------------------------------ weight-only quantized experts

T_CODES = {"bf16": 0, "f16": 1, "f32": 2, "f64": 3}


def round_to(x, t):
    """Round float64 values once to type t (nearest, ties to even), returned as float64."""
    if t not in T_CODES:
        raise ValueError("t must be one of %s" % (tuple(T_CODES),))
    xf = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    y = np.zeros(xf.shape, dtype=np.float64)
    _check(_lib().orc_round_to_type(xf.size, _ptr(xf), T_CODES[t], _ptr(y)))
    return y


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even), as float64."""
    return round_to(x, "bf16")


def dequantize_linear(weights_q, scale, zero_point=None, block=None, t="bf16"):
    """W[g, k, n] = T((weights_q[g, k, n] - zero_point[g, k//block, n]) * scale[g, k//block, n])."""
    q = np.asarray(weights_q)
    if t not in T_CODES:
        raise ValueError("t must be one of %s" % (tuple(T_CODES),))
    s = np.asarray(scale, dtype=np.float64)
    z = None if zero_point is None else np.asarray(zero_point)
    blk = 0 if block is None else int(block)
    qi, si = _i32(q), np.ascontiguousarray(s)
    zi = None if z is None else _i32(z)
    qs, ss = _shape(q), _shape(s)
    zs = _shape(z) if z is not None else np.zeros(0, np.int64)
    W = np.zeros(q.shape, dtype=np.float64) if q.ndim == 3 else np.zeros(0)
    _check(_lib().orc_dequantize_linear(q.ndim, _ptr(qs), _ptr(qi), _q8_code(q), s.ndim, _ptr(ss), _ptr(si),
                                        z.ndim if z is not None else -1, _ptr(zs), _ptr(zi),
                                        _q8_code(z) if z is not None else 0, blk, T_CODES[t], _ptr(W)))
    return W


def grouped_matmul_qweights(input, weights_q, scale, zero_point, block, group_indices, bias=None, t="bf16"):
    """GroupedMatMul(input, DequantizeLinear(weights_q, scale, zero_point), group_indices, bias)."""
    return grouped_matmul(input, dequantize_linear(weights_q, scale, zero_point, block, t), group_indices, bias)


def grouped_qweights_abs_scale(input, weights_q, scale, zero_point, block, group_indices, bias=None, t="bf16"):
    """The float error-bound denominator of grouped_matmul_qweights: |input| @ |W| + |bias|."""
    return grouped_abs_scale(input, dequantize_linear(weights_q, scale, zero_point, block, t), group_indices, bias)
