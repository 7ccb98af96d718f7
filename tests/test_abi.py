"""C-ABI checks that need no GPU: the library loads, exports every function
include/mm.h declares, and its host-side shape inference and validation behave
as documented.  No call here reaches a kernel launch: every compute entry point
is called only with arguments that fail validation first, and the output-shape
helpers never touch device memory (the data pointers below are dummies).
"""

import ctypes
import os
import re

import pytest

import quantized_gemm_gb300 as qg
from quantized_gemm_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mm.h")

DUMMY = 0x1000  # never dereferenced: shape helpers and failing validation only


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qg._lib()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(mm_[a-z0-9_]+)\s*\(",
                                 src, flags=re.M)))


def test_header_declares_the_four_operators():
    names = _declared_functions()
    for n in ("mm_matmul", "mm_gemm", "mm_qlinear_matmul", "mm_grouped_matmul", "mm_get_device_status",
              "mm_grouped_matmul_workspace_size", "mm_qlinear_matmul_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_library_built_for_sm_103a_only():
    assert "arch=compute_103a,code=sm_103a" in qbuild.ARCH
    assert all("sm_100" not in a and "sm_90" not in a for a in qbuild.ARCH)


def T(shape, dtype=2, strides=None, data=DUMMY):
    d = qg.MMTensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.strides[i] = st
    return d


def _shape(lib, a, b):
    nd = ctypes.c_int32()
    sh = (ctypes.c_int64 * 8)()
    st = lib.mm_matmul_output_shape(ctypes.byref(a), ctypes.byref(b), ctypes.byref(nd), sh)
    return st, tuple(sh[i] for i in range(nd.value))


@pytest.mark.parametrize("sa,sb,want", [
    ((3,), (3,), ()), ((4,), (2, 4, 3), (2, 3)), ((2, 3), (3, 4), (2, 4)),
    ((2, 3, 4), (2, 4, 3), (2, 3, 3)), ((1, 2, 3, 4), (1, 2, 4, 3), (1, 2, 3, 3)),
    ((2, 3, 4, 5), (5,), (2, 3, 4)), ((2, 2, 3), (1, 3, 4), (2, 2, 4)), ((2, 3, 4), (4, 5), (2, 3, 5)),
    ((3,), (3, 2), (2,)), ((8, 32, 2048, 128), (1, 32, 128, 2048), (8, 32, 2048, 2048)),
    ((7, 1, 2, 3), (5, 3, 4), (7, 5, 2, 4)), ((0, 2, 3), (3, 4), (0, 2, 4)),
])
def test_matmul_output_shape_follows_numpy(lib, sa, sb, want):
    import numpy as np
    st, got = _shape(lib, T(sa), T(sb))
    assert st == 0 and got == want == np.matmul(np.zeros(sa), np.zeros(sb)).shape


@pytest.mark.parametrize("sa,sb", [((2, 3), (4, 2)), ((2, 2, 3), (3, 3, 2)), ((), (3,))])
def test_matmul_output_shape_rejects(lib, sa, sb):
    st, _ = _shape(lib, T(sa), T(sb))
    assert st == 2  # MM_ERR_SHAPE


def test_gemm_output_shape(lib):
    nd = ctypes.c_int32()
    sh = (ctypes.c_int64 * 8)()
    a, b = T((5, 3)), T((4, 5))
    assert lib.mm_gemm_output_shape(ctypes.byref(a), ctypes.byref(b), 1, 1, ctypes.byref(nd), sh) == 0
    assert (nd.value, sh[0], sh[1]) == (2, 3, 4)
    assert lib.mm_gemm_output_shape(ctypes.byref(a), ctypes.byref(b), 0, 0, ctypes.byref(nd), sh) == 2


def test_validation_errors_before_any_launch(lib):
    ref = ctypes.byref
    A, B = T((4, 8)), T((8, 16))
    # wrong output shape / type / layout
    assert lib.mm_matmul(ref(A), ref(B), ref(T((4, 15))), None) == 2
    assert lib.mm_matmul(ref(A), ref(B), ref(T((4, 16), dtype=1)), None) == 3
    assert lib.mm_matmul(ref(A), ref(B), ref(T((4, 16), strides=(1, 4))), None) == 2
    # mixed operand types, 8-bit types on MatMul
    assert lib.mm_matmul(ref(A), ref(T((8, 16), dtype=3)), ref(T((4, 16))), None) == 3
    assert lib.mm_matmul(ref(T((4, 8), dtype=8)), ref(T((8, 16), dtype=8)), ref(T((4, 16), dtype=8)), None) == 3
    # NULL data with elements, negative stride, rank > 8
    assert lib.mm_matmul(ref(T((4, 8), data=None)), ref(B), ref(T((4, 16))), None) == 1
    assert lib.mm_matmul(ref(T((4, 8), strides=(-8, 1))), ref(B), ref(T((4, 16))), None) == 1
    bad = T((2,) * 8)
    bad.ndim = 9
    assert lib.mm_matmul(ref(bad), ref(B), ref(T((4, 16))), None) == 1
    # Gemm: C not unidirectionally broadcastable, rank-3 operand, integer T with a non-finite alpha
    assert lib.mm_gemm(ref(A), ref(B), ref(T((3, 16))), 1.0, 1.0, 0, 0, ref(T((4, 16))), None) == 2
    assert lib.mm_gemm(ref(T((1, 4, 8))), ref(B), None, 1.0, 1.0, 0, 0, ref(T((4, 16))), None) == 2
    Ai, Bi, Yi = T((4, 8), dtype=4), T((8, 16), dtype=4), T((4, 16), dtype=4)
    assert lib.mm_gemm(ref(Ai), ref(Bi), None, float("nan"), 1.0, 0, 0, ref(Yi), None) == 4
    # GroupedMatMul: types, shapes, bias shape
    x, w, gi = T((6, 8), 0), T((3, 8, 16), 0), T((6, 2), 4)
    out = T((6, 2, 16), 0)
    assert lib.mm_grouped_matmul(ref(x), ref(w), ref(T((6, 2), 2)), None, ref(out), None, 0, None) == 3
    assert lib.mm_grouped_matmul(ref(x), ref(T((3, 7, 16), 0)), ref(gi), None, ref(out), None, 0, None) == 2
    assert lib.mm_grouped_matmul(ref(x), ref(w), ref(gi), ref(T((3, 15), 0)), ref(out), None, 0, None) == 2
    assert lib.mm_grouped_matmul(ref(x), ref(w), ref(gi), None, ref(T((6, 2, 16), 1)), None, 0, None) == 3


def test_qlinear_validation(lib):
    ref = ctypes.byref
    a, b, y = T((4, 8), 8), T((8, 16), 8), T((4, 16), 8)
    s0, z0 = T((), 2), T((), 8)
    ok = [a, s0, z0, b, s0, z0, s0, z0, y]
    # a per-row scale of the wrong length; a zero point of the wrong type; f64 scale
    bad_rows = [a, T((5,), 2), T((5,), 8), b, s0, z0, s0, z0, y]
    assert lib.mm_qlinear_matmul(*[ref(t) for t in bad_rows], None, 0, None) == 2
    bad_zp = [a, s0, T((), 9), b, s0, z0, s0, z0, y]
    assert lib.mm_qlinear_matmul(*[ref(t) for t in bad_zp], None, 0, None) == 3
    bad_scale = [a, T((), 3), z0, b, s0, z0, s0, z0, y]
    assert lib.mm_qlinear_matmul(*[ref(t) for t in bad_scale], None, 0, None) == 3
    # output type must be y_zero_point's
    bad_y = ok[:-1] + [T((4, 16), 9)]
    assert lib.mm_qlinear_matmul(*[ref(t) for t in bad_y], None, 0, None) == 3
    # per-column parameter must have N (not K) elements
    bad_cols = [a, s0, z0, b, T((8,), 2), T((8,), 8), s0, z0, y]
    assert lib.mm_qlinear_matmul(*[ref(t) for t in bad_cols], None, 0, None) == 2


def test_policy_and_status_strings(lib):
    assert lib.mm_set_path_policy(7) == 1
    assert lib.mm_set_path_policy(3) == 1          # MM_PATH_NONE is a result, not a policy
    for p in (1, 2, 4, 0):
        assert lib.mm_set_path_policy(p) == 0
    for s in range(9):
        assert lib.mm_status_string(s)
    assert qg.mm_version() == "0.1.0"


def test_grouped_qweights_4bit_validation(lib):
    # 4-bit weights and zero points (MM_I4 = 10, MM_U4 = 11, packed two per
    # byte): unit stride along N, N even and even outer strides, so that every
    # row starts on a byte boundary
    ref = ctypes.byref
    x, gi = T((6, 8), 0), T((6, 2), 4)
    call = lib.mm_grouped_matmul_qweights
    s16, out16 = T((3, 1, 16), 0), T((6, 2, 16), 0)

    def run(wq, s=s16, zp=None, out=out16):
        return call(ref(x), ref(wq), ref(s), None if zp is None else ref(zp), 0, ref(gi), None, ref(out), None, 0,
                    None)
    assert run(T((3, 8, 15), 10), T((3, 1, 15), 0), out=T((6, 2, 15), 0)) == 2            # odd N
    assert run(T((3, 8, 16), 10, strides=(256, 32, 2))) == 2                                 # N not unit-stride
    assert run(T((3, 8, 16), 10, strides=(136, 17, 1))) == 2                                 # odd row stride
    assert run(T((3, 8, 16), 11), zp=T((3, 1, 16), 11, strides=(17, 16, 1))) == 2           # zero point, odd stride
    assert run(T((3, 8, 16), 10), zp=T((3, 1, 16), 11)) == 3                                 # zero point of the other type
    assert run(T((3, 8, 16), 10), zp=T((3, 1, 16), 8)) == 3                                  # an 8-bit zero point
    # no other operator takes 4-bit values
    assert lib.mm_matmul(ref(T((4, 8), 10)), ref(T((8, 6), 10)), ref(T((4, 6), 10)), None) == 3
    assert lib.mm_grouped_matmul(ref(x), ref(T((3, 8, 16), 11)), ref(gi), None, ref(out16), None, 0, None) == 3


def test_grouped_qweights_validation(lib):
    # input bf16 [6,8]; int8 weights [3,8,16]; scales bf16 [3, ceil(8/B), 16]
    ref = ctypes.byref
    x, gi, out = T((6, 8), 0), T((6, 2), 4), T((6, 2, 16), 0)
    wq, s1, z1 = T((3, 8, 16), 8), T((3, 1, 16), 0), T((3, 1, 16), 8)
    call = lib.mm_grouped_matmul_qweights
    # block 4 needs scales [3, 2, 16]
    assert call(ref(x), ref(wq), ref(s1), None, 4, ref(gi), None, ref(out), None, 0, None) == 2
    # a negative block size
    assert call(ref(x), ref(wq), ref(s1), None, -1, ref(gi), None, ref(out), None, 0, None) == 1
    # weights must be 8-bit, the scale of type T, the zero point of the weights' type
    assert call(ref(x), ref(T((3, 8, 16), 0)), ref(s1), None, 0, ref(gi), None, ref(out), None, 0, None) == 3
    assert call(ref(x), ref(wq), ref(T((3, 1, 16), 2)), None, 0, ref(gi), None, ref(out), None, 0, None) == 3
    assert call(ref(x), ref(wq), ref(s1), ref(T((3, 1, 16), 9)), 0, ref(gi), None, ref(out), None, 0, None) == 3
    # zero point of another shape; K mismatch with the input
    assert call(ref(x), ref(wq), ref(s1), ref(T((3, 2, 16), 8)), 0, ref(gi), None, ref(out), None, 0, None) == 2
    assert call(ref(x), ref(T((3, 7, 16), 8)), ref(s1), ref(z1), 0, ref(gi), None, ref(out), None, 0, None) == 2
    # output of the wrong type
    assert call(ref(x), ref(wq), ref(s1), ref(z1), 0, ref(gi), None, ref(T((6, 2, 16), 1)), None, 0, None) == 3
    nbytes = ctypes.c_size_t(123)
    assert lib.mm_grouped_matmul_qweights_workspace_size(ref(x), ref(wq), ref(s1), None, 3, ref(gi),
                                                         ref(nbytes)) == 2
