"""Python binding of the GB300 ONNX matrix-product library (include/mm.h).

Argument marshalling only: every function below turns torch tensors into the
C ABI's ``mm_tensor`` descriptors (device pointer, type, shape, element
strides), allocates the output (and, where the fast path needs one, the
workspace) with torch's allocator, and calls the library's entry point of the
same name on the current CUDA stream.  All arithmetic runs in the library's
CUDA kernels; there is no fallback of any kind, and importing a function whose
shared library was not built raises immediately.
"""

import ctypes
import os
import struct

import torch

__all__ = [
    "MMError", "mm_matmul", "mm_gemm", "mm_qlinear_matmul", "mm_grouped_matmul",
    "mm_get_device_status", "mm_set_path_policy", "mm_last_path", "mm_set_wait_limit_ns", "mm_version",
    "library_path",
    "mm_qlinear_matmul_workspace_size", "mm_grouped_matmul_workspace_size", "mm_grouped_matmul_noalloc",
    "mm_grouped_matmul_qweights", "mm_grouped_matmul_qweights_workspace_size",
    "MM_PATH_AUTO", "MM_PATH_SIMT", "MM_PATH_TENSOR", "MM_PATH_NONE", "MM_PATH_VECTOR", "mm_stream_probe",
    "mm_alu_probe", "MM_ALU_CHAINS",
]

MM_MAX_DIMS = 8
MM_PATH_AUTO, MM_PATH_SIMT, MM_PATH_TENSOR, MM_PATH_NONE, MM_PATH_VECTOR = 0, 1, 2, 3, 4
_STATUS = ["MM_OK", "MM_ERR_INVALID_ARG", "MM_ERR_SHAPE", "MM_ERR_DTYPE", "MM_ERR_UNSUPPORTED",
           "MM_ERR_WORKSPACE", "MM_ERR_CUDA", "MM_ERR_TIMEOUT", "MM_ERR_INDEX_RANGE"]

_DTYPES = {
    torch.bfloat16: 0, torch.float16: 1, torch.float32: 2, torch.float64: 3,
    torch.int32: 4, torch.int64: 5, torch.uint32: 6, torch.uint64: 7,
    torch.int8: 8, torch.uint8: 9,
}
# 4-bit types (include/mm.h MM_I4 / MM_U4), which torch has no dtype for:
# passed as uint8 bytes holding two values each (see _desc4).
_PACKED4 = {"int4": 10, "uint4": 11}


def library_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqgemm_gb300.so")


class MMTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * MM_MAX_DIMS), ("strides", ctypes.c_int64 * MM_MAX_DIMS)]


class MMError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        self.name = _STATUS[status] if 0 <= status < len(_STATUS) else "unknown"
        super().__init__("%s: %s" % (where, _lib().mm_status_string(status).decode()))


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("the CUDA library %s is not built; run __graft_entry__.build() "
                               "(or python -m quantized_gemm_gb300.build)" % path)
        lib = ctypes.CDLL(path)
        P, I32, I64, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        T = ctypes.POINTER(MMTensor)
        sigs = {
            "mm_status_string": ([I32], ctypes.c_char_p),
            "mm_version": ([], ctypes.c_char_p),
            "mm_set_path_policy": ([I32], I32),
            "mm_last_path": ([], I32),
            "mm_matmul_output_shape": ([T, T, ctypes.POINTER(I32), ctypes.POINTER(I64)], I32),
            "mm_matmul": ([T, T, T, P], I32),
            "mm_gemm_output_shape": ([T, T, I64, I64, ctypes.POINTER(I32), ctypes.POINTER(I64)], I32),
            "mm_gemm": ([T, T, T, F, F, I64, I64, T, P], I32),
            "mm_qlinear_matmul_workspace_size": ([T, T, ctypes.POINTER(SZ)], I32),
            "mm_qlinear_matmul": ([T, T, T, T, T, T, T, T, T, P, SZ, P], I32),
            "mm_grouped_matmul_workspace_size": ([T, T, T, ctypes.POINTER(SZ)], I32),
            "mm_grouped_matmul": ([T, T, T, T, T, P, SZ, P], I32),
            "mm_get_device_status": ([P], I32),
            "mm_grouped_matmul_noalloc_max_scratch": ([], SZ),
            "mm_set_wait_limit_ns": ([ctypes.c_uint64], I32),
            "mm_grouped_matmul_noalloc": ([T, T, T, T, T, P], I32),
            "mm_grouped_matmul_qweights_workspace_size": ([T, T, T, T, I64, T, ctypes.POINTER(SZ)], I32),
            "mm_grouped_matmul_qweights": ([T, T, T, T, I64, T, T, T, P, SZ, P], I32),
            "mm_stream_probe": ([P, P, SZ, I32, P], I32),
            "mm_alu_probe": ([I32, P, I64, P, P], I32),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


# MMTensor's bytes: pointer, dtype, ndim, shape[8], strides[8] (packed in one
# call, which is cheaper than filling the ctypes arrays element by element).
_MM_TENSOR_BYTES = struct.Struct("<Qii%dq%dq" % (MM_MAX_DIMS, MM_MAX_DIMS))
_ZEROS = (0,) * MM_MAX_DIMS


def _desc(t):
    """mm_tensor describing torch tensor ``t`` (None -> NULL)."""
    if t is None:
        return None
    dt = _DTYPES.get(t.dtype)
    if dt is None:
        raise TypeError("unsupported dtype %s" % t.dtype)
    nd = t.dim()
    if nd > MM_MAX_DIMS:
        raise ValueError("at most %d dimensions" % MM_MAX_DIMS)
    return MMTensor.from_buffer_copy(_MM_TENSOR_BYTES.pack(
        t.data_ptr() if t.numel() > 0 else 0, dt, nd, *(tuple(t.shape) + _ZEROS[nd:]), *(t.stride() + _ZEROS[nd:])))


def _desc4(t, kind):
    """mm_tensor of 4-bit values stored packed in uint8 tensor ``t`` [..., N/2]:
    logical shape [..., N], element strides twice the byte strides (the last
    one 1); the even element of a byte is its low nibble."""
    if t is None:
        return None
    if kind not in _PACKED4:
        raise ValueError("packed4 must be 'int4' or 'uint4'")
    if t.dtype != torch.uint8 or t.dim() < 1 or t.stride(-1) != 1:
        raise ValueError("packed 4-bit values arrive as a uint8 tensor with a unit stride in its last dimension")
    nd = t.dim()
    shape = tuple(t.shape[:-1]) + (2 * t.shape[-1],)
    strides = tuple(2 * st for st in t.stride()[:-1]) + (1,)
    return MMTensor.from_buffer_copy(_MM_TENSOR_BYTES.pack(
        t.data_ptr() if t.numel() > 0 else 0, _PACKED4[kind], nd, *(shape + _ZEROS[nd:]), *(strides + _ZEROS[nd:])))


def _ref(d):
    return None if d is None else ctypes.byref(d)


# The current stream's handle for a device index, without building a
# torch.cuda.Stream object (the public route below when torch lacks it).
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t, stream):
    if stream is None:
        if _RAW_STREAM is not None and t.is_cuda:
            return ctypes.c_void_p(_RAW_STREAM(t.get_device()))
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != 0:
        raise MMError(status, where)


def _out_shape(fn, *args):
    nd = ctypes.c_int32()
    shape = (ctypes.c_int64 * MM_MAX_DIMS)()
    _check(fn(*args, ctypes.byref(nd), shape), fn.__name__)
    return tuple(shape[i] for i in range(nd.value))


def _workspace(nbytes, device, given=None):
    """(tensor, size) of a workspace of at least ``nbytes``: ``given`` when it is large enough."""
    if nbytes == 0:
        return None, 0
    if given is not None:
        if given.numel() * given.element_size() < nbytes:
            raise ValueError("workspace of %d bytes is smaller than the %d required" % (given.numel(), nbytes))
        return given, given.numel() * given.element_size()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return ws, nbytes


def mm_qlinear_matmul_workspace_size(a, b):
    nbytes = ctypes.c_size_t()
    _check(_lib().mm_qlinear_matmul_workspace_size(_ref(_desc(a)), _ref(_desc(b)), ctypes.byref(nbytes)),
           "mm_qlinear_matmul_workspace_size")
    return nbytes.value


def mm_grouped_matmul_workspace_size(input, weights, group_indices):
    nbytes = ctypes.c_size_t()
    _check(_lib().mm_grouped_matmul_workspace_size(_ref(_desc(input)), _ref(_desc(weights)), _ref(_desc(group_indices)),
                                                   ctypes.byref(nbytes)), "mm_grouped_matmul_workspace_size")
    return nbytes.value


def mm_version():
    return _lib().mm_version().decode()


def mm_set_path_policy(policy):
    _check(_lib().mm_set_path_policy(policy), "mm_set_path_policy")


def mm_last_path():
    return _lib().mm_last_path()


def mm_set_wait_limit_ns(ns):
    """Limit of each tensor-core pipeline wait, in ns (0 = default 2 s)."""
    _check(_lib().mm_set_wait_limit_ns(int(ns)), "mm_set_wait_limit_ns")


def mm_stream_probe(dst, src=None, mode=0, stream=None):
    """Memory-stream measurement kernel on the bytes of ``dst``: mode 0 writes
    them, 1 copies ``src`` into them (same size), 2 writes them with bulk (TMA)
    stores."""
    nbytes = dst.numel() * dst.element_size()
    if src is not None and src.numel() * src.element_size() != nbytes:
        raise ValueError("src and dst must have the same size in bytes")
    _check(_lib().mm_stream_probe(dst.data_ptr(), None if src is None else src.data_ptr(), nbytes, int(mode),
                                  _stream(dst, stream)), "mm_stream_probe")


# Independent multiply-add chains per thread of mm_alu_probe (include/mm.h).
MM_ALU_CHAINS = 16


def mm_alu_probe(op, iters, out=None, stream=None):
    """Arithmetic-rate probe (op 0 int32 multiply-add, 1 fp64 FMA, 2 fp32 FMA):
    returns the number of multiply-adds the launch performs; with ``out`` (a
    device tensor of at least that many / (MM_ALU_CHAINS * iters) 8-byte
    elements, one per thread) it also launches the probe on the current stream."""
    n = ctypes.c_int64(0)
    ptr = None if out is None else out.data_ptr()
    st = None if out is None else _stream(out, stream)
    _check(_lib().mm_alu_probe(int(op), ptr, int(iters), ctypes.byref(n), st), "mm_alu_probe")
    return n.value


def mm_matmul(A, B, out=None, stream=None):
    """Y = A @ B with numpy.matmul semantics (MatMul, opset 13)."""
    lib = _lib()
    dA, dB = _desc(A), _desc(B)
    # A given output is checked by the library itself (MM_ERR_SHAPE).
    Y = out if out is not None else torch.empty(_out_shape(lib.mm_matmul_output_shape, _ref(dA), _ref(dB)),
                                                dtype=A.dtype, device=A.device)
    _check(lib.mm_matmul(_ref(dA), _ref(dB), _ref(_desc(Y)), _stream(A, stream)), "mm_matmul")
    return Y


def mm_gemm(A, B, C=None, alpha=1.0, beta=1.0, transA=0, transB=0, out=None, stream=None):
    """Y = alpha * A' @ B' + beta * C (Gemm, opset 13)."""
    lib = _lib()
    dA, dB = _desc(A), _desc(B)
    Y = out if out is not None else torch.empty(
        _out_shape(lib.mm_gemm_output_shape, _ref(dA), _ref(dB), int(transA), int(transB)), dtype=A.dtype,
        device=A.device)
    _check(lib.mm_gemm(_ref(dA), _ref(dB), _ref(_desc(C)), float(alpha), float(beta), int(transA), int(transB),
                       _ref(_desc(Y)), _stream(A, stream)), "mm_gemm")
    return Y


def mm_qlinear_matmul(a, a_scale, a_zero_point, b, b_scale, b_zero_point, y_scale, y_zero_point,
                      out=None, stream=None, workspace=None):
    """Quantized matmul of int8/uint8 tensors (QLinearMatMul, opset 10); y has y_zero_point's type."""
    lib = _lib()
    da, db = _desc(a), _desc(b)
    y = out if out is not None else torch.empty(_out_shape(lib.mm_matmul_output_shape, _ref(da), _ref(db)),
                                                dtype=y_zero_point.dtype, device=a.device)
    nbytes = ctypes.c_size_t()
    _check(lib.mm_qlinear_matmul_workspace_size(_ref(da), _ref(db), ctypes.byref(nbytes)),
           "mm_qlinear_matmul_workspace_size")
    ws, wsb = _workspace(nbytes.value, a.device, workspace)
    _check(lib.mm_qlinear_matmul(_ref(da), _ref(_desc(a_scale)), _ref(_desc(a_zero_point)), _ref(db),
                                 _ref(_desc(b_scale)), _ref(_desc(b_zero_point)), _ref(_desc(y_scale)),
                                 _ref(_desc(y_zero_point)), _ref(_desc(y)),
                                 None if ws is None else ws.data_ptr(), wsb, _stream(a, stream)),
           "mm_qlinear_matmul")
    return y


def mm_grouped_matmul(input, weights, group_indices, bias=None, out=None, stream=None, workspace=None):
    """output[m, i] = input[m] @ weights[group_indices[m, i]] (+ bias[g]) (GroupedMatMul, opset 29)."""
    lib = _lib()
    dx, dw, dg = _desc(input), _desc(weights), _desc(group_indices)
    M, S, N = input.shape[0], group_indices.shape[1], weights.shape[2]
    y = torch.empty((M, S, N), dtype=input.dtype, device=input.device) if out is None else out
    nbytes = ctypes.c_size_t()
    _check(lib.mm_grouped_matmul_workspace_size(_ref(dx), _ref(dw), _ref(dg), ctypes.byref(nbytes)),
           "mm_grouped_matmul_workspace_size")
    ws, wsb = _workspace(nbytes.value, input.device, workspace)
    _check(lib.mm_grouped_matmul(_ref(dx), _ref(dw), _ref(dg), _ref(_desc(bias)), _ref(_desc(y)),
                                 None if ws is None else ws.data_ptr(), wsb, _stream(input, stream)),
           "mm_grouped_matmul")
    return y


def _qdesc(t, packed4):
    return _desc(t) if packed4 is None else _desc4(t, packed4)


def mm_grouped_matmul_qweights_workspace_size(input, weights_q, w_scale, w_zero_point, block_size, group_indices,
                                              packed4=None):
    nbytes = ctypes.c_size_t()
    _check(_lib().mm_grouped_matmul_qweights_workspace_size(
        _ref(_desc(input)), _ref(_qdesc(weights_q, packed4)), _ref(_desc(w_scale)),
        _ref(_qdesc(w_zero_point, packed4)), int(block_size), _ref(_desc(group_indices)), ctypes.byref(nbytes)),
        "mm_grouped_matmul_qweights_workspace_size")
    return nbytes.value


def mm_grouped_matmul_qweights(input, weights_q, w_scale, w_zero_point, block_size, group_indices, bias=None,
                               out=None, stream=None, workspace=None, packed4=None):
    """GroupedMatMul of quantized experts: input[m] @ W[g] (+ bias[g]) with
    W = DequantizeLinear(weights_q, w_scale, w_zero_point) in blocks of
    ``block_size`` rows of K (0: one scale per group and column), fused.
    weights_q and w_zero_point are int8/uint8 tensors, or with ``packed4``
    ('int4' or 'uint4') uint8 tensors [G, K, N/2] / [G, Kb, N/2] holding two
    4-bit values per byte (the even column in the low nibble)."""
    lib = _lib()
    M, S = input.shape[0], group_indices.shape[1]
    N = weights_q.shape[2] * (2 if packed4 is not None else 1)
    y = torch.empty((M, S, N), dtype=input.dtype, device=input.device) if out is None else out
    ws, wsb = _workspace(mm_grouped_matmul_qweights_workspace_size(input, weights_q, w_scale, w_zero_point,
                                                                   block_size, group_indices, packed4),
                         input.device, workspace)
    _check(lib.mm_grouped_matmul_qweights(_ref(_desc(input)), _ref(_qdesc(weights_q, packed4)), _ref(_desc(w_scale)),
                                          _ref(_qdesc(w_zero_point, packed4)), int(block_size),
                                          _ref(_desc(group_indices)),
                                          _ref(_desc(bias)), _ref(_desc(y)), None if ws is None else ws.data_ptr(),
                                          wsb, _stream(input, stream)),
           "mm_grouped_matmul_qweights")
    return y


def mm_grouped_matmul_noalloc(input, weights, group_indices, bias=None, out=None, stream=None):
    """GroupedMatMul for callers that cannot allocate device memory per call.

    Same result as mm_grouped_matmul, computed with scratch taken from a fixed
    array the library keeps on each device (no workspace argument, no
    allocation by the library).  ``out`` must be given by such callers; when
    it is None this binding allocates it with torch for convenience.
    """
    y = torch.empty((input.shape[0], group_indices.shape[1], weights.shape[2]), dtype=input.dtype,
                    device=input.device) if out is None else out
    _check(_lib().mm_grouped_matmul_noalloc(_ref(_desc(input)), _ref(_desc(weights)), _ref(_desc(group_indices)),
                                            _ref(_desc(bias)), _ref(_desc(y)), _stream(input, stream)),
           "mm_grouped_matmul_noalloc")
    return y


def mm_get_device_status(stream=None, device=None):
    """Synchronise the stream; return (and clear) the device-side status name, e.g. 'MM_OK'."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    s = _lib().mm_get_device_status(ctypes.c_void_p(stream.cuda_stream))
    return _STATUS[s]
