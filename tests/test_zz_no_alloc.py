"""GroupedMatMul without allocation (mm_grouped_matmul_noalloc), through the C ABI.

Some callers cannot allocate device memory when they call the library (their
device memory is fixed at start-up, or cudaMalloc would block and synchronise
the device in the middle of their work).  mm_grouped_matmul_noalloc serves them
by taking its scratch from a fixed array the library keeps on each device.
These tests call it directly through ctypes on preallocated tensors, twice in
a row with different problems (the array keeps the previous call's contents,
so stale routing state must not leak into the second result), and compare each
result with the existing workspace-taking entry point and with the oracle,
within the per-element bf16/f16 bound used by every float test.  A problem whose scratch exceeds the
array is rejected with MM_ERR_WORKSPACE.

The file name makes pytest collect it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_gemm_gb300 as qg
from helpers import TOL, max_rel_err, rand_tensor, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(x, w, gi, bias, out):
    lib = qg._lib()
    d = [qg._desc(t) for t in (x, w, gi, bias, out)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.mm_grouped_matmul_noalloc(*[None if t is None else ctypes.byref(t) for t in d], stream)


def _case(M, K, N, G, S, dtype, ind, with_bias, seed):
    x = rand_tensor((M, K), dtype, seed, DEV)
    w = rand_tensor((G, K, N), dtype, seed + 1, DEV)
    gi = torch.from_numpy(np.random.default_rng(seed + 2).integers(0, G, (M, S))).to(ind).to(DEV)
    bias = rand_tensor((G, N), dtype, seed + 3, DEV) if with_bias else None
    return x, w, gi, bias


def _check_against_existing(x, w, gi, bias):
    out = torch.empty((x.shape[0], gi.shape[1], w.shape[2]), dtype=x.dtype, device=DEV)
    assert _noalloc(x, w, gi, bias, out) == 0
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    ref = qg.mm_grouped_matmul(x, w, gi, bias)        # the existing entry point (caller workspace)
    torch.cuda.synchronize()
    hx, hw, hg = to_np(x), to_np(w), gi.cpu().numpy()
    hb = None if bias is None else to_np(bias)
    scale = oracle.grouped_abs_scale(hx, hw, hg, hb)
    # Against the existing entry point, and against the oracle (which shares
    # no code with either, so a fault in the kernels both entry points run
    # cannot pass unseen).
    assert max_rel_err(to_np(out), to_np(ref), scale) <= TOL[x.dtype]
    assert max_rel_err(to_np(out), oracle.grouped_matmul(hx, hw, hg, hb), scale) <= TOL[x.dtype]


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    qg.mm_set_path_policy(qg.MM_PATH_AUTO)
    first = _case(300, 256, 520, 6, 2, torch.bfloat16, torch.int32, True, 11)
    second = _case(137, 72, 264, 9, 3, torch.float16, torch.int64, False, 21)
    _check_against_existing(*first)
    _check_against_existing(*second)


def test_noalloc_rejects_problems_beyond_its_scratch():
    limit = qg._lib().mm_grouped_matmul_noalloc_max_scratch()
    K = 2048
    M = limit // (2 * K) + 8          # M * S * K bf16 rows alone exceed the array
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((2, K, 64), dtype=torch.bfloat16, device=DEV)
    gi = torch.zeros((M, 1), dtype=torch.int32, device=DEV)
    out = torch.empty((M, 1, 64), dtype=torch.bfloat16, device=DEV)
    assert _noalloc(x, w, gi, None, out) == 5     # MM_ERR_WORKSPACE
