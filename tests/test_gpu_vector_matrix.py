"""Vector-matrix products (one row of A') on the tensor cores, against the oracle.

A one-row A' (Gemm with M = 1, MatMul's promoted 1-D A, A stored [K, 1] with
transA) is a K-major tile whatever its row stride: the tensor-core kernels
take it as a 128-row tile whose other rows read the fill value and are never
stored.  These tests cover both layouts of B', ragged N and K, every C
broadcast shape, a broadcast batch, fp32 (three tf32 products), and check
that the planner sends large one-row products to the tensor cores.
"""

import contextlib

import pytest
import torch

import oracle
import quantized_gemm_gb300 as qg
from helpers import TOL, max_rel_err, rand_tensor, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@contextlib.contextmanager
def tensor_path():
    qg.mm_set_path_policy(qg.MM_PATH_TENSOR)
    try:
        yield
    finally:
        qg.mm_set_path_policy(qg.MM_PATH_AUTO)


def _gemm_check(A, B, C, alpha, beta, tA, tB):
    Y = qg.mm_gemm(A, B, C, alpha, beta, tA, tB)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    a, b = to_np(A), to_np(B)
    c = None if C is None else to_np(C)
    kw = dict(alpha=alpha, beta=beta, transA=tA, transB=tB)
    err = max_rel_err(to_np(Y), oracle.gemm(a, b, c, **kw), oracle.gemm_abs_scale(a, b, c, **kw))
    assert err <= TOL[A.dtype], err


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("K", [64, 1096, 4160])
@pytest.mark.parametrize("tB", [0, 1])
@pytest.mark.parametrize("cshape", [None, (1, 520), (520,), (1, 1), ()], ids=str)
def test_gemm_one_row(dtype, K, tB, cshape):
    # N = 520: a partial last column tile; K = 1096 a partial last k-block.
    N = 520
    A = rand_tensor((1, K), dtype, 800, DEV)
    B = rand_tensor((N, K) if tB else (K, N), dtype, 801, DEV)
    C = None if cshape is None else rand_tensor(cshape, dtype, 802, DEV)
    with tensor_path():
        _gemm_check(A, B, C, 0.5, 2.0, 0, tB)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
def test_gemm_one_row_stored_as_column(dtype):
    # transA = 1 with A stored [K, 1]: A' has row stride 1 and column stride 1.
    K, N = 1024, 264
    A = rand_tensor((K, 1), dtype, 803, DEV)
    B = rand_tensor((N, K), dtype, 804, DEV)
    with tensor_path():
        _gemm_check(A, B, rand_tensor((1, N), dtype, 805, DEV), 1.5, -0.5, 1, 1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
def test_matmul_promoted_vector(dtype):
    # A [K] @ B [K, N], A [K] @ a K-major view of B, A [K] @ B [3, K, N]
    # (the vector broadcast over the batch).  N is a multiple of 8: B's
    # stored row stride.
    K, N = 2048, 704
    a = rand_tensor((K,), dtype, 806, DEV)
    for B in (rand_tensor((K, N), dtype, 807, DEV), rand_tensor((N, K), dtype, 808, DEV).t(),
              rand_tensor((3, K, N), dtype, 809, DEV)):
        with tensor_path():
            Y = qg.mm_matmul(a, B)
        assert qg.mm_last_path() == qg.MM_PATH_TENSOR
        an, bn = to_np(a), to_np(B)
        assert max_rel_err(to_np(Y), oracle.matmul(an, bn), oracle.matmul_abs_scale(an, bn)) <= TOL[dtype]


def test_gemm_one_row_fp32_three_tf32():
    K, N = 4096, 4096
    A = rand_tensor((1, K), torch.float32, 810, DEV)
    B = rand_tensor((N, K), torch.float32, 811, DEV)
    with tensor_path():
        _gemm_check(A, B, rand_tensor((N,), torch.float32, 812, DEV), 1.0, 1.0, 0, 1)


def test_planner_sends_large_one_row_products_to_tensor_cores():
    A = rand_tensor((1, 4096), torch.bfloat16, 813, DEV)
    B = rand_tensor((4096, 4096), torch.bfloat16, 814, DEV)
    _gemm_check(A, B, None, 1.0, 1.0, 0, 1)
