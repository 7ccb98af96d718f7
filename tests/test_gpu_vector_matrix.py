"""Products with few rows of A', against the oracle.

A one-row A' (Gemm with M = 1, MatMul's promoted 1-D A, A stored [K, 1] with
transA) is a K-major tile whatever its row stride: the tensor-core kernels
take it as a 128-row tile whose other rows read the fill value and are never
stored.  These tests cover both layouts of B', ragged N and K, every C
broadcast shape, a broadcast batch and fp32 (three tf32 products) there.

Products with 1 to 4 rows of A' also have CUDA-core kernels that stream B'
once (MM_PATH_VECTOR), which the planner prefers: one for K-major B' (k
contiguous in A' and B') and one for MN-major B' (n contiguous; k split over a
cluster of CTAs whose partial sums meet in distributed shared memory).  The
second half covers both with every row count, odd and ragged N, ragged K
(padded views, so a last piece of fewer than 8 values; K smaller than the
cluster), C shapes, broadcast batches, promoted vectors, strided A' and the
three float types, and checks which path the planner takes.
"""

import contextlib

import numpy as np
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


# ------------------------------------------------------------------ the few-row kernel

@contextlib.contextmanager
def vector_path():
    qg.mm_set_path_policy(qg.MM_PATH_VECTOR)
    try:
        yield
    finally:
        qg.mm_set_path_policy(qg.MM_PATH_AUTO)


def _vec_gemm_check(A, B, C, alpha, beta, tA, tB):
    with vector_path():
        Y = qg.mm_gemm(A, B, C, alpha, beta, tA, tB)
    assert qg.mm_last_path() == qg.MM_PATH_VECTOR
    assert qg.mm_get_device_status() == "MM_OK"
    a, b = to_np(A), to_np(B)
    c = None if C is None else to_np(C)
    kw = dict(alpha=alpha, beta=beta, transA=tA, transB=tB)
    err = max_rel_err(to_np(Y), oracle.gemm(a, b, c, **kw), oracle.gemm_abs_scale(a, b, c, **kw))
    assert err <= TOL[A.dtype], err


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32], ids=str)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(520, 64), (1037, 1096), (257, 4160), (64, 8200)])
def test_vector_gemm(dtype, M, N, K):
    # B stored [N, K] (transB = 1): K-major B'.  K = 64 runs only the ragged
    # loop; 4160 and 8200 full rounds of in-flight pieces plus whole pieces;
    # odd N a last warp with one real column.
    A = rand_tensor((M, K), dtype, 820 + M, DEV)
    B = rand_tensor((N, K), dtype, 830, DEV)
    C = rand_tensor((1, N), dtype, 831, DEV)
    _vec_gemm_check(A, B, C, 0.5, 2.0, 0, 1)


@pytest.mark.parametrize("cshape", [None, (3, 1), (3, 700), (700,), ()], ids=str)
def test_vector_gemm_c_shapes(cshape):
    A = rand_tensor((3, 2048), torch.bfloat16, 840, DEV)
    B = rand_tensor((700, 2048), torch.bfloat16, 841, DEV)
    C = None if cshape is None else rand_tensor(cshape, torch.bfloat16, 842, DEV)
    _vec_gemm_check(A, B, C, -1.5, 0.75, 0, 1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=str)
@pytest.mark.parametrize("K", [1, 7, 1001, 4099])
def test_vector_gemm_ragged_k_in_padded_views(dtype, K):
    # Rows of A and B padded to a 16-byte multiple: aligned pieces, then a last
    # piece of K % 8 (bf16) or K % 4 (f32) values read one by one.
    step = 16 // torch.tensor([], dtype=dtype).element_size()
    Kp = (K + step - 1) // step * step + step
    M, N = 4, 333
    A = rand_tensor((M, Kp), dtype, 850, DEV)[:, :K]
    B = rand_tensor((N, Kp), dtype, 851, DEV)[:, :K]
    _vec_gemm_check(A, B, rand_tensor((N,), dtype, 852, DEV), 1.0, 1.0, 0, 1)


def test_vector_gemm_transposed_a_stored_as_column():
    # transA = 1 with A stored [K, 1]: A' is one row with k contiguous.
    K, N = 3000, 1000
    A = rand_tensor((K, 1), torch.float16, 853, DEV)
    B = rand_tensor((N, K), torch.float16, 854, DEV)
    _vec_gemm_check(A, B, None, 2.0, 0.0, 1, 1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=str)
def test_vector_matmul_batched_and_promoted(dtype):
    # A [2, 3, K] @ a K-major view of B [2, 1, N, K] (B broadcast over dim 1),
    # a promoted vector [K] @ K-major views, and N = 1 (a [K, 1] B).
    K, N = 2056, 264
    cases = [
        (rand_tensor((2, 3, K), dtype, 860, DEV), rand_tensor((2, 1, N, K), dtype, 861, DEV).transpose(-1, -2)),
        (rand_tensor((K,), dtype, 862, DEV), rand_tensor((N, K), dtype, 863, DEV).t()),
        (rand_tensor((K,), dtype, 864, DEV), rand_tensor((5, N, K), dtype, 865, DEV).transpose(-1, -2)),
        (rand_tensor((2, K), dtype, 866, DEV), rand_tensor((K, 1), dtype, 867, DEV)),
    ]
    for a, B in cases:
        with vector_path():
            Y = qg.mm_matmul(a, B)
        assert qg.mm_last_path() == qg.MM_PATH_VECTOR
        an, bn = to_np(a), to_np(B)
        assert max_rel_err(to_np(Y), oracle.matmul(an, bn), oracle.matmul_abs_scale(an, bn)) <= TOL[dtype]


def test_vector_gemm_large_is_exact_on_integer_inputs():
    # Small integers in fp32: every product and partial sum is exact, so the
    # result is the oracle's bit for bit, whatever the order of the additions.
    g = torch.Generator().manual_seed(870)
    A = torch.randint(-3, 4, (2, 8192), generator=g).to(torch.float32).to(DEV)
    B = torch.randint(-3, 4, (8192, 8192), generator=g).to(torch.float32).to(DEV)
    with vector_path():
        Y = qg.mm_gemm(A, B, None, 1.0, 1.0, 0, 1)
    assert qg.mm_last_path() == qg.MM_PATH_VECTOR
    assert np.array_equal(to_np(Y), oracle.gemm(to_np(A), to_np(B), None, transB=1))


def test_vector_path_rejects_what_it_does_not_take():
    A = rand_tensor((5, 256), torch.bfloat16, 871, DEV)          # 5 rows
    B = rand_tensor((64, 256), torch.bfloat16, 872, DEV)
    A2 = rand_tensor((2, 256), torch.bfloat16, 873, DEV)
    B2 = rand_tensor((256, 68), torch.bfloat16, 874, DEV)[:, :64]  # MN-major B', rows 136 bytes apart
    A3 = rand_tensor((2, 256), torch.float64, 875, DEV)
    B3 = rand_tensor((64, 256), torch.float64, 876, DEV)          # f64
    A4 = rand_tensor((2, 260), torch.bfloat16, 877, DEV)[:, 1:257]  # rows start off a 16-byte boundary
    for a, b, tB in ((A, B, 1), (A2, B2, 0), (A3, B3, 1), (A4, B, 1)):
        with vector_path():
            with pytest.raises(qg.MMError) as e:
                qg.mm_gemm(a, b, None, 1.0, 1.0, 0, tB)
        assert e.value.name == "MM_ERR_UNSUPPORTED"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32], ids=str)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(520, 64), (1037, 1096), (264, 5), (64, 8200)])
def test_vector_gemm_mn_major(dtype, M, N, K):
    # B stored [K, N] (transB = 0): MN-major B'.  N = 1037 ends in a lane with
    # a partial piece; K = 5 leaves most CTAs of the cluster without rows;
    # K = 1096 and 8200 give every warp full rounds and single rows.
    A = rand_tensor((M, K), dtype, 880 + M, DEV)
    B = rand_tensor((K, (N + 7) // 8 * 8), dtype, 885, DEV)[:, :N]   # rows 16-byte aligned
    C = rand_tensor((N,), dtype, 886, DEV)
    _vec_gemm_check(A, B, C, 0.5, 2.0, 0, 0)


def test_vector_gemm_mn_major_strided_a_and_c_shapes():
    # transA = 1 with A stored [K, 3]: A' has k stride 3; C per row.
    K, N = 2000, 776
    A = rand_tensor((K, 3), torch.bfloat16, 887, DEV)
    B = rand_tensor((K, N), torch.bfloat16, 888, DEV)
    for cshape in [None, (3, 1), (3, N)]:
        C = None if cshape is None else rand_tensor(cshape, torch.bfloat16, 889, DEV)
        _vec_gemm_check(A, B, C, 1.25, -0.5, 1, 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=str)
def test_vector_matmul_mn_major_batched(dtype):
    # a [K] @ B [5, K, N]; A [2, 3, K] @ B [2, 1, K, N] (B broadcast over dim 1).
    K, N = 1500, 600
    for a, B in ((rand_tensor((K,), dtype, 890, DEV), rand_tensor((5, K, N), dtype, 891, DEV)),
                 (rand_tensor((2, 3, K), dtype, 892, DEV), rand_tensor((2, 1, K, N), dtype, 893, DEV))):
        with vector_path():
            Y = qg.mm_matmul(a, B)
        assert qg.mm_last_path() == qg.MM_PATH_VECTOR
        an, bn = to_np(a), to_np(B)
        assert max_rel_err(to_np(Y), oracle.matmul(an, bn), oracle.matmul_abs_scale(an, bn)) <= TOL[dtype]


def test_vector_gemm_mn_major_exact_on_integer_inputs():
    # Small integers in fp32: exact sums, so bit for bit equal to the oracle.
    g = torch.Generator().manual_seed(894)
    A = torch.randint(-3, 4, (3, 8192), generator=g).to(torch.float32).to(DEV)
    B = torch.randint(-3, 4, (8192, 4100), generator=g).to(torch.float32).to(DEV)
    with vector_path():
        Y = qg.mm_gemm(A, B, None, 1.0, 1.0, 0, 0)
    assert qg.mm_last_path() == qg.MM_PATH_VECTOR
    assert np.array_equal(to_np(Y), oracle.gemm(to_np(A), to_np(B), None))


def test_planner_paths_for_few_row_products():
    # 1-4 rows: the few-row kernels for both layouts of B'; 5 or more rows:
    # the tensor cores.
    A = rand_tensor((1, 4096), torch.bfloat16, 813, DEV)
    B = rand_tensor((4096, 4096), torch.bfloat16, 814, DEV)
    a, b = to_np(A), to_np(B)
    for tB, path in ((1, qg.MM_PATH_VECTOR), (0, qg.MM_PATH_VECTOR)):
        Y = qg.mm_gemm(A, B, None, 1.0, 1.0, 0, tB)
        assert qg.mm_last_path() == path
        err = max_rel_err(to_np(Y), oracle.gemm(a, b, None, transB=tB), oracle.gemm_abs_scale(a, b, None, transB=tB))
        assert err <= TOL[torch.bfloat16], err
    A8 = rand_tensor((8, 4096), torch.bfloat16, 815, DEV)
    qg.mm_gemm(A8, B, None, 1.0, 1.0, 0, 1)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    # 3 rows of bf16: the few-row kernel for K-major B', the tensor cores
    # (as fast there) for MN-major B'; fp32 takes the few-row kernel for both.
    A3 = rand_tensor((3, 4096), torch.bfloat16, 816, DEV)
    for tB, path in ((1, qg.MM_PATH_VECTOR), (0, qg.MM_PATH_TENSOR)):
        qg.mm_gemm(A3, B, None, 1.0, 1.0, 0, tB)
        assert qg.mm_last_path() == path
    qg.mm_gemm(A3.float(), B.float(), None, 1.0, 1.0, 0, 0)
    assert qg.mm_last_path() == qg.MM_PATH_VECTOR
