"""Failure detection on the GPU without a fault.

The tensor-core kernels bound every pipeline wait.  Here the limit is cut to
1 microsecond, so waits that normally last the whole main loop run out: the
kernel must record MM_ERR_TIMEOUT in the device status word, wind down (its
in-flight copies and MMAs land under a separate fixed limit, its tensor memory
is released) and return.  The host reads the status, restores the limit, and
the same context must then compute a correct result.  Nothing here traps,
faults or hangs the GPU.
"""

import pytest
import torch

import oracle
import quantized_gemm_gb300 as qg
from helpers import max_rel_err, rand_tensor, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_pipeline_wait_timeout_is_reported_and_context_survives():
    A = rand_tensor((1024, 4096), torch.bfloat16, 1, DEV)
    B = rand_tensor((4096, 1024), torch.bfloat16, 2, DEV)
    assert qg.mm_get_device_status() == "MM_OK"
    qg.mm_set_path_policy(qg.MM_PATH_TENSOR)
    try:
        qg.mm_set_wait_limit_ns(1000)
        qg.mm_matmul(A, B)
        assert qg.mm_get_device_status() == "MM_ERR_TIMEOUT"
        assert qg.mm_get_device_status() == "MM_OK"      # reading clears it
    finally:
        qg.mm_set_wait_limit_ns(0)
    try:
        Y = qg.mm_matmul(A, B)
        assert qg.mm_get_device_status() == "MM_OK"
        assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    finally:
        qg.mm_set_path_policy(qg.MM_PATH_AUTO)
    a, b = to_np(A), to_np(B)
    assert max_rel_err(to_np(Y), oracle.matmul(a, b), oracle.matmul_abs_scale(a, b)) <= 1e-2
