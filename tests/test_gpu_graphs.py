"""The entry points inside CUDA graphs.

An application that replays a fixed sequence of products captures the calls
in a CUDA graph once and replays it, paying one graph launch instead of one
host call per kernel.  The calls enqueue only kernels and asynchronous
memsets on the caller's stream, so after a first call on the device (which
caches per-device properties such as the SM count) they can be captured.
These tests capture Gemm (tensor-core, CUDA-core and few-row paths),
QLinearMatMul and GroupedMatMul with caller-provided outputs and workspaces, replay the graph
twice on new input values, and compare every output bit for bit with direct
calls on the same inputs.
"""

import numpy as np
import pytest
import torch

import quantized_gemm_gb300 as qg
from helpers import rand_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _qlinear_inputs(seed):
    g = np.random.default_rng(seed)
    M, K, N = 300, 1024, 264
    return {
        "a": torch.from_numpy(g.integers(-128, 128, (M, K)).astype(np.int8)).to(DEV),
        "a_scale": torch.from_numpy(g.uniform(0.003, 0.01, (M, 1)).astype(np.float32)).to(DEV),
        "a_zero_point": torch.from_numpy(g.integers(-20, 21, (M, 1)).astype(np.int8)).to(DEV),
        "b": torch.from_numpy(g.integers(-128, 128, (K, N)).astype(np.int8)).to(DEV),
        "b_scale": torch.from_numpy(g.uniform(0.003, 0.01, (1, N)).astype(np.float32)).to(DEV),
        "b_zero_point": torch.from_numpy(g.integers(-20, 21, (1, N)).astype(np.int8)).to(DEV),
        "y_scale": torch.tensor(0.16, dtype=torch.float32, device=DEV),
        "y_zero_point": torch.tensor(-9, dtype=torch.int8, device=DEV),
    }


QKEYS = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")


def test_products_captured_in_a_cuda_graph_match_direct_calls():
    # Inputs live in fixed buffers that the graph reads; each replay sees the
    # values copied into them before it.
    A = rand_tensor((640, 1024), torch.bfloat16, 60, DEV)
    B = rand_tensor((520, 1024), torch.bfloat16, 61, DEV)
    C = rand_tensor((1, 520), torch.bfloat16, 62, DEV)
    Af = rand_tensor((96, 72), torch.float32, 63, DEV)
    Bf = rand_tensor((72, 40), torch.float32, 64, DEV)
    q = _qlinear_inputs(65)
    x = rand_tensor((400, 512), torch.bfloat16, 66, DEV)
    w = rand_tensor((6, 512, 264), torch.bfloat16, 67, DEV)
    bias = rand_tensor((6, 264), torch.bfloat16, 68, DEV)
    gi = torch.from_numpy(np.random.default_rng(69).integers(0, 6, (400, 2)).astype(np.int32)).to(DEV)
    Av = rand_tensor((2, 1024), torch.bfloat16, 72, DEV)     # two rows: the few-row kernel

    Y = torch.empty((640, 520), dtype=torch.bfloat16, device=DEV)
    Yf = torch.empty((96, 40), dtype=torch.float32, device=DEV)
    Yv = torch.empty((2, 520), dtype=torch.bfloat16, device=DEV)
    yq = torch.empty((300, 264), dtype=torch.int8, device=DEV)
    wsq = torch.empty(qg.mm_qlinear_matmul_workspace_size(q["a"], q["b"]), dtype=torch.uint8, device=DEV)
    out = torch.empty((400, 2, 264), dtype=torch.bfloat16, device=DEV)
    wsg = torch.empty(qg.mm_grouped_matmul_workspace_size(x, w, gi), dtype=torch.uint8, device=DEV)

    def step():
        qg.mm_gemm(A, B, C, 0.5, 2.0, 0, 1, out=Y)
        qg.mm_matmul(Af, Bf, out=Yf)
        qg.mm_qlinear_matmul(*[q[k] for k in QKEYS], out=yq, workspace=wsq)
        qg.mm_grouped_matmul(x, w, gi, bias, out=out, workspace=wsg)
        qg.mm_gemm(Av, B, C, 1.0, -1.0, 0, 1, out=Yv)

    def direct():
        return (qg.mm_gemm(A, B, C, 0.5, 2.0, 0, 1), qg.mm_matmul(Af, Bf),
                qg.mm_qlinear_matmul(*[q[k] for k in QKEYS]), qg.mm_grouped_matmul(x, w, gi, bias),
                qg.mm_gemm(Av, B, C, 1.0, -1.0, 0, 1))

    # First calls on the device, outside any capture, on a side stream as
    # torch's capture does.
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed in (70, 71):
        g = np.random.default_rng(seed)
        for t in (A, B, C, x, w, bias, Av):
            t.copy_(torch.from_numpy(g.standard_normal(tuple(t.shape))).to(t.dtype))
        for t in (Af, Bf):
            t.copy_(torch.from_numpy(g.standard_normal(tuple(t.shape))).to(t.dtype))
        gi.copy_(torch.from_numpy(g.integers(0, 6, tuple(gi.shape)).astype(np.int32)))
        for k, v in _qlinear_inputs(seed).items():
            q[k].copy_(v)
        graph.replay()
        torch.cuda.synchronize()
        want = direct()
        torch.cuda.synchronize()
        for got, ref in zip((Y, Yf, yq, out, Yv), want):
            assert torch.equal(got, ref)
    assert qg.mm_get_device_status() == "MM_OK"
