"""GroupedMatMul with weight-only quantized experts (GroupedMatMul - 29,
Summary: DequantizeLinear of the weights, then GroupedMatMul, fused) against
the oracle, on the CUDA-core path and on the tensor-core path whose converter
warps dequantize int8/uint8 weights in shared memory."""

import contextlib

import numpy as np
import pytest
import torch

import oracle
import quantized_gemm_gb300 as qg
from helpers import TOL, max_rel_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
T_NAME = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32", torch.float64: "f64"}


@contextlib.contextmanager
def path(p):
    qg.mm_set_path_policy(p)
    try:
        yield
    finally:
        qg.mm_set_path_policy(qg.MM_PATH_AUTO)


def _case(M, K, N, G, S, dtype, wdtype, block, with_zp, with_bias, seed, p=None):
    g = np.random.default_rng(seed)
    kb = -(-K // (block or K))
    x = torch.from_numpy(g.standard_normal((M, K))).to(dtype)
    if wdtype == torch.int8:
        wq = torch.from_numpy(g.integers(-128, 128, (G, K, N)).astype(np.int8))
        zp = torch.from_numpy(g.integers(-10, 11, (G, kb, N)).astype(np.int8)) if with_zp else None
    else:
        wq = torch.from_numpy(g.integers(0, 256, (G, K, N)).astype(np.uint8))
        zp = torch.from_numpy(g.integers(118, 139, (G, kb, N)).astype(np.uint8)) if with_zp else None
    scale = torch.from_numpy(g.uniform(0.5, 1.5, (G, kb, N)) / 128.0).to(dtype)
    bias = torch.from_numpy(g.standard_normal((G, N))).to(dtype) if with_bias else None
    probs = p if p is not None else np.full(G, 1.0 / G)
    gi = torch.from_numpy(g.choice(G, size=(M, S), p=probs).astype(np.int32))
    d = {"input": x, "weights_q": wq, "w_scale": scale, "w_zero_point": zp, "block_size": block,
         "group_indices": gi, "bias": bias}
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _run(d):
    return qg.mm_grouped_matmul_qweights(d["input"], d["weights_q"], d["w_scale"], d["w_zero_point"],
                                         d["block_size"], d["group_indices"], d["bias"])


def _oracle(d):
    t = T_NAME[d["input"].dtype]
    h = {k: (to_np(v) if isinstance(v, torch.Tensor) and v.is_floating_point()
             else (v.cpu().numpy() if isinstance(v, torch.Tensor) else v)) for k, v in d.items()}
    args = (h["input"], h["weights_q"], h["w_scale"], h["w_zero_point"], h["block_size"], h["group_indices"],
            h["bias"], t)
    return oracle.grouped_matmul_qweights(*args), oracle.grouped_qweights_abs_scale(*args)


def _check(d, tol):
    y = _run(d)
    ref, scale = _oracle(d)
    assert max_rel_err(to_np(y), ref, scale) <= tol
    return y


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32, torch.float64], ids=str)
@pytest.mark.parametrize("wdtype", [torch.int8, torch.uint8], ids=str)
@pytest.mark.parametrize("block,with_zp", [(0, True), (3, False), (64, True)])
def test_qweights_simt(dtype, wdtype, block, with_zp):
    d = _case(20, 70, 24, 3, 2, dtype, wdtype, block, with_zp, True, 50)
    with path(qg.MM_PATH_SIMT):
        _check(d, TOL[dtype])
    assert qg.mm_last_path() == qg.MM_PATH_SIMT


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("wdtype", [torch.int8, torch.uint8], ids=str)
@pytest.mark.parametrize("block,with_zp,with_bias", [(0, True, True), (0, False, False), (64, True, False),
                                                     (128, False, True)])
def test_qweights_tensor(dtype, wdtype, block, with_zp, with_bias):
    # K = 330: a partial last k-block (and, for block 128, a partial last
    # quantization block); N = 384: a partial column tile.
    d = _case(300, 330, 384, 4, 2, dtype, wdtype, block, with_zp, with_bias, 51, p=[0.5, 0.3, 0.15, 0.05])
    with path(qg.MM_PATH_TENSOR):
        _check(d, TOL[dtype])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"


@pytest.mark.parametrize("wdtype", [torch.int8, torch.uint8], ids=str)
@pytest.mark.parametrize("block", [0, 192])
def test_qweights_tensor_long_k(wdtype, block):
    # K = 1000: 16 k-blocks per tile, so each of the five staging slots is
    # reused several times within a tile and across the row tiles of a group;
    # with one scale row per column (block 0) every k-block of a column tile
    # takes the same scale and zero-point rows, with blocks of 192 rows of K
    # they change every 3 k-blocks.
    d = _case(520, 1000, 400, 3, 2, torch.bfloat16, wdtype, block, True, False, 61, p=[0.6, 0.3, 0.1])
    with path(qg.MM_PATH_TENSOR):
        _check(d, TOL[torch.bfloat16])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("wdtype", [torch.int8, torch.uint8], ids=str)
def test_qweights_tensor_dequantized_values_exact(dtype, wdtype):
    # One-hot input rows: output[m, i, :] = W[g, k(m), :] with a single term,
    # so the tensor-core result must equal the oracle's dequantized weights
    # bit for bit (their one rounding to T included).
    M, K, N, G = 384, 320, 256, 3
    d = _case(M, K, N, G, 1, dtype, wdtype, 64, True, False, 52)
    x = torch.zeros((M, K), dtype=dtype)
    ks = np.arange(M) % K
    x[np.arange(M), ks] = 1
    d["input"] = x.to(DEV)
    with path(qg.MM_PATH_TENSOR):
        y = _run(d)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    t = T_NAME[dtype]
    w = oracle.dequantize_linear(d["weights_q"].cpu().numpy(), to_np(d["w_scale"]),
                                 d["w_zero_point"].cpu().numpy(), 64, t)
    gi = d["group_indices"].cpu().numpy()
    want = w[gi[:, 0], ks, :]
    assert np.array_equal(to_np(y)[:, 0, :], want)


@pytest.mark.parametrize("wdtype", [torch.int8, torch.uint8], ids=str)
def test_qweights_tensor_extreme_scales_exact(wdtype):
    # bf16 scales by blocks of 8 columns (one converter thread's columns):
    # even blocks cycle over 1 + 2^-7, 2^-120, 0.75 and 3 * 2^90 (the
    # converters' fused multiply-add form), odd blocks over 2^110, 3 * 2^105,
    # 1 + 2^-7 and 2^-120 (a scale of 2^100 or more: the subtract-then-multiply
    # form).  With one-hot input rows both must give the oracle's dequantized
    # weights bit for bit (1 + 2^-7 times odd integers rounds at ties).
    M, K, N, G = 256, 192, 256, 2
    d = _case(M, K, N, G, 1, torch.bfloat16, wdtype, 0, True, False, 56)
    ordinary = [1 + 2.0 ** -7, 2.0 ** -120, 0.75, 3 * 2.0 ** 90]
    huge = [2.0 ** 110, 3 * 2.0 ** 105, 1 + 2.0 ** -7, 2.0 ** -120]
    cols = [(huge if (n // 8) % 2 else ordinary)[n % 4] for n in range(N)]
    d["w_scale"] = torch.tensor(cols, dtype=torch.float64).reshape(1, 1, N).expand(G, 1, N).to(
        torch.bfloat16).contiguous().to(DEV)
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    ks = np.arange(M) % K
    x[np.arange(M), ks] = 1
    d["input"] = x.to(DEV)
    with path(qg.MM_PATH_TENSOR):
        y = _run(d)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    w = oracle.dequantize_linear(d["weights_q"].cpu().numpy(), to_np(d["w_scale"]),
                                 d["w_zero_point"].cpu().numpy(), 0, "bf16")
    gi = d["group_indices"].cpu().numpy()
    assert np.array_equal(to_np(y)[:, 0, :], w[gi[:, 0], ks, :])


def test_qweights_tensor_invalid_indices():
    d = _case(300, 256, 256, 3, 2, torch.bfloat16, torch.int8, 0, True, False, 53)
    gi = torch.from_numpy(np.random.default_rng(54).integers(-1, 4, size=(300, 2)).astype(np.int64)).to(DEV)
    d["group_indices"] = gi
    with path(qg.MM_PATH_TENSOR):
        y = _run(d)
    bad = ((gi < 0) | (gi >= 3)).cpu().numpy()
    d2 = dict(d)
    d2["group_indices"] = torch.where(gi.cpu() < 0, 0, torch.where(gi.cpu() >= 3, 0, gi.cpu())).to(DEV)
    ref, scale = _oracle(d2)
    err = np.abs(to_np(y) - ref) / (scale + 1e-30)
    assert np.max(err[~bad]) <= TOL[torch.bfloat16]
    assert np.all(to_np(y)[bad] == 0)
    assert qg.mm_get_device_status() == "MM_ERR_INDEX_RANGE"


def test_qweights_matches_dequantize_then_grouped():
    # The fused call against the composition the page describes, both on the
    # GPU: dequantize with the oracle's rounding, then mm_grouped_matmul.
    d = _case(500, 512, 512, 2, 2, torch.bfloat16, torch.int8, 0, True, True, 55)
    with path(qg.MM_PATH_TENSOR):
        y = _run(d)
    w = oracle.dequantize_linear(d["weights_q"].cpu().numpy(), to_np(d["w_scale"]),
                                 d["w_zero_point"].cpu().numpy(), 0, "bf16")
    wt = torch.from_numpy(w).to(torch.bfloat16).to(DEV)
    y2 = qg.mm_grouped_matmul(d["input"], wt, d["group_indices"], d["bias"])
    ref, scale = _oracle(d)
    assert max_rel_err(to_np(y), ref, scale) <= 1e-2
    assert max_rel_err(to_np(y2), ref, scale) <= 1e-2


# ------------------------------------------------------------------ 4-bit experts (int4 / uint4, two per byte)

def _pack4(v):
    """Values in [-8, 15] as packed bytes [..., N/2], the even column in the low nibble."""
    u = (np.asarray(v) & 15).astype(np.uint8)
    return u[..., 0::2] | (u[..., 1::2] << 4)


def _case4(M, K, N, G, S, dtype, kind, block, with_zp, with_bias, seed, p=None):
    g = np.random.default_rng(seed)
    kb = -(-K // (block or K))
    signed = kind == "int4"
    q = g.integers(-8, 8, (G, K, N)) if signed else g.integers(0, 16, (G, K, N))
    zp = (g.integers(-3, 4, (G, kb, N)) if signed else g.integers(6, 10, (G, kb, N))) if with_zp else None
    x = torch.from_numpy(g.standard_normal((M, K))).to(dtype)
    scale = torch.from_numpy(g.uniform(0.5, 1.5, (G, kb, N)) / 8.0).to(dtype)
    bias = torch.from_numpy(g.standard_normal((G, N))).to(dtype) if with_bias else None
    probs = p if p is not None else np.full(G, 1.0 / G)
    gi = torch.from_numpy(g.choice(G, size=(M, S), p=probs).astype(np.int32))
    wq = _pack4(q)
    assert np.array_equal(oracle.unpack_4bit(wq, signed), q)    # the layout the oracle reads
    d = {"input": x, "weights_q": torch.from_numpy(wq), "w_scale": scale,
         "w_zero_point": None if zp is None else torch.from_numpy(_pack4(zp)), "block_size": block,
         "group_indices": gi, "bias": bias}
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    d["packed4"] = kind
    return d


def _run4(d):
    return qg.mm_grouped_matmul_qweights(d["input"], d["weights_q"], d["w_scale"], d["w_zero_point"],
                                         d["block_size"], d["group_indices"], d["bias"], packed4=d["packed4"])


def _unpacked4(d):
    signed = d["packed4"] == "int4"
    wq = oracle.unpack_4bit(d["weights_q"].cpu().numpy(), signed)
    zp = None if d["w_zero_point"] is None else oracle.unpack_4bit(d["w_zero_point"].cpu().numpy(), signed)
    return wq, zp


def _check4(d, tol):
    y = _run4(d)
    t = T_NAME[d["input"].dtype]
    wq, zp = _unpacked4(d)
    args = (to_np(d["input"]), wq, to_np(d["w_scale"]), zp, d["block_size"], d["group_indices"].cpu().numpy(),
            None if d["bias"] is None else to_np(d["bias"]), t)
    ref, scale = oracle.grouped_matmul_qweights(*args), oracle.grouped_qweights_abs_scale(*args)
    assert max_rel_err(to_np(y), ref, scale) <= tol
    return y


@pytest.mark.parametrize("policy", [qg.MM_PATH_SIMT, qg.MM_PATH_TENSOR], ids=["simt", "tensor"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("kind", ["int4", "uint4"])
@pytest.mark.parametrize("block,with_zp,with_bias", [(0, True, True), (0, False, False), (64, True, False)])
def test_qweights_4bit(policy, dtype, kind, block, with_zp, with_bias):
    # K = 330: a partial last k-block; N = 384 (192 bytes a row): a partial
    # column tile on the tensor cores.
    d = _case4(300, 330, 384, 4, 2, dtype, kind, block, with_zp, with_bias, 71, p=[0.5, 0.3, 0.15, 0.05])
    with path(policy):
        _check4(d, TOL[dtype])
    assert qg.mm_last_path() == policy
    assert qg.mm_get_device_status() == "MM_OK"


@pytest.mark.parametrize("kind", ["int4", "uint4"])
def test_qweights_4bit_f32_simt(kind):
    d = _case4(100, 70, 48, 3, 2, torch.float32, kind, 16, True, True, 72)
    _check4(d, TOL[torch.float32])
    assert qg.mm_last_path() == qg.MM_PATH_SIMT


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=str)
@pytest.mark.parametrize("kind", ["int4", "uint4"])
def test_qweights_4bit_tensor_dequantized_values_exact(dtype, kind):
    # One-hot input rows: output[m, i, :] = W[g, k(m), :], so the converters'
    # nibble unpacking and arithmetic must give the oracle's dequantized
    # weights bit for bit, over 16 k-blocks (K = 1024) and two column tiles.
    M, K, N, G = 1024, 1024, 512, 2
    d = _case4(M, K, N, G, 1, dtype, kind, 128, True, False, 73)
    x = torch.zeros((M, K), dtype=dtype)
    ks = np.arange(M) % K
    x[np.arange(M), ks] = 1
    d["input"] = x.to(DEV)
    with path(qg.MM_PATH_TENSOR):
        y = _run4(d)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    wq, zp = _unpacked4(d)
    w = oracle.dequantize_linear(wq, to_np(d["w_scale"]), zp, 128, T_NAME[dtype])
    gi = d["group_indices"].cpu().numpy()
    assert np.array_equal(to_np(y)[:, 0, :], w[gi[:, 0], ks, :])


@pytest.mark.parametrize("kind", ["int4", "uint4"])
def test_qweights_4bit_tensor_extreme_scales_exact(kind):
    # As for 8-bit weights: bf16 scales by blocks of 8 columns, ordinary ones
    # (fused multiply-add form) and ones of 2^100 and more (subtract-then-
    # multiply form) alternating, must give the oracle's dequantized weights
    # bit for bit with one-hot input rows.
    M, K, N, G = 256, 192, 256, 2
    d = _case4(M, K, N, G, 1, torch.bfloat16, kind, 0, True, False, 74)
    ordinary = [1 + 2.0 ** -7, 2.0 ** -120, 0.75, 3 * 2.0 ** 90]
    huge = [2.0 ** 110, 3 * 2.0 ** 105, 1 + 2.0 ** -7, 2.0 ** -120]
    cols = [(huge if (n // 8) % 2 else ordinary)[n % 4] for n in range(N)]
    d["w_scale"] = torch.tensor(cols, dtype=torch.float64).reshape(1, 1, N).expand(G, 1, N).to(
        torch.bfloat16).contiguous().to(DEV)
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    ks = np.arange(M) % K
    x[np.arange(M), ks] = 1
    d["input"] = x.to(DEV)
    with path(qg.MM_PATH_TENSOR):
        y = _run4(d)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    wq, zp = _unpacked4(d)
    w = oracle.dequantize_linear(wq, to_np(d["w_scale"]), zp, 0, "bf16")
    gi = d["group_indices"].cpu().numpy()
    assert np.array_equal(to_np(y)[:, 0, :], w[gi[:, 0], ks, :])
