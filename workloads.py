"""Seeded synthetic inputs for the five benchmark workloads and the parity tests.

This module only draws random inputs; it holds none of the operators'
arithmetic and is shared, unchanged, by the CUDA-path tests, the oracle-side
checks and bench.py.  Every generator takes an explicit seed.  Inputs of the
large bfloat16 workloads are drawn on the target device with a seeded
torch.Generator (drawing 3.8 G values on the host would take minutes); the
int8 workload is drawn on the host so that its stored y_scale can be derived
on any machine.

Workloads (shapes and distributions as specified for the benchmark):

1. ``matmul_f32``      f32 MatMul A[4,128,64] @ B[64,96] (B broadcast over the
                       batch) and the 1-D promotion A[64] @ B[4,64,96]; N(0,1).
2. ``gemm_bf16``       bf16 Gemm M=N=K=8192, transB=1 (B stored [N,K]),
                       alpha=0.5, beta=2.0, C bf16 [1,8192]; A, B ~ N(0,1)/sqrt(8192)
                       (drawn in fp32, rounded to bf16), C ~ N(0,1).
3. ``matmul_bf16_bcast`` bf16 MatMul A[8,32,2048,128] @ B[1,32,128,2048]
                       (B broadcast on dim 0); N(0,1).
4. ``qlinear_s8``      QLinearMatMul a int8 [16384,4096] ~ U{-128..127},
                       a_scale [16384,1] ~ U(0.003,0.01) f32, a_zero_point
                       [16384,1] ~ U{-20..20}; b int8 [4096,4096] ~ U{-128..127},
                       b_scale [1,4096] ~ U(0.003,0.01), b_zero_point [1,4096]
                       ~ U{-20..20}; y_zero_point = -9; y_scale is the stored
                       value that makes about 1% of outputs saturate.
5. ``grouped_bf16``    GroupedMatMul input [16384,4096] ~ N(0,1), weights
                       [64,4096,14336] ~ N(0,1)/64, bias [64,14336] ~ 0.1*N(0,1),
                       group_indices int32 [16384,2]: two distinct groups per
                       token drawn without replacement from a Zipf(s=1.1)
                       popularity p_g ~ (g+1)^-1.1 over G=64.

Variants of 4 and 5 at the same sizes (``QLINEAR_VARIANTS``; ``grouped_bf16``
with ``dtype`` float16 and int64 indices) cover the other operand types,
float16 scales and batch-indexed quantisation parameters; ``grouped_qweights``
is the GroupedMatMul workload with int8 weight-only quantized experts.
"""

import json
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
YSCALE_FILE = os.path.join(HERE, "tests", "golden", "qlinear_s8_yscale.json")

WORKLOADS = {
    "matmul_f32": "f32 MatMul A[4,128,64] @ B[64,96]; A[64] @ B[4,64,96]",
    "gemm_bf16": "bf16 Gemm 8192x8192x8192, transB=1, alpha=0.5, beta=2.0, C[1,8192]",
    "matmul_bf16_bcast": "bf16 MatMul A[8,32,2048,128] @ B[1,32,128,2048]",
    "qlinear_s8": "QLinearMatMul s8 a[16384,4096] per-row, b[4096,4096] per-column, y s8",
    "grouped_bf16": "GroupedMatMul bf16 M=16384 S=2 G=64 K=4096 N=14336, Zipf(1.1) routing",
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, device="cpu", seed=0, std=1.0, dtype=torch.float32):
    """N(0, std^2) drawn in fp32 and rounded (RNE) to ``dtype``."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform_int(shape, lo, hi, dtype, device="cpu", seed=0):
    """Integers uniform on {lo, ..., hi}."""
    return torch.randint(lo, hi + 1, shape, generator=_gen(device, seed), device=device,
                         dtype=torch.int64).to(dtype)


def uniform(shape, lo, hi, device="cpu", seed=0, dtype=torch.float32):
    x = torch.rand(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    return (x * (hi - lo) + lo).to(dtype)


def zipf_two_distinct(M, G, S=2, s=1.1, device="cpu", seed=0, dtype=torch.int32):
    """[M, S] group indices: S distinct groups per token, p_g proportional to (g+1)^-s."""
    p = torch.arange(1, G + 1, dtype=torch.float64).pow(-s)
    p = (p / p.sum()).to(torch.float32)
    idx = torch.multinomial(p.expand(M, G), S, replacement=False, generator=_gen("cpu", seed))
    return idx.to(dtype).to(device)


# ------------------------------------------------------------------ the five workloads

def matmul_f32(device="cpu", seed=0):
    return {
        "A": normal((4, 128, 64), device, seed), "B": normal((64, 96), device, seed + 1),
        "A1": normal((64,), device, seed + 2), "B1": normal((4, 64, 96), device, seed + 3),
    }


def gemm_bf16(device="cuda", seed=0, M=8192, N=8192, K=8192, dtype=torch.bfloat16):
    """The headline Gemm; with dtype float32 the same draws kept in fp32."""
    std = 1.0 / math.sqrt(K)
    return {
        "A": normal((M, K), device, seed, std, dtype),
        "B": normal((N, K), device, seed + 1, std, dtype),   # stored [N, K]: transB = 1
        "C": normal((1, N), device, seed + 2, 1.0, dtype),
        "alpha": 0.5, "beta": 2.0, "transA": 0, "transB": 1,
    }


def matmul_bf16_bcast(device="cuda", seed=0, batch=(8, 32), M=2048, N=2048, K=128):
    return {
        "A": normal(tuple(batch) + (M, K), device, seed, 1.0, torch.bfloat16),
        "B": normal((1, batch[1], K, N), device, seed + 1, 1.0, torch.bfloat16),
    }


def qlinear_yscale():
    with open(YSCALE_FILE) as f:
        return float(json.load(f)["y_scale"])


def qlinear_s8(device="cpu", seed=0, M=16384, N=4096, K=4096, y_scale=None):
    return qlinear(device, seed, M, N, K, y_scale=y_scale)


def qlinear(device="cpu", seed=0, M=16384, N=4096, K=4096, y_scale=None, a_u8=False, b_u8=False, y_u8=False,
            scale_dtype=torch.float32, batch=None):
    """The int8 QLinearMatMul workload and its variants.

    A uint8 operand is the int8 draw plus 128, with its zero points plus 128,
    so x - zero_point (and with it every accumulator) has the same distribution
    as in the int8 workload; a uint8 output takes y_zero_point -9 + 128.  With
    ``scale_dtype`` float16 every scale is rounded to float16.  With ``batch``
    B, a is [B, M/B, K] (the int8 draw reshaped) with per-row parameters
    [B, M/B, 1], and b [B, K, N] has per-column parameters [B, 1, N]: each batch
    index has its own b and its own scales and zero points.
    """
    nb = 1 if batch is None else batch
    d = {
        "a": uniform_int((M, K), -128, 127, torch.int8, "cpu", seed),
        "a_scale": uniform((M, 1), 0.003, 0.01, "cpu", seed + 1),
        "a_zero_point": uniform_int((M, 1), -20, 20, torch.int8, "cpu", seed + 2),
        "b": uniform_int((nb, K, N), -128, 127, torch.int8, "cpu", seed + 3),
        "b_scale": uniform((nb, 1, N), 0.003, 0.01, "cpu", seed + 4),
        "b_zero_point": uniform_int((nb, 1, N), -20, 20, torch.int8, "cpu", seed + 5),
        "y_scale": torch.tensor(qlinear_yscale() if y_scale is None else y_scale, dtype=torch.float32),
        "y_zero_point": torch.tensor(-9, dtype=torch.int8),
    }
    if batch is None:
        for k in ("b", "b_scale", "b_zero_point"):
            d[k] = d[k][0]
    else:
        for k in ("a", "a_scale", "a_zero_point"):
            d[k] = d[k].reshape((batch, M // batch) + tuple(d[k].shape[1:]))
    for k, flag in (("a", a_u8), ("a_zero_point", a_u8), ("b", b_u8), ("b_zero_point", b_u8),
                    ("y_zero_point", y_u8)):
        if flag:
            d[k] = (d[k].to(torch.int16) + 128).to(torch.uint8)
    for k in ("a_scale", "b_scale", "y_scale"):
        d[k] = d[k].to(scale_dtype)
    return {k: v.contiguous().to(device) for k, v in d.items()}


QLINEAR_VARIANTS = {
    "qlinear_u8": dict(a_u8=True, b_u8=True, y_u8=True),
    "qlinear_u8s8_f16scales": dict(a_u8=True, y_u8=False, scale_dtype=torch.float16),
    "qlinear_s8_batched4": dict(batch=4),
}


def grouped_bf16(device="cuda", seed=0, M=16384, K=4096, N=14336, G=64, S=2, dtype=torch.bfloat16,
                 index_dtype=torch.int32):
    return {
        "input": normal((M, K), device, seed, 1.0, dtype),
        "weights": normal((G, K, N), device, seed + 1, 1.0 / 64, dtype),
        "bias": normal((G, N), device, seed + 2, 0.1, dtype),
        "group_indices": zipf_two_distinct(M, G, S, 1.1, device, seed + 3, index_dtype),
    }


def grouped_qweights(device="cuda", seed=0, M=16384, K=4096, N=14336, G=64, S=2, block=0, dtype=torch.bfloat16,
                     bits=8):
    """The GroupedMatMul workload with weight-only int8 experts.

    Same input, routing and bias as ``grouped_bf16``; weights_q int8 [G,K,N]
    uniform on {-128..127}, zero points int8 uniform on {-8..8} and scales
    uniform on (1.5e-4, 2.7e-4) rounded to ``dtype``, one per group and output
    column (block 0) or per ``block`` rows of K, so that the dequantized
    weights have about the standard deviation 1/64 of the bf16 workload.

    bits=4: int4 experts stored two per byte along N (uint8 [G, K, N/2] and
    zero points [G, Kb, N/2], the even column in the low nibble; pass
    ``packed4="int4"``): values uniform on {-8..7} (uniform random bytes),
    zero points on {-1..1}, scales 16 times larger (2.4e-3, 4.3e-3).
    """
    kb = 1 if block == 0 else -(-K // block)
    if bits == 4:
        z = uniform_int((G, kb, N), -1, 1, torch.int8, device, seed + 5).to(torch.int16) & 15
        return {
            "input": normal((M, K), device, seed, 1.0, dtype),
            "weights_q": uniform_int((G, K, N // 2), 0, 255, torch.uint8, device, seed + 1),
            "w_scale": uniform((G, kb, N), 2.4e-3, 4.3e-3, device, seed + 4, dtype),
            "w_zero_point": (z[..., 0::2] | (z[..., 1::2] << 4)).to(torch.uint8),
            "block_size": block,
            "bias": normal((G, N), device, seed + 2, 0.1, dtype),
            "group_indices": zipf_two_distinct(M, G, S, 1.1, device, seed + 3),
            "packed4": "int4",
        }
    return {
        "input": normal((M, K), device, seed, 1.0, dtype),
        "weights_q": uniform_int((G, K, N), -128, 127, torch.int8, device, seed + 1),
        "w_scale": uniform((G, kb, N), 1.5e-4, 2.7e-4, device, seed + 4, dtype),
        "w_zero_point": uniform_int((G, kb, N), -8, 8, torch.int8, device, seed + 5),
        "block_size": block,
        "bias": normal((G, N), device, seed + 2, 0.1, dtype),
        "group_indices": zipf_two_distinct(M, G, S, 1.1, device, seed + 3),
    }

