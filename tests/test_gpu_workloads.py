"""Parity at the benchmark sizes, in the launch configuration bench.py times.

Each workload runs once at full size through the public API (auto planner,
which must choose the tensor-core kernels for the four large workloads).  Two
checks then cover its output:

* every column of sampled rows: the numpy oracle recomputes tile-boundary and
  seeded random rows (a row of a product depends only on the matching row of
  A, so the oracle is given those rows);
* every row of sampled columns: the C++ oracle recomputes the whole output on
  a column subset (a column depends only on the matching column of B' and of
  the per-column parameters) that holds the first and last columns and one
  column of every 128-wide column block.  Every row tile of the persistent
  raster, every (row tile, column tile) pair of the subset and, for
  GroupedMatMul, every routed row of every group is checked.

Float results are held to the per-element bound, QLinearMatMul results must
be bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
import oracle.native
import quantized_gemm_gb300 as qg
import workloads
from helpers import max_rel_err, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(n, extra, seed):
    fixed = [0, 1, 127, 128, 255, 256, n // 2, n - 129, n - 128, n - 1]
    rnd = np.random.default_rng(seed).choice(n, size=extra, replace=False)
    return sorted(set(int(r) for r in fixed + list(rnd) if 0 <= r < n))


def _cols(n, seed, least=64):
    """Column subset: both ends, the edges around column 128 and 256, one seeded
    column in every 128-wide block, and seeded extras up to `least` columns."""
    g = np.random.default_rng(seed)
    cols = {0, 1, 127, 128, 255, 256, n - 2, n - 1}
    cols |= {int(b + g.integers(0, min(128, n - b))) for b in range(0, n, 128)}
    rest = np.setdiff1d(np.arange(n), np.fromiter(cols, dtype=np.int64))
    if len(cols) < least and rest.size:
        cols |= set(int(c) for c in g.choice(rest, size=min(least - len(cols), rest.size), replace=False))
    return np.array(sorted(c for c in cols if 0 <= c < n), dtype=np.int64)


def test_matmul_f32_full():
    """The small f32 workload runs on the CUDA cores (FFMA) in the tiled
    kernel: the [4,128,64] @ [64,96] product (3.1 M multiply-adds, below the
    2^24 at which three tf32 products pay) and the promoted 1-D one (24576
    elements of B', below the 2^17 at which the few-row kernel pays)."""
    d = workloads.matmul_f32(device=DEV)
    for (a, b), path in (((d["A"], d["B"]), qg.MM_PATH_SIMT), ((d["A1"], d["B1"]), qg.MM_PATH_SIMT)):
        y = qg.mm_matmul(a, b)
        assert qg.mm_last_path() == path
        an, bn = to_np(a), to_np(b)
        assert max_rel_err(to_np(y), oracle.matmul(an, bn), oracle.matmul_abs_scale(an, bn)) <= 1e-5


def test_gemm_bf16_8192_sampled_rows():
    d = workloads.gemm_bf16(device=DEV)
    Y = qg.mm_gemm(d["A"], d["B"], d["C"], d["alpha"], d["beta"], d["transA"], d["transB"])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    rows = _rows(8192, 22, 1)
    A = to_np(d["A"][rows])
    B = to_np(d["B"])
    C = to_np(d["C"])
    kw = dict(alpha=d["alpha"], beta=d["beta"], transA=0, transB=1)
    ref = oracle.gemm(A, B, C, **kw)
    assert max_rel_err(to_np(Y[rows]), ref, oracle.gemm_abs_scale(A, B, C, **kw)) <= 1e-2
    assert torch.isfinite(Y.float()).all()
    # every row, on a column subset (transB = 1: output column j is row j of B)
    cols = _cols(8192, 21)
    ct = torch.from_numpy(cols).to(DEV)
    A = to_np(d["A"])
    Bs = to_np(d["B"][ct])
    Cs = to_np(d["C"][:, ct])
    ref = oracle.native.gemm(A, Bs, Cs, **kw)
    assert max_rel_err(to_np(Y[:, ct]), ref, oracle.native.gemm_abs_scale(A, Bs, Cs, **kw)) <= 1e-2


def test_gemm_f32_8192_sampled_rows():
    """The headline Gemm in fp32: three-tf32 tensor-core products within 1e-5."""
    d = workloads.gemm_bf16(device=DEV, dtype=torch.float32)
    Y = qg.mm_gemm(d["A"], d["B"], d["C"], d["alpha"], d["beta"], d["transA"], d["transB"])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    rows = _rows(8192, 10, 11)
    A = to_np(d["A"][rows])
    B = to_np(d["B"])
    C = to_np(d["C"])
    kw = dict(alpha=d["alpha"], beta=d["beta"], transA=0, transB=1)
    ref = oracle.gemm(A, B, C, **kw)
    assert max_rel_err(to_np(Y[rows]), ref, oracle.gemm_abs_scale(A, B, C, **kw)) <= 1e-5
    cols = _cols(8192, 22)
    ct = torch.from_numpy(cols).to(DEV)
    A = to_np(d["A"])
    Bs = to_np(d["B"][ct])
    Cs = to_np(d["C"][:, ct])
    ref = oracle.native.gemm(A, Bs, Cs, **kw)
    assert max_rel_err(to_np(Y[:, ct]), ref, oracle.native.gemm_abs_scale(A, Bs, Cs, **kw)) <= 1e-5


def test_matmul_bf16_bcast_sampled():
    d = workloads.matmul_bf16_bcast(device=DEV)
    Y = qg.mm_matmul(d["A"], d["B"])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    g = np.random.default_rng(2)
    for b0, b1 in [(0, 0), (7, 31), (3, 17)] + [tuple(g.integers(0, (8, 32))) for _ in range(3)]:
        rows = _rows(2048, 6, int(b0 * 32 + b1))
        A = to_np(d["A"][b0, b1][rows])
        B = to_np(d["B"][0, b1])
        ref = oracle.matmul(A, B)
        assert max_rel_err(to_np(Y[b0, b1][rows]), ref, oracle.matmul_abs_scale(A, B)) <= 1e-2
    # every row of every batch index, on a column subset
    cols = _cols(2048, 23)
    ct = torch.from_numpy(cols).to(DEV)
    A = to_np(d["A"])
    Bs = to_np(d["B"][..., ct])
    ref = oracle.native.matmul(A, Bs)
    assert max_rel_err(to_np(Y[..., ct]), ref, oracle.native.matmul_abs_scale(A, Bs)) <= 1e-2


def test_qlinear_s8_sampled_rows_bit_exact():
    d = workloads.qlinear_s8(device=DEV)
    keys = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")
    y = qg.mm_qlinear_matmul(*[d[k] for k in keys])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    rows = _rows(16384, 14, 3)
    h = {k: d[k].cpu().numpy() for k in keys}
    ref = oracle.qlinear_matmul(h["a"][rows], h["a_scale"][rows], h["a_zero_point"][rows], h["b"], h["b_scale"],
                                h["b_zero_point"], h["y_scale"], h["y_zero_point"])
    got = y[rows].cpu().numpy()
    assert np.array_equal(got, ref), "%d mismatching outputs" % int((got != ref).sum())
    sat = float(((y == 127) | (y == -128)).float().mean())
    assert 0.001 < sat < 0.05      # the workload's y_scale saturates about 1% of outputs
    _qlinear_all_rows(h, y.cpu().numpy(), 24)


def _qlinear_all_rows(h, yh, seed):
    """Every row against the C++ oracle on a column subset of b and its per-column parameters."""
    cols = _cols(h["b"].shape[-1], seed)

    def colsel(x):
        x = np.asarray(x)
        return x[..., cols] if x.ndim >= 1 and x.shape[-1] == h["b"].shape[-1] and x.size > 1 else x
    ref = oracle.native.qlinear_matmul(h["a"], h["a_scale"], h["a_zero_point"], colsel(h["b"]), colsel(h["b_scale"]),
                                       colsel(h["b_zero_point"]), h["y_scale"], h["y_zero_point"])
    got = yh[..., cols]
    assert np.array_equal(got, ref), "%d mismatching outputs" % int((got != ref).sum())


@pytest.mark.parametrize("name", sorted(workloads.QLINEAR_VARIANTS))
def test_qlinear_variants_sampled_rows_bit_exact(name):
    """uint8 and mixed operands, float16 scales, batch-indexed parameters at full size."""
    d = workloads.qlinear(device=DEV, **workloads.QLINEAR_VARIANTS[name])
    keys = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")
    y = qg.mm_qlinear_matmul(*[d[k] for k in keys])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    h = {k: d[k].cpu().numpy() for k in keys}
    yh = y.cpu().numpy()
    batched = h["a"].ndim == 3
    for bi in range(h["a"].shape[0] if batched else 1):
        sel = (lambda x: x[bi]) if batched else (lambda x: x)
        rows = _rows(sel(h["a"]).shape[0], 8, 10 + bi)
        ref = oracle.qlinear_matmul(sel(h["a"])[rows], sel(h["a_scale"])[rows], sel(h["a_zero_point"])[rows],
                                    sel(h["b"]), sel(h["b_scale"]), sel(h["b_zero_point"]), h["y_scale"],
                                    h["y_zero_point"])
        got = sel(yh)[rows]
        assert np.array_equal(got, ref), "%d mismatching outputs" % int((got != ref).sum())
    _qlinear_all_rows(h, yh, 25)
    info = np.iinfo(yh.dtype)
    sat = float(((yh == info.max) | (yh == info.min)).mean())
    assert 0.001 < sat < 0.05


def test_grouped_f16_int64_indices_sampled():
    d = workloads.grouped_bf16(device=DEV, dtype=torch.float16, index_dtype=torch.int64)
    _grouped_check(d, seed=6)


def test_grouped_bf16_8_groups_sampled():
    """Eight groups of 4096 routed rows on average: the CTA-pair tiles."""
    d = workloads.grouped_bf16(device=DEV, G=8)
    _grouped_check(d, seed=8)


def test_grouped_bf16_sampled_tokens_and_columns():
    d = workloads.grouped_bf16(device=DEV)
    _grouped_check(d, seed=4)


def _grouped_check(d, seed):
    out = qg.mm_grouped_matmul(d["input"], d["weights"], d["group_indices"], d["bias"])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    toks = _rows(16384, 6, seed)
    cols = np.sort(np.random.default_rng(seed + 1).choice(14336, size=512, replace=False))
    gi = d["group_indices"][toks].cpu().numpy()
    used = sorted(set(gi.ravel().tolist()))
    remap = {g: j for j, g in enumerate(used)}
    gi_local = np.vectorize(remap.get)(gi).astype(np.int64)
    used_t = torch.tensor(used, device=DEV)
    cols_t = torch.from_numpy(cols).to(DEV)
    w = to_np(d["weights"][used_t][:, :, cols_t])
    bias = to_np(d["bias"][used_t][:, cols_t])
    x = to_np(d["input"][toks])
    ref = oracle.grouped_matmul(x, w, gi_local, bias)
    scale = oracle.grouped_abs_scale(x, w, gi_local, bias)
    got = to_np(out[toks][:, :, cols_t])
    assert max_rel_err(got, ref, scale) <= 1e-2
    # every routed row of every group, on a column subset
    cols = _cols(d["weights"].shape[2], seed + 2)
    ct = torch.from_numpy(cols).to(DEV)
    x = to_np(d["input"])
    w = to_np(d["weights"][:, :, ct])
    bias = to_np(d["bias"][:, ct])
    gi = d["group_indices"].cpu().numpy()
    ref = oracle.native.grouped_matmul(x, w, gi, bias)
    scale = oracle.native.grouped_abs_scale(x, w, gi, bias)
    assert max_rel_err(to_np(out[:, :, ct]), ref, scale) <= 1e-2


@pytest.mark.parametrize("block", [0, 128])
def test_grouped_qweights_sampled_tokens_and_columns(block):
    """int8 weight-only experts at the GroupedMatMul workload's size, fused dequantization."""
    d = workloads.grouped_qweights(device=DEV, block=block)
    out = qg.mm_grouped_matmul_qweights(d["input"], d["weights_q"], d["w_scale"], d["w_zero_point"],
                                        d["block_size"], d["group_indices"], d["bias"])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    toks = _rows(16384, 6, 9)
    cols = np.sort(np.random.default_rng(10).choice(14336, size=512, replace=False))
    gi = d["group_indices"][toks].cpu().numpy()
    used = sorted(set(gi.ravel().tolist()))
    gi_local = np.vectorize({g: j for j, g in enumerate(used)}.get)(gi).astype(np.int64)
    used_t = torch.tensor(used, device=DEV)
    cols_t = torch.from_numpy(cols).to(DEV)
    wq = d["weights_q"][used_t][:, :, cols_t].cpu().numpy()
    sc = to_np(d["w_scale"][used_t][:, :, cols_t])
    zp = d["w_zero_point"][used_t][:, :, cols_t].cpu().numpy()
    bias = to_np(d["bias"][used_t][:, cols_t])
    x = to_np(d["input"][toks])
    args = (x, wq, sc, zp, block, gi_local, bias, "bf16")
    ref = oracle.grouped_matmul_qweights(*args)
    scale = oracle.grouped_qweights_abs_scale(*args)
    got = to_np(out[toks][:, :, cols_t])
    assert max_rel_err(got, ref, scale) <= 1e-2
    # every routed row of every group, on a column subset
    cols = _cols(14336, 26)
    ct = torch.from_numpy(cols).to(DEV)
    args = (to_np(d["input"]), d["weights_q"][:, :, ct].cpu().numpy(), to_np(d["w_scale"][:, :, ct]),
            d["w_zero_point"][:, :, ct].cpu().numpy(), block, d["group_indices"].cpu().numpy(),
            to_np(d["bias"][:, ct]), "bf16")
    ref = oracle.native.grouped_matmul_qweights(*args)
    scale = oracle.native.grouped_qweights_abs_scale(*args)
    assert max_rel_err(to_np(out[:, :, ct]), ref, scale) <= 1e-2



def test_grouped_qweights_int4_all_rows_on_column_subset():
    """int4 weight-only experts (two per byte) at the GroupedMatMul workload's
    size: every routed row of every group on a column subset, against the C++
    oracle given the unpacked values."""
    d = workloads.grouped_qweights(device=DEV, bits=4)
    out = qg.mm_grouped_matmul_qweights(d["input"], d["weights_q"], d["w_scale"], d["w_zero_point"],
                                        d["block_size"], d["group_indices"], d["bias"], packed4=d["packed4"])
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"
    cols = _cols(14336, 27)
    ct = torch.from_numpy(cols).to(DEV)
    # the bytes holding the subset's columns, unpacked: column c is element
    # 2j + c % 2 of the unpacked subset when byte j is byte c // 2
    bt = torch.from_numpy(cols // 2).to(DEV)
    pick = 2 * np.arange(len(cols)) + cols % 2
    wq = oracle.unpack_4bit(d["weights_q"][:, :, bt].cpu().numpy(), True)[:, :, pick]
    zp = oracle.unpack_4bit(d["w_zero_point"][:, :, bt].cpu().numpy(), True)[:, :, pick]
    args = (to_np(d["input"]), wq, to_np(d["w_scale"][:, :, ct]), zp, 0, d["group_indices"].cpu().numpy(),
            to_np(d["bias"][:, ct]), "bf16")
    ref = oracle.native.grouped_matmul_qweights(*args)
    scale = oracle.native.grouped_qweights_abs_scale(*args)
    assert max_rel_err(to_np(out[:, :, ct]), ref, scale) <= 1e-2
