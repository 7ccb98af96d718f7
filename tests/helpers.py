"""Test helpers: tensor conversions, tolerances and seeded random tensors.

Float parity is the per-element bound
    |Y - Y_ref| / (sum_k |A_ik| |B_kj| * |alpha| + |beta * C_ij| + 1e-30) <= tol
with tol = 1e-2 for bf16/f16 inputs (fp32 accumulation, one rounding to the
16-bit type), 1e-5 for f32 (fp32 FFMA accumulation, never TF32) and 1e-12 for
f64.  Integer and quantized results must be bit-exact.
"""

import numpy as np
import torch

TOL = {torch.bfloat16: 1e-2, torch.float16: 1e-2, torch.float32: 1e-5, torch.float64: 1e-12}

INT_TORCH = {torch.int32: np.int32, torch.int64: np.int64, torch.uint32: np.uint32, torch.uint64: np.uint64}


def to_np(t):
    """Exact host copy: floats widened to float64, integers kept in their type."""
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32, torch.float64):
        return t.to(torch.float64).numpy()
    if t.dtype in (torch.uint32, torch.uint64):
        signed = torch.int32 if t.dtype == torch.uint32 else torch.int64
        return t.view(signed).numpy().view(INT_TORCH[t.dtype])
    return t.numpy()


def from_np(a, device):
    """Device tensor holding numpy array ``a`` (unsigned 32/64-bit types included)."""
    a = np.array(a, order="C", copy=True)   # keeps 0-d arrays 0-d
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).view(torch.uint32).to(device)
    if a.dtype == np.uint64:
        return torch.from_numpy(a.view(np.int64)).view(torch.uint64).to(device)
    return torch.from_numpy(a).to(device)


def max_rel_err(got, ref, scale):
    got = np.asarray(got, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (scale + 1e-30)))


def rand_tensor(shape, dtype, seed, device, lo=None, hi=None):
    """Seeded tensor: N(0,1) for floats, full-range uniform for integers."""
    rng = np.random.default_rng(seed)
    if dtype in TOL:
        x = rng.standard_normal(shape).astype(np.float32)
        t = torch.from_numpy(x).to(dtype)
        return t.to(device)
    npdt = INT_TORCH.get(dtype, {torch.int8: np.int8, torch.uint8: np.uint8}.get(dtype))
    info = np.iinfo(npdt)
    lo = info.min if lo is None else lo
    hi = info.max if hi is None else hi
    x = rng.integers(lo, hi, size=shape, dtype=npdt, endpoint=True)
    return from_np(x, device)
