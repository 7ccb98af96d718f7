"""GPU parity of the CUDA-core (SIMT) kernels against the oracle, through the C ABI.

The planner is forced onto the SIMT path, so every operator and every type is
checked on it: MatMul/Gemm for all eight T (integers bit-exact, floats within
the per-element bound), QLinearMatMul for every int8/uint8 combination and
parameter granularity (bit-exact), GroupedMatMul for all four T and both index
types, plus strided/broadcast views and the empty and degenerate cases.
"""

import contextlib
import json
import pathlib

import numpy as np
import pytest
import torch

import oracle
import quantized_gemm_gb300 as qg
from helpers import TOL, from_np, max_rel_err, rand_tensor, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = pathlib.Path(__file__).parent / "golden"
FLOATS = [torch.bfloat16, torch.float16, torch.float32, torch.float64]
INTS = [torch.int32, torch.int64, torch.uint32, torch.uint64]


@contextlib.contextmanager
def policy(p):
    qg.mm_set_path_policy(p)
    try:
        yield
    finally:
        qg.mm_set_path_policy(qg.MM_PATH_AUTO)


def check_matmul(A, B, Y):
    a, b = to_np(A), to_np(B)
    ref = oracle.matmul(a, b)
    y = to_np(Y)
    assert y.shape == ref.shape
    if A.dtype in TOL:
        assert max_rel_err(y, ref, oracle.matmul_abs_scale(a, b)) <= TOL[A.dtype]
    else:
        assert np.array_equal(y, ref)


SHAPES = [((3,), (3,)), ((4,), (2, 4, 3)), ((2, 3), (3, 4)), ((2, 3, 4, 5), (5,)), ((2, 2, 3), (1, 3, 4)),
          ((2, 3, 4), (4, 5)), ((3,), (3, 2)), ((7, 1, 65, 33), (5, 33, 70)), ((130, 200), (200, 67)),
          ((2, 0, 5), (5, 3)), ((4, 0), (0, 6)), ((0, 3, 4), (4, 2))]


@pytest.mark.parametrize("dtype", FLOATS + INTS, ids=str)
@pytest.mark.parametrize("sa,sb", SHAPES)
def test_matmul_simt(dtype, sa, sb):
    A = rand_tensor(sa, dtype, 1, DEV)
    B = rand_tensor(sb, dtype, 2, DEV)
    with policy(qg.MM_PATH_SIMT):
        Y = qg.mm_matmul(A, B)
    torch.cuda.synchronize()
    check_matmul(A, B, Y)


@pytest.mark.parametrize("dtype", [torch.float32, torch.int64, torch.bfloat16], ids=str)
def test_matmul_strided_and_broadcast_views(dtype):
    base = rand_tensor((3, 40, 24), dtype, 3, DEV)
    A = base.transpose(1, 2)                    # [3, 24, 40], column-major matrices
    B = rand_tensor((40, 1, 9), dtype, 4, DEV).expand(40, 5, 9)[:, 2, :]   # [40, 9] with row stride 45
    Bb = rand_tensor((1, 40, 9), dtype, 5, DEV).expand(3, 40, 9)          # batch stride 0
    with policy(qg.MM_PATH_SIMT):
        check_matmul(A, B, qg.mm_matmul(A, B))
        check_matmul(A, Bb, qg.mm_matmul(A, Bb))


def test_matmul_page_examples_on_gpu():
    for ex in json.load(open(GOLDEN / "matmul_examples.json"))["examples"]:
        A = torch.tensor(ex["inputs"]["A"]["values"], dtype=torch.float32, device=DEV)
        B = torch.tensor(ex["inputs"]["B"]["values"], dtype=torch.float32, device=DEV)
        Y = qg.mm_matmul(A, B)
        check_matmul(A, B, Y)
        printed = np.array(ex["outputs"]["Y"]["values"], dtype=np.float64)
        assert np.allclose(to_np(Y), printed, rtol=2e-5, atol=2e-6), ex["name"]


def _gemm_ref(A, B, C, alpha, beta, tA, tB):
    a, b = to_np(A), to_np(B)
    c = None if C is None else to_np(C)
    ref = oracle.gemm(a, b, c, alpha=alpha, beta=beta, transA=tA, transB=tB)
    return ref, (None if A.dtype not in TOL else oracle.gemm_abs_scale(a, b, c, alpha=alpha, beta=beta,
                                                                        transA=tA, transB=tB))


@pytest.mark.parametrize("dtype", FLOATS + INTS, ids=str)
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("c_shape", [None, (), (1,), (70,), (1, 70), (33, 1), (33, 70)])
def test_gemm_simt(dtype, tA, tB, c_shape):
    M, K, N = 33, 47, 70
    A = rand_tensor((K, M) if tA else (M, K), dtype, 11, DEV)
    B = rand_tensor((N, K) if tB else (K, N), dtype, 12, DEV)
    C = None if c_shape is None else rand_tensor(c_shape, dtype, 13, DEV)
    alpha, beta = (0.5, 2.0) if dtype in TOL else (3.0, -2.0)
    with policy(qg.MM_PATH_SIMT):
        Y = qg.mm_gemm(A, B, C, alpha, beta, tA, tB)
    ref, scale = _gemm_ref(A, B, C, alpha, beta, tA, tB)
    if dtype in TOL:
        assert max_rel_err(to_np(Y), ref, scale) <= TOL[dtype]
    else:
        assert np.array_equal(to_np(Y), ref)


def test_gemm_page_examples_on_gpu():
    for ex in json.load(open(GOLDEN / "gemm_examples.json"))["examples"]:
        at = ex["attributes"]
        kw = dict(alpha=at.get("alpha", 1.0), beta=at.get("beta", 1.0),
                  transA=at.get("transA", 0), transB=at.get("transB", 0))
        A = torch.tensor(ex["inputs"]["A"]["values"], dtype=torch.float32, device=DEV)
        B = torch.tensor(ex["inputs"]["B"]["values"], dtype=torch.float32, device=DEV)
        C = None
        if "C" in ex["inputs"]:
            C = torch.tensor(ex["inputs"]["C"]["values"], dtype=torch.float32, device=DEV).reshape(
                ex["inputs"]["C"]["shape"])
        Y = qg.mm_gemm(A, B, C, **kw)
        ref, scale = _gemm_ref(A, B, C, kw["alpha"], kw["beta"], kw["transA"], kw["transB"])
        assert max_rel_err(to_np(Y), ref, scale) <= 1e-5, ex["name"]


def test_gemm_empty_k_gives_beta_c():
    A = torch.empty((5, 0), dtype=torch.float32, device=DEV)
    B = torch.empty((0, 7), dtype=torch.float32, device=DEV)
    C = rand_tensor((5, 1), torch.float32, 3, DEV)
    Y = qg.mm_gemm(A, B, C, 1.0, 3.0)
    assert torch.equal(Y, (3.0 * C).expand(5, 7))


# ------------------------------------------------------------------ QLinearMatMul

def _q_args(d):
    return [d[k] for k in ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale",
                           "y_zero_point")]


def _q_check(d):
    y = qg.mm_qlinear_matmul(*_q_args(d))
    ref = oracle.qlinear_matmul(*[t.cpu().numpy() for t in _q_args(d)])
    got = y.cpu().numpy()
    assert got.dtype == ref.dtype and got.shape == ref.shape
    assert np.array_equal(got, ref)


def _qlinear_case(M, K, N, ta, tb, ty, granularity, scale_dtype=torch.float32, batch=(), seed=0):
    g = np.random.default_rng(seed)
    rng = lambda t, shape: rand_tensor(shape, t, int(g.integers(1 << 30)), DEV)
    a = rng(ta, batch + (M, K))
    b = rng(tb, batch + (K, N))
    if granularity == "tensor":
        sa_shape, sb_shape = (), ()
    elif batch:
        sa_shape, sb_shape = batch + (M, 1), batch + (1, N)
    elif granularity == "vector":
        sa_shape, sb_shape = (M,), (N,)
    else:
        sa_shape, sb_shape = (M, 1), (1, N)
    lo_a, hi_a = (-20, 20) if ta == torch.int8 else (100, 140)
    lo_b, hi_b = (-20, 20) if tb == torch.int8 else (100, 140)
    d = {
        "a": a, "b": b,
        "a_scale": torch.from_numpy(g.uniform(0.003, 0.01, sa_shape).astype(np.float32)).to(scale_dtype).to(DEV),
        "a_zero_point": rand_tensor(sa_shape, ta, int(g.integers(1 << 30)), DEV, lo_a, hi_a),
        "b_scale": torch.from_numpy(g.uniform(0.003, 0.01, sb_shape).astype(np.float32)).to(scale_dtype).to(DEV),
        "b_zero_point": rand_tensor(sb_shape, tb, int(g.integers(1 << 30)), DEV, lo_b, hi_b),
        # about rms(a_scale*b_scale) * rms(acc) / 50: a mix of in-range and saturated outputs
        "y_scale": torch.tensor(0.005 * np.sqrt(K), dtype=scale_dtype, device=DEV),
        "y_zero_point": torch.tensor(-9 if ty == torch.int8 else 120, dtype=ty, device=DEV),
    }
    return d


@pytest.mark.parametrize("ta,tb,ty", [(torch.int8, torch.int8, torch.int8), (torch.uint8, torch.uint8, torch.uint8),
                                      (torch.int8, torch.uint8, torch.int8), (torch.uint8, torch.int8, torch.uint8)],
                         ids=str)
@pytest.mark.parametrize("granularity", ["tensor", "vector", "matrix"])
@pytest.mark.parametrize("scale_dtype", [torch.float32, torch.float16], ids=str)
def test_qlinear_simt(ta, tb, ty, granularity, scale_dtype):
    with policy(qg.MM_PATH_SIMT):
        _q_check(_qlinear_case(67, 131, 45, ta, tb, ty, granularity, scale_dtype))


def test_qlinear_batched_simt():
    with policy(qg.MM_PATH_SIMT):
        _q_check(_qlinear_case(20, 37, 19, torch.int8, torch.int8, torch.int8, "matrix", batch=(2, 3)))


def test_qlinear_page_examples_on_gpu():
    for ex in json.load(open(GOLDEN / "qlinearmatmul_examples.json"))["examples"]:
        i = ex["inputs"]
        ts = {k: torch.from_numpy(np.array(i[k]["values"], dtype=i[k]["dtype"]).reshape(i[k]["shape"])).to(DEV)
              for k in i}
        y = qg.mm_qlinear_matmul(*_q_args(ts))
        want = np.array(ex["outputs"]["y"]["values"], dtype=ex["outputs"]["y"]["dtype"])
        assert np.array_equal(y.cpu().numpy(), want), ex["name"]


def test_qlinear_ties_and_int32_wrap_on_gpu():
    # ties: acc = 1,3,5,-1,-3 with y_scale 2 -> 0,2,2,0,-2
    a = torch.tensor([[1], [3], [5], [-1], [-3]], dtype=torch.int8, device=DEV)
    one = torch.tensor(1.0, device=DEV)
    z8 = torch.tensor(0, dtype=torch.int8, device=DEV)
    b = torch.tensor([[1]], dtype=torch.int8, device=DEV)
    y = qg.mm_qlinear_matmul(a, one, z8, b, one, z8, torch.tensor(2.0, device=DEV), z8)
    assert y.flatten().tolist() == [0, 2, 2, 0, -2]
    # int32 wrap: 65025 * 33026 > 2^31 - 1 wraps negative -> -128
    K = 33026
    a = torch.full((1, K), 255, dtype=torch.uint8, device=DEV)
    bb = torch.full((K, 1), 255, dtype=torch.uint8, device=DEV)
    zu = torch.tensor(0, dtype=torch.uint8, device=DEV)
    y = qg.mm_qlinear_matmul(a, one, zu, bb, one, zu, torch.tensor(2.0 ** 24, device=DEV), z8)
    assert y.item() == -128


# ------------------------------------------------------------------ GroupedMatMul

def _grouped_check(x, w, gi, bias, out):
    xa, wa = to_np(x), to_np(w)
    ba = None if bias is None else to_np(bias)
    gia = gi.cpu().numpy()
    ref = oracle.grouped_matmul(xa, wa, gia, ba)
    scale = oracle.grouped_abs_scale(xa, wa, gia, ba)
    assert out.shape == ref.shape
    assert max_rel_err(to_np(out), ref, scale) <= TOL[x.dtype]


@pytest.mark.parametrize("dtype", FLOATS, ids=str)
@pytest.mark.parametrize("ind", [torch.int32, torch.int64], ids=str)
@pytest.mark.parametrize("with_bias", [False, True])
def test_grouped_simt(dtype, ind, with_bias):
    M, K, N, G, S = 37, 70, 300, 5, 3
    x = rand_tensor((M, K), dtype, 21, DEV)
    w = rand_tensor((G, K, N), dtype, 22, DEV)
    gi = torch.from_numpy(np.random.default_rng(23).integers(0, G, (M, S))).to(ind).to(DEV)
    bias = rand_tensor((G, N), dtype, 24, DEV) if with_bias else None
    with policy(qg.MM_PATH_SIMT):
        out = qg.mm_grouped_matmul(x, w, gi, bias)
    _grouped_check(x, w, gi, bias, out)
    assert qg.mm_get_device_status() == "MM_OK"


def test_grouped_invalid_indices_zero_rows_and_flag():
    M, K, N, G = 6, 16, 40, 3
    x = rand_tensor((M, K), torch.float32, 31, DEV)
    w = rand_tensor((G, K, N), torch.float32, 32, DEV)
    gi = torch.tensor([[0, 1], [-1, 2], [2, 3], [1, 1], [0, 100], [2, 0]], dtype=torch.int64, device=DEV)
    for pol in (qg.MM_PATH_SIMT, qg.MM_PATH_AUTO):
        with policy(pol):
            out = qg.mm_grouped_matmul(x, w, gi)
        assert qg.mm_get_device_status() == "MM_ERR_INDEX_RANGE"
        assert qg.mm_get_device_status() == "MM_OK"   # reading clears it
        bad = (gi < 0) | (gi >= G)
        assert torch.all(out[bad] == 0)
        good = ~bad
        gi_ok = torch.where(good, gi, torch.zeros_like(gi))
        ref = oracle.grouped_matmul(to_np(x), to_np(w), gi_ok.cpu().numpy())
        scale = oracle.grouped_abs_scale(to_np(x), to_np(w), gi_ok.cpu().numpy())
        err = np.abs(to_np(out) - ref) / (scale + 1e-30)
        assert np.max(err[good.cpu().numpy()]) <= 1e-5


def test_grouped_empty_and_page_examples():
    f = torch.float32
    x = torch.arange(6, dtype=f, device=DEV).reshape(2, 3)
    w = torch.arange(24, dtype=f, device=DEV).reshape(2, 3, 4)
    assert qg.mm_grouped_matmul(x, w, torch.empty((2, 0), dtype=torch.int64, device=DEV)).shape == (2, 0, 4)
    assert qg.mm_grouped_matmul(torch.empty((0, 3), dtype=f, device=DEV), w,
                                torch.empty((0, 2), dtype=torch.int64, device=DEV)).shape == (0, 2, 4)
    # _with_unused_group (GroupedMatMul - 29, Examples): hand-derived output
    x = torch.tensor([[1, 2], [3, 4], [5, 6], [7, 8]], dtype=f, device=DEV)
    w = torch.arange(12, dtype=f, device=DEV).reshape(3, 2, 2)
    gi = torch.tensor([[0], [0], [2], [2]], dtype=torch.int64, device=DEV)
    out = qg.mm_grouped_matmul(x, w, gi)
    assert out.cpu().tolist() == [[[4, 7]], [[8, 15]], [[100, 111]], [[136, 151]]]


@pytest.mark.parametrize("dtype", [np.int32, np.uint32, np.int64, np.uint64], ids=lambda t: np.dtype(t).name)
@pytest.mark.parametrize("alpha,beta", [(0.37, -1.25), (-2.5, 0.5), (0.5, 1.0)])
def test_gemm_integer_non_integral_alpha_beta(dtype, alpha, beta):
    # trunc(alpha * acc + beta * C) in float64, the accumulator wrapped in T
    # first (the integer-Gemm reading): bit-exact against the oracle on values
    # that stay inside T's range.
    g = np.random.default_rng(80)
    lo = 0 if np.dtype(dtype).kind == "u" else -20
    A = g.integers(lo, 21, (70, 33)).astype(dtype)
    B = g.integers(lo, 21, (33, 45)).astype(dtype)
    C = g.integers(lo, 21, (1, 45)).astype(dtype)
    if np.dtype(dtype).kind == "u" and (alpha < 0 or beta < 0):
        A, C = A // 4, C * 0          # keep unsigned results non-negative
        alpha, beta = abs(alpha), abs(beta)
    ref = oracle.gemm(A, B, C, alpha=alpha, beta=beta)
    Y = qg.mm_gemm(from_np(A, DEV), from_np(B, DEV), from_np(C, DEV), alpha, beta, 0, 0)
    assert qg.mm_last_path() == qg.MM_PATH_SIMT
    assert np.array_equal(Y.cpu().numpy(), ref)


def test_gemm_integer_non_integral_saturates():
    # Outside T's range the reading leaves the value undefined; the kernels saturate.
    A = from_np(np.array([[2 ** 31 - 1, 2 ** 31 - 1]], np.int32), DEV)
    B = from_np(np.array([[1], [-1]], np.int32), DEV)
    Y = qg.mm_gemm(A, B, None, 1.5, 1.0, 0, 0)                     # acc = 0 -> 0
    assert Y.item() == 0
    Y = qg.mm_gemm(A[:, :1], B[:1], None, 1.5, 1.0, 0, 0)          # 1.5 * (2^31 - 1) > 2^31 - 1
    assert Y.item() == 2 ** 31 - 1


# Shapes that select each register tile of the tiled CUDA-core kernel (8 x 8
# threads' outputs in 128 x 128 blocks when there are at least as many such
# blocks as SMs, 4 x 4 in 64 x 64 blocks, else 2 x 2), with ragged M, N and K
# tails, in every layout its loads distinguish: 16-byte vectors along k (A
# row-major, B stored [N, K]), along m / n (A stored [K, M], B row-major) and
# element by element (an odd row stride).
TILE_CASES = [
    (torch.float32, 1300, 1800, 97),    # 8 x 8 (165 blocks of 128 x 128)
    (torch.int32, 1300, 1800, 97),
    (torch.bfloat16, 1300, 1800, 97),
    (torch.float32, 900, 700, 200),     # 4 x 4
    (torch.uint32, 900, 700, 200),
    (torch.float64, 700, 900, 61),      # 64-bit: 4 x 4 (165 blocks of 64 x 64)
    (torch.int64, 700, 900, 61),
    (torch.float64, 100, 90, 150),      # 2 x 2
]


@pytest.mark.parametrize("dtype,M,N,K", TILE_CASES, ids=lambda v: str(v))
@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1), (0, 1)])
def test_gemm_simt_register_tiles(dtype, M, N, K, tA, tB):
    A = rand_tensor((K, M) if tA else (M, K), dtype, 41, DEV)
    B = rand_tensor((N, K) if tB else (K, N), dtype, 42, DEV)
    alpha, beta = (1.0, 0.0)
    with policy(qg.MM_PATH_SIMT):
        Y = qg.mm_gemm(A, B, None, alpha, beta, tA, tB)
    assert qg.mm_last_path() == qg.MM_PATH_SIMT
    ref, scale = _gemm_ref(A, B, None, alpha, beta, tA, tB)
    if dtype in TOL:
        assert max_rel_err(to_np(Y), ref, scale) <= TOL[dtype]
    else:
        assert np.array_equal(to_np(Y), ref)


@pytest.mark.parametrize("dtype", [torch.float32, torch.int32, torch.float64], ids=str)
def test_gemm_simt_register_tiles_scalar_loads(dtype):
    # Row strides of 1301 / 1803 elements: no 16-byte alignment, so both
    # operands take the element-by-element loads, with a C broadcast row.
    M, N, K = 1300, 1800, 70
    Ab = rand_tensor((M, K + 1), dtype, 43, DEV)[:, 1:]
    Bb = rand_tensor((K, N + 3), dtype, 44, DEV)[:, 3:]
    C = rand_tensor((N,), dtype, 45, DEV)
    alpha, beta = (0.5, 2.0) if dtype in TOL else (3.0, -2.0)
    with policy(qg.MM_PATH_SIMT):
        Y = qg.mm_gemm(Ab, Bb, C, alpha, beta, 0, 0)
    ref, scale = _gemm_ref(Ab, Bb, C, alpha, beta, 0, 0)
    if dtype in TOL:
        assert max_rel_err(to_np(Y), ref, scale) <= TOL[dtype]
    else:
        assert np.array_equal(to_np(Y), ref)
