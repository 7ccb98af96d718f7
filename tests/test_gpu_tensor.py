"""GPU parity of the tcgen05 tensor-core path against the oracle, through the C ABI.

The planner is forced onto the tensor-core kernels (and each test checks that
they actually ran: mm_last_path() == MM_PATH_TENSOR).  Shapes span several
128 x 256 tiles with ragged edges in M, N and K; both operand majornesses
(transA / transB), batch broadcast on either operand, every C broadcast shape,
exact-integer QLinearMatMul at extreme values, and GroupedMatMul routing edge
cases (empty groups, one group, invalid indices).
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
HALF = [torch.bfloat16, torch.float16]


@contextlib.contextmanager
def tensor_path():
    qg.mm_set_path_policy(qg.MM_PATH_TENSOR)
    try:
        yield
    finally:
        qg.mm_set_path_policy(qg.MM_PATH_AUTO)


def ran_on_tensor_cores():
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert qg.mm_get_device_status() == "MM_OK"


@pytest.mark.parametrize("dtype", HALF, ids=str)
@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (296, 520, 328), (136, 264, 72), (64, 40, 1000), (520, 96, 8)])
def test_gemm_tensor(dtype, tA, tB, M, N, K):
    # Every dimension that is a stored row stride is a multiple of 8 (16 bytes),
    # as TMA requires; the ragged tiles come from M, N, K modulo 128/256/64.
    A = rand_tensor((K, M) if tA else (M, K), dtype, 1, DEV)
    B = rand_tensor((N, K) if tB else (K, N), dtype, 2, DEV)
    C = rand_tensor((1, N), dtype, 3, DEV)
    with tensor_path():
        Y = qg.mm_gemm(A, B, C, 0.5, 2.0, tA, tB)
    ran_on_tensor_cores()
    a, b, c = to_np(A), to_np(B), to_np(C)
    ref = oracle.gemm(a, b, c, alpha=0.5, beta=2.0, transA=tA, transB=tB)
    scale = oracle.gemm_abs_scale(a, b, c, alpha=0.5, beta=2.0, transA=tA, transB=tB)
    assert max_rel_err(to_np(Y), ref, scale) <= TOL[dtype]


@pytest.mark.parametrize("M,N,K", [(640, 264, 1024), (1024, 520, 1096), (1304, 264, 1024), (1128, 264, 1024),
                                   (1064, 520, 1024)])
@pytest.mark.parametrize("tA,tB", [(0, 1), (0, 0), (1, 0)])
def test_gemm_tensor_pairs_ragged(M, N, K, tA, tB):
    # K >= 1024: CTA pairs (256-row tiles); 640 and 1304 rows end in a partial
    # pair tile, K = 1096 in a partial k-block, N = 264 in a partial column tile.
    # With K-major A a last tile of at most 128 rows runs as one M = 128 MMA of
    # 64 rows per CTA: 640 (128 rows: both CTAs full), 1128 (104: the second
    # CTA holds 40), 1304 and 1064 (24 and 40: the second CTA holds none).
    # Every M is a multiple of 8: with transA it is A's stored row stride.
    A = rand_tensor((K, M) if tA else (M, K), torch.bfloat16, 90, DEV)
    B = rand_tensor((N, K) if tB else (K, N), torch.bfloat16, 91, DEV)
    C = rand_tensor((1, N), torch.bfloat16, 92, DEV)
    with tensor_path():
        Y = qg.mm_gemm(A, B, C, 0.75, 1.5, tA, tB)
    ran_on_tensor_cores()
    assert qg.mm_get_device_status() == "MM_OK"
    a, b, c = to_np(A), to_np(B), to_np(C)
    kw = dict(alpha=0.75, beta=1.5, transA=tA, transB=tB)
    assert max_rel_err(to_np(Y), oracle.gemm(a, b, c, **kw), oracle.gemm_abs_scale(a, b, c, **kw)) <= 1e-2


# More tiles than the persistent grid, with ragged edges.  Singles: 1104 x
# 4600 is 9 x 18 = 162 tiles on 152 CTAs (ragged M, N and K).  Pairs (K >=
# 1024): 1304 x 4104 is 6 x 17 = 102 pair tiles on 76 pairs, the last row
# tile 24 rows (an M = 128 tail tile when A is K-major), the last column tile
# 8 columns.  M and N are multiples of 8: stored row strides under transA /
# transB = 0.
@pytest.mark.parametrize("M,N,K", [(1104, 4600, 328), (1304, 4104, 1096)])
@pytest.mark.parametrize("tA,tB", [(0, 1), (0, 0), (1, 1)])
def test_gemm_tensor_many_tiles_ragged(M, N, K, tA, tB):
    A = rand_tensor((K, M) if tA else (M, K), torch.bfloat16, 93, DEV)
    B = rand_tensor((N, K) if tB else (K, N), torch.bfloat16, 94, DEV)
    C = rand_tensor((M, 1), torch.bfloat16, 95, DEV)
    with tensor_path():
        Y = qg.mm_gemm(A, B, C, 0.5, 2.0, tA, tB)
    ran_on_tensor_cores()
    a, b, c = to_np(A), to_np(B), to_np(C)
    kw = dict(alpha=0.5, beta=2.0, transA=tA, transB=tB)
    assert max_rel_err(to_np(Y), oracle.gemm(a, b, c, **kw), oracle.gemm_abs_scale(a, b, c, **kw)) <= 1e-2


def test_matmul_tensor_many_tiles_batched_f16():
    # A [9, 640, 328] @ B [1, 328, 1024]: 9 x 5 x 4 = 180 single-CTA tiles on
    # 152 CTAs, B broadcast over the batch.
    A = rand_tensor((9, 640, 328), torch.float16, 96, DEV)
    B = rand_tensor((1, 328, 1024), torch.float16, 97, DEV)
    with tensor_path():
        Y = qg.mm_matmul(A, B)
    ran_on_tensor_cores()
    a, b = to_np(A), to_np(B)
    assert max_rel_err(to_np(Y), oracle.matmul(a, b), oracle.matmul_abs_scale(a, b)) <= TOL[torch.float16]


# Single-CTA products with fewer tiles than SMs and a full C: 640 x 2560 is
# 5 x 10 = 50 tiles, 296 x 3000 is 3 x 12 = 36 tiles with a ragged last
# row and column tile.  K < 1024: single CTAs.
@pytest.mark.parametrize("dtype", HALF, ids=str)
@pytest.mark.parametrize("M,N,K", [(640, 2560, 512), (296, 3000, 328)])
@pytest.mark.parametrize("tA,tB", [(0, 1), (0, 0), (1, 0)])
def test_gemm_tensor_few_tiles(dtype, M, N, K, tA, tB):
    A = rand_tensor((K, M) if tA else (M, K), dtype, 98, DEV)
    B = rand_tensor((N, K) if tB else (K, N), dtype, 99, DEV)
    C = rand_tensor((M, N), dtype, 100, DEV)
    with tensor_path():
        Y = qg.mm_gemm(A, B, C, 0.5, -1.0, tA, tB)
    ran_on_tensor_cores()
    a, b, c = to_np(A), to_np(B), to_np(C)
    kw = dict(alpha=0.5, beta=-1.0, transA=tA, transB=tB)
    assert max_rel_err(to_np(Y), oracle.gemm(a, b, c, **kw), oracle.gemm_abs_scale(a, b, c, **kw)) <= TOL[dtype]


@pytest.mark.parametrize("M,N,K", [(129, 257, 72), (131, 9, 200)])
def test_gemm_tensor_odd_m_n(M, N, K):
    # transA = 0, transB = 1: the stored strides are K and K; M and N are odd,
    # so the output rows are not 16-byte aligned and take the scalar stores.
    A = rand_tensor((M, K), torch.bfloat16, 13, DEV)
    B = rand_tensor((N, K), torch.bfloat16, 14, DEV)
    with tensor_path():
        Y = qg.mm_gemm(A, B, None, 1.0, 1.0, 0, 1)
    ran_on_tensor_cores()
    a, b = to_np(A), to_np(B)
    ref = oracle.gemm(a, b, transB=1)
    assert max_rel_err(to_np(Y), ref, oracle.gemm_abs_scale(a, b, transB=1)) <= 1e-2


@pytest.mark.parametrize("c_shape", [None, (), (1,), (296,), (1, 296), (200, 1), (200, 296)])
def test_gemm_tensor_c_broadcast(c_shape):
    M, N, K = 200, 296, 136
    A = rand_tensor((M, K), torch.bfloat16, 4, DEV)
    B = rand_tensor((K, N), torch.bfloat16, 5, DEV)
    C = None if c_shape is None else rand_tensor(c_shape, torch.bfloat16, 6, DEV)
    with tensor_path():
        Y = qg.mm_gemm(A, B, C, -1.5, 0.25)
    ran_on_tensor_cores()
    c = None if C is None else to_np(C)
    ref = oracle.gemm(to_np(A), to_np(B), c, alpha=-1.5, beta=0.25)
    scale = oracle.gemm_abs_scale(to_np(A), to_np(B), c, alpha=-1.5, beta=0.25)
    assert max_rel_err(to_np(Y), ref, scale) <= 1e-2


@pytest.mark.parametrize("dtype", HALF, ids=str)
@pytest.mark.parametrize("sa,sb", [((3, 2, 130, 72), (1, 2, 72, 264)), ((1, 2, 130, 72), (3, 2, 72, 264)),
                                   ((4, 300, 128), (128, 264)), ((2, 64, 200), (2, 200, 512))])
def test_matmul_tensor_batched_broadcast(dtype, sa, sb):
    A = rand_tensor(sa, dtype, 7, DEV)
    B = rand_tensor(sb, dtype, 8, DEV)
    with tensor_path():
        Y = qg.mm_matmul(A, B)
    ran_on_tensor_cores()
    a, b = to_np(A), to_np(B)
    assert max_rel_err(to_np(Y), oracle.matmul(a, b), oracle.matmul_abs_scale(a, b)) <= TOL[dtype]


def test_matmul_tensor_transposed_views():
    # A given as the transpose of a contiguous [K, M] tensor (MN-major A).
    At = rand_tensor((2, 96, 160), torch.bfloat16, 9, DEV)
    A = At.transpose(1, 2)
    B = rand_tensor((96, 304), torch.bfloat16, 10, DEV)
    with tensor_path():
        Y = qg.mm_matmul(A, B)
    ran_on_tensor_cores()
    a, b = to_np(A), to_np(B)
    assert max_rel_err(to_np(Y), oracle.matmul(a, b), oracle.matmul_abs_scale(a, b)) <= 1e-2


def test_tensor_path_rejects_unaligned_layout():
    A = rand_tensor((100, 33), torch.bfloat16, 11, DEV)   # row stride 33 elements: not 16-byte aligned
    B = rand_tensor((33, 64), torch.bfloat16, 12, DEV)
    with tensor_path():
        with pytest.raises(qg.MMError) as e:
            qg.mm_matmul(A, B)
    assert e.value.name == "MM_ERR_UNSUPPORTED"
    Y = qg.mm_matmul(A, B)     # the planner falls back to the CUDA-core kernel
    assert qg.mm_last_path() == qg.MM_PATH_SIMT
    a, b = to_np(A), to_np(B)
    assert max_rel_err(to_np(Y), oracle.matmul(a, b), oracle.matmul_abs_scale(a, b)) <= 1e-2


# ------------------------------------------------------------------ QLinearMatMul

def _q(d):
    keys = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")
    with tensor_path():
        y = qg.mm_qlinear_matmul(*[d[k] for k in keys])
    ran_on_tensor_cores()
    ref = oracle.qlinear_matmul(*[d[k].cpu().numpy() for k in keys])
    got = y.cpu().numpy()
    assert got.dtype == ref.dtype and got.shape == ref.shape
    mism = np.argwhere(got != ref)
    assert mism.size == 0, "%d mismatches, first at %s: %s vs %s" % (
        len(mism), mism[0], got[tuple(mism[0])], ref[tuple(mism[0])])


def _qcase(M, K, N, ta, tb, ty, gran, sdt=torch.float32, batch_a=(), batch_b=(), seed=0):
    g = np.random.default_rng(seed)
    r = lambda t, shape, lo=None, hi=None: rand_tensor(shape, t, int(g.integers(1 << 30)), DEV, lo, hi)
    za_rng = (-20, 20) if ta == torch.int8 else (100, 140)
    zb_rng = (-20, 20) if tb == torch.int8 else (100, 140)
    if gran == "tensor":
        sas, sbs = (), ()
    elif gran == "vector":
        sas, sbs = (M,), (N,)
    else:
        sas, sbs = batch_a + (M, 1), batch_b + (1, N)
    return {
        "a": r(ta, batch_a + (M, K)), "b": r(tb, batch_b + (K, N)),
        "a_scale": torch.from_numpy(np.asarray(g.uniform(0.003, 0.01, sas), np.float32)).to(sdt).to(DEV),
        "a_zero_point": r(ta, sas, *za_rng),
        "b_scale": torch.from_numpy(np.asarray(g.uniform(0.003, 0.01, sbs), np.float32)).to(sdt).to(DEV),
        "b_zero_point": r(tb, sbs, *zb_rng),
        "y_scale": torch.tensor(0.005 * np.sqrt(K), dtype=sdt, device=DEV),
        "y_zero_point": torch.tensor(-9 if ty == torch.int8 else 120, dtype=ty, device=DEV),
    }


@pytest.mark.parametrize("ta,tb,ty", [(torch.int8, torch.int8, torch.int8), (torch.uint8, torch.uint8, torch.uint8),
                                      (torch.int8, torch.uint8, torch.uint8), (torch.uint8, torch.int8, torch.int8)],
                         ids=str)
@pytest.mark.parametrize("gran", ["tensor", "vector", "matrix"])
@pytest.mark.parametrize("M,K,N", [(300, 520, 264), (129, 1000, 257), (200, 64, 40)])
def test_qlinear_tensor(ta, tb, ty, gran, M, K, N):
    _q(_qcase(M, K, N, ta, tb, ty, gran))


@pytest.mark.parametrize("M,K,N,gran,batch", [(600, 1096, 264, "vector", ()), (1000, 2048, 520, "matrix", ()),
                                               (385, 1024, 136, "vector", ()), (300, 1024, 264, "matrix", (2,))])
def test_qlinear_tensor_long_k_ragged(M, K, N, gran, batch):
    # K >= 1024 (several exact 1024-deep segments) with ragged edges: 600,
    # 1000 and 385 rows end in partial 128-row tiles of 88, 104 and 1 valid
    # rows, K = 1096 in a partial k-block and a 72-deep last segment, N = 264
    # and 136 in partial column tiles; the last case has batch-indexed per-row
    # and per-column parameters.
    _q(_qcase(M, K, N, torch.int8, torch.uint8, torch.int8, gran, batch_a=batch, batch_b=batch, seed=M))


@pytest.mark.parametrize("layout", ["transposed", "odd_offset"])
def test_qlinear_tensor_strided_operands(layout):
    # The preparation kernel reads a and b through their strides: column-major
    # operands (no unit stride along a row) and rows that start one byte past
    # an aligned address (no vector load is aligned) take its byte-wise loads,
    # in both the row path (a) and the column-strip path (b).
    d = _qcase(300, 1100, 264, torch.int8, torch.uint8, torch.int8, "vector", seed=11)
    for key in ("a", "b"):
        x = d[key]
        if layout == "transposed":
            d[key] = x.t().contiguous().t()
        else:
            wide = torch.zeros((x.shape[0], x.shape[1] + 1), dtype=x.dtype, device=DEV)
            wide[:, 1:] = x
            d[key] = wide[:, 1:]
        assert not d[key].is_contiguous()
    _q(d)


def test_qlinear_tensor_f16_scales_and_batch():
    _q(_qcase(150, 300, 200, torch.int8, torch.int8, torch.int8, "matrix", torch.float16,
              batch_a=(2, 3), batch_b=(2, 3)))
    _q(_qcase(150, 300, 200, torch.uint8, torch.int8, torch.int8, "tensor", torch.float16,
              batch_a=(3,), batch_b=(1,)))


def _swamping_case(K, rows=256, cols=256):
    """Large operand values whose products rise to +-3.9e6 and then cancel.

    uint8 a with a_zero_point 128 and uint8 b with b_zero_point 0.  In every
    256-deep block of k: 120 terms of (+127)*255 = +32385, 16 terms of
    s_r * j (s_r in {-1, 0, 1} per row, j = 0..15), 120 terms of
    (-128)*253 = -32384.  Each block sums to 120 + 120 * s_r in {0, 120, 240},
    so with unit scales the uint8 output is the exact accumulator: a bit lost
    in any partial sum, however the kernel splits the zero points off, changes
    the result.
    """
    a = torch.empty((rows, K), dtype=torch.uint8)
    b = torch.empty((K, cols), dtype=torch.uint8)
    s_r = torch.tensor([(-1, 0, 1)[r % 3] for r in range(rows)], dtype=torch.int32)
    for k0 in range(0, K, 256):
        a[:, k0:k0 + 120] = 255
        a[:, k0 + 120:k0 + 136] = (128 + s_r).to(torch.uint8)[:, None]
        a[:, k0 + 136:k0 + 256] = 0
        b[k0:k0 + 120, :] = 255
        b[k0 + 120:k0 + 136, :] = torch.arange(16, dtype=torch.uint8)[:, None]
        b[k0 + 136:k0 + 256, :] = 253
    one = torch.tensor(1.0, device=DEV)
    return {
        "a": a.to(DEV), "a_scale": one, "a_zero_point": torch.tensor(128, dtype=torch.uint8, device=DEV),
        "b": b.to(DEV), "b_scale": one, "b_zero_point": torch.tensor(0, dtype=torch.uint8, device=DEV),
        "y_scale": one * (K // 256), "y_zero_point": torch.tensor(0, dtype=torch.uint8, device=DEV),
    }


@pytest.mark.parametrize("K", [256, 1024])
def test_qlinear_tensor_accumulation_is_exact(K):
    d = _swamping_case(K)
    _q(d)
    keys = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")
    with tensor_path():
        y = qg.mm_qlinear_matmul(*[d[k] for k in keys]).cpu()
    want = torch.tensor([(0, 120, 240)[r % 3] for r in range(256)], dtype=torch.uint8)[:, None].expand(256, 256)
    assert torch.equal(y, want)


def _extreme_case(K, types, rows=256, cols=256, seed=0):
    """Operands at the bottom of the 8-bit range, cancelled by the zero points.

    a = za + u and b = zb + v with u, v in {0, 1}: int8 operands with zero point
    -128, or uint8 operands with zero point 0.  The true accumulator is
    sum_k u*v (about 100, at most 255), written exactly to a uint8 output with
    unit scales.  Moved into [-128, 127] (int8 as is, uint8 minus 128) both
    operands are u - 128 and v - 128, so products are 16384 - 128(u + v) + u*v
    and any 1024 of them sum to nearly 2^24: every bit of every partial sum
    the kernel forms reaches the output.
    """
    g = np.random.default_rng(seed)
    pv = 200.0 / K
    u = (g.random((rows, K)) < 0.5).astype(np.int16)
    v = (g.random((K, cols)) < pv).astype(np.int16)
    want = (u.astype(np.int64) @ v.astype(np.int64))
    assert want.max() <= 255

    def operand(x, t):
        zp = -128 if t == torch.int8 else 0
        np_t = np.int8 if t == torch.int8 else np.uint8
        return torch.from_numpy((x + zp).astype(np_t)).to(DEV), torch.tensor(zp, dtype=t, device=DEV)

    a, za = operand(u, types[0])
    b, zb = operand(v, types[1])
    one = torch.tensor(1.0, device=DEV)
    d = {"a": a, "a_scale": one, "a_zero_point": za, "b": b, "b_scale": one, "b_zero_point": zb,
         "y_scale": one, "y_zero_point": torch.tensor(0, dtype=torch.uint8, device=DEV)}
    return d, torch.from_numpy(want.astype(np.uint8))


@pytest.mark.parametrize("types", [(torch.int8, torch.int8), (torch.uint8, torch.uint8),
                                   (torch.int8, torch.uint8)], ids=["s8s8", "u8u8", "s8u8"])
@pytest.mark.parametrize("K", [1024, 2048, 4160])
def test_qlinear_tensor_exact_at_full_range(types, K):
    d, want = _extreme_case(K, types)
    keys = ("a", "a_scale", "a_zero_point", "b", "b_scale", "b_zero_point", "y_scale", "y_zero_point")
    with tensor_path():
        y = qg.mm_qlinear_matmul(*[d[k] for k in keys]).cpu()
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    assert torch.equal(y, want)
    _q(d)


@pytest.mark.parametrize("ys", [2.0, float(np.nextafter(np.float32(2), np.float32(3))),
                                float(np.nextafter(np.float32(2), np.float32(1))), 3.0, 0.25, 0.0625],
                         ids=["tie", "above_tie", "below_tie", "third", "quarter", "sixteenth"])
def test_qlinear_tensor_rounding_near_half_integers(ys):
    """Quotients on, or one ulp beside, half-integers: the requantisation must
    round exactly as the correctly rounded division followed by rint does."""
    g = np.random.default_rng(7)
    a = torch.from_numpy(g.integers(-1, 2, (256, 256)).astype(np.int8)).to(DEV)
    b = torch.from_numpy(g.integers(-1, 2, (256, 256)).astype(np.int8)).to(DEV)
    z8 = torch.tensor(0, dtype=torch.int8, device=DEV)
    d = {"a": a, "a_scale": torch.tensor(0.5, device=DEV), "a_zero_point": z8,
         "b": b, "b_scale": torch.tensor(0.25, device=DEV), "b_zero_point": z8,
         "y_scale": torch.tensor(ys * 0.125, dtype=torch.float32, device=DEV), "y_zero_point": z8}
    _q(d)


def test_f16_mma_keeps_integer_sums_exact():
    # The same premise on the f16 Gemm path: integer products of magnitude
    # 65025 accumulated to +-8.3e6 and cancelled; the f16 output holds the
    # small exact remainder (|y| <= 2048 is exact in f16).
    K, M, N = 256, 128, 256
    A = torch.zeros((M, K), dtype=torch.float16)
    B = torch.zeros((K, N), dtype=torch.float16)
    A[:, :127] = 255.0
    A[:, 127:129] = torch.arange(M, dtype=torch.float16)[:, None] % 7 - 3
    A[:, 129:] = -255.0
    B[:, :] = 255.0
    B[127:129, :] = (torch.arange(N) % 5).to(torch.float16)[None, :]
    Ad, Bd = A.to(DEV), B.to(DEV)
    with tensor_path():
        Y = qg.mm_matmul(Ad, Bd)
    ran_on_tensor_cores()
    ref = oracle.matmul(A.double().numpy(), B.double().numpy())
    assert np.array_equal(Y.double().cpu().numpy(), ref)


# ------------------------------------------------------------------ GroupedMatMul

def _grouped(x, w, gi, bias):
    with tensor_path():
        out = qg.mm_grouped_matmul(x, w, gi, bias)
    assert qg.mm_last_path() == qg.MM_PATH_TENSOR
    xa, wa = to_np(x), to_np(w)
    ba = None if bias is None else to_np(bias)
    gia = gi.cpu().numpy()
    G = w.shape[0]
    bad = (gia < 0) | (gia >= G)
    gclip = np.where(bad, 0, gia)
    ref = oracle.grouped_matmul(xa, wa, gclip, ba)
    scale = oracle.grouped_abs_scale(xa, wa, gclip, ba)
    err = np.abs(to_np(out) - ref) / (scale + 1e-30)
    assert np.max(err[~bad], initial=0) <= TOL[x.dtype]
    assert np.all(to_np(out)[bad] == 0)
    return bad.any()


@pytest.mark.parametrize("dtype", HALF, ids=str)
@pytest.mark.parametrize("ind", [torch.int32, torch.int64], ids=str)
@pytest.mark.parametrize("with_bias", [False, True])
def test_grouped_tensor(dtype, ind, with_bias):
    M, K, N, G, S = 300, 200, 520, 6, 2
    x = rand_tensor((M, K), dtype, 21, DEV)
    w = rand_tensor((G, K, N), dtype, 22, DEV)
    p = np.array([0.5, 0.2, 0.0, 0.2, 0.05, 0.05])       # group 2 unused
    gi = torch.from_numpy(np.random.default_rng(23).choice(G, size=(M, S), p=p)).to(ind).to(DEV)
    bias = rand_tensor((G, N), dtype, 24, DEV) if with_bias else None
    _grouped(x, w, gi, bias)
    assert qg.mm_get_device_status() == "MM_OK"


@pytest.mark.parametrize("dtype", HALF, ids=str)
@pytest.mark.parametrize("with_bias", [False, True])
def test_grouped_tensor_cta_pairs(dtype, with_bias):
    # K >= 1024 and groups of 1100 rows on average: the planner runs 256-row
    # CTA-pair tiles.  Group sizes are not multiples of 256 (one is below 128,
    # one is empty), K = 1096 leaves a partial k-block, N = 520 a partial
    # column tile.
    M, K, N, G, S = 2200, 1096, 520, 4, 2
    x = rand_tensor((M, K), dtype, 31, DEV)
    w = rand_tensor((G, K, N), dtype, 32, DEV)
    p = np.array([0.63, 0.345, 0.0, 0.025])
    gi = torch.from_numpy(np.random.default_rng(33).choice(G, size=(M, S), p=p)).to(torch.int32).to(DEV)
    bias = rand_tensor((G, N), dtype, 34, DEV) if with_bias else None
    _grouped(x, w, gi, bias)
    assert qg.mm_get_device_status() == "MM_OK"


# Group sizes whose last 256-row pair tile holds every kind of remainder: none
# (256, 512), at most 64 rows (1, 63, 64, 257, 320: the second CTA of the tail
# tile holds none), 65-128 rows (65, 127, 128, 384, 600: the tail tile splits
# 64 + the rest), and 129-255 rows (129, 200, 255, 385, 1500: a full-height
# pair tile), plus an empty group.
_TAIL_SIZES = [1, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 320, 384, 385, 512, 600, 1500, 0]


@pytest.mark.parametrize("dtype", HALF, ids=str)
@pytest.mark.parametrize("with_bias", [False, True])
def test_grouped_tensor_cta_pair_tail_tiles(dtype, with_bias):
    # 5246 routed rows over 18 groups (291 a group on average) and K >= 1024:
    # CTA pairs, each group's last tile of at most 128 rows as one M = 128 MMA.
    G, S, K, N = len(_TAIL_SIZES), 2, 1024, 520
    ids = np.repeat(np.arange(G), _TAIL_SIZES)
    np.random.default_rng(38).shuffle(ids)
    M = ids.size // S
    gi = torch.from_numpy(ids.reshape(M, S)).to(torch.int32).to(DEV)
    x = rand_tensor((M, K), dtype, 39, DEV)
    w = rand_tensor((G, K, N), dtype, 40, DEV)
    bias = rand_tensor((G, N), dtype, 41, DEV) if with_bias else None
    _grouped(x, w, gi, bias)
    assert qg.mm_get_device_status() == "MM_OK"


@pytest.mark.parametrize("pairs", [False, True])
def test_grouped_tensor_padded_and_transposed_input(pairs):
    # The same product with the input in two layouts, both copied into group
    # order by the routing: rows 16-byte aligned with a padded row stride
    # (16-byte vector copies) and stored transposed (column stride M:
    # element-wise copies).  K = 1024 with 300 routed rows a group on average
    # takes CTA pairs (tail tiles included), K = 512 single CTAs.
    M, S, G, N = 900, 2, 6, 520
    K = 1024 if pairs else 512
    g = np.random.default_rng(42)
    gi = torch.from_numpy(g.choice(G, size=(M, S), p=[0.4, 0.25, 0.15, 0.1, 0.07, 0.03]).astype(np.int32)).to(DEV)
    x_pad = rand_tensor((M, K + 64), torch.bfloat16, 43, DEV)
    x_rows = x_pad[:, :K]                                   # row stride K + 64, unit column stride
    x_cols = x_rows.t().contiguous().t()                    # the same values, column stride M
    w = rand_tensor((G, K, N), torch.bfloat16, 44, DEV)
    bias = rand_tensor((G, N), torch.bfloat16, 45, DEV)
    for x in (x_rows, x_cols):
        _grouped(x, w, gi, bias)
        assert qg.mm_get_device_status() == "MM_OK"


def test_grouped_tensor_cta_pairs_invalid_indices():
    M, K, N, G = 2200, 1024, 256, 2
    x = rand_tensor((M, K), torch.bfloat16, 35, DEV)
    w = rand_tensor((G, K, N), torch.bfloat16, 36, DEV)
    gi = torch.from_numpy(np.random.default_rng(37).integers(-1, G + 1, size=(M, 2))).to(torch.int64).to(DEV)
    assert _grouped(x, w, gi, None)
    assert qg.mm_get_device_status() == "MM_ERR_INDEX_RANGE"


def test_grouped_tensor_single_group_and_k_tail():
    x = rand_tensor((260, 72), torch.bfloat16, 25, DEV)
    w = rand_tensor((1, 72, 264), torch.bfloat16, 26, DEV)
    gi = torch.zeros((260, 1), dtype=torch.int64, device=DEV)
    _grouped(x, w, gi, rand_tensor((1, 264), torch.bfloat16, 27, DEV))
    assert qg.mm_get_device_status() == "MM_OK"


def test_grouped_tensor_invalid_indices():
    M, K, N, G = 140, 64, 256, 4
    x = rand_tensor((M, K), torch.bfloat16, 28, DEV)
    w = rand_tensor((G, K, N), torch.bfloat16, 29, DEV)
    gi = torch.from_numpy(np.random.default_rng(30).integers(-2, G + 2, size=(M, 2))).to(torch.int32).to(DEV)
    assert _grouped(x, w, gi, None)
    assert qg.mm_get_device_status() == "MM_ERR_INDEX_RANGE"
    assert qg.mm_get_device_status() == "MM_OK"


# The few-row tensor-core configuration (at most 64 rows of A', fewer
# 256-column tiles than SMs): each tile's k-blocks are split over a cluster of
# up to 8 CTAs and the partial sums added through distributed shared memory.
# Splits of 1, 2, 4 and 8 (K of 64, 128, 1000 and 8192; N from one ragged tile
# to 32 tiles), both layouts of B', C absent, a row vector or full, and a
# batched MatMul whose B is broadcast.
@pytest.mark.parametrize("M,N,K", [(5, 200, 64), (16, 1000, 128), (33, 8192, 1000), (64, 520, 8192),
                                   (17, 8200, 4104)])
@pytest.mark.parametrize("tB", [0, 1])
@pytest.mark.parametrize("c_kind", [None, "row", "full"])
def test_gemm_tensor_few_rows_split_k(M, N, K, tB, c_kind):
    A = rand_tensor((M, K), torch.bfloat16, 131, DEV)
    B = rand_tensor((N, K) if tB else (K, N), torch.bfloat16, 132, DEV)
    C = None if c_kind is None else rand_tensor((1, N) if c_kind == "row" else (M, N), torch.bfloat16, 133, DEV)
    with tensor_path():
        Y = qg.mm_gemm(A, B, C, 0.75, 1.5, 0, tB)
    ran_on_tensor_cores()
    a, b = to_np(A), to_np(B)
    c = None if C is None else to_np(C)
    kw = dict(alpha=0.75, beta=1.5, transB=tB)
    assert max_rel_err(to_np(Y), oracle.gemm(a, b, c, **kw), oracle.gemm_abs_scale(a, b, c, **kw)) <= TOL[torch.bfloat16]


def test_matmul_tensor_few_rows_batched_f16():
    A = rand_tensor((2, 3, 24, 640), torch.float16, 134, DEV)
    B = rand_tensor((640, 1304), torch.float16, 135, DEV)   # row pitch a multiple of 16 bytes
    with tensor_path():
        Y = qg.mm_matmul(A, B)
    ran_on_tensor_cores()
    a, b = to_np(A), to_np(B)
    assert max_rel_err(to_np(Y), oracle.matmul(a, b), oracle.matmul_abs_scale(a, b)) <= TOL[torch.float16]
