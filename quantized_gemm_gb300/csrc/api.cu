// C-ABI entry points (include/mm.h): argument validation, shape inference,
// operand views, path planning and kernel dispatch.  All shape logic here is
// host code; every arithmetic step of an operator runs in a CUDA kernel.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "tc.h"

using namespace qg;

namespace {

std::atomic<int> g_policy{MM_PATH_AUTO};
thread_local int g_last_path = MM_PATH_NONE;

// Device-side status word (one instance per device); kernels receive its
// address as a parameter, so no relocatable device code is needed.
__device__ unsigned g_device_status;

unsigned* device_status_ptr() {
  static std::mutex mu;
  static unsigned* ptrs[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}

int elem_size(int dt) {
  switch (dt) {
    case MM_BF16: case MM_F16: return 2;
    case MM_F32: case MM_I32: case MM_U32: return 4;
    case MM_F64: case MM_I64: case MM_U64: return 8;
    case MM_I8: case MM_U8: return 1;
    default: return 0;
  }
}

bool is_int_type(int dt) { return dt == MM_I32 || dt == MM_I64 || dt == MM_U32 || dt == MM_U64; }
bool is_matmul_type(int dt) { return dt >= MM_BF16 && dt <= MM_U64; }   // MatMul-13 / Gemm-13 T
bool is_q8(int dt) { return dt == MM_I8 || dt == MM_U8; }
bool is_q4(int dt) { return dt == MM_I4 || dt == MM_U4; }

int64_t numel(const mm_tensor* t) {
  int64_t n = 1;
  for (int d = 0; d < t->ndim; ++d) n *= t->shape[d];
  return n;
}

mm_status check_tensor(const mm_tensor* t) {
  if (!t) return MM_ERR_INVALID_ARG;
  if (t->ndim < 0 || t->ndim > MM_MAX_DIMS) return MM_ERR_INVALID_ARG;
  if (elem_size(t->dtype) == 0 && !is_q4(t->dtype)) return MM_ERR_DTYPE;
  for (int d = 0; d < t->ndim; ++d)
    if (t->shape[d] < 0 || t->strides[d] < 0) return MM_ERR_INVALID_ARG;
  if (!t->data && numel(t) != 0) return MM_ERR_INVALID_ARG;
  return MM_OK;
}

// Dense row-major (strides of size-1 dimensions are not constrained; an empty
// tensor has no elements to place and is always accepted).
bool is_dense(const mm_tensor* t) {
  if (numel(t) == 0) return true;
  int64_t expect = 1;
  for (int d = t->ndim - 1; d >= 0; --d) {
    if (t->shape[d] != 1 && t->strides[d] != expect) return false;
    expect *= t->shape[d];
  }
  return true;
}

mm_status check_output(const mm_tensor* y, int dtype, int ndim, const int64_t* shape) {
  mm_status s = check_tensor(y);
  if (s != MM_OK) return s;
  if (y->dtype != dtype) return MM_ERR_DTYPE;
  if (y->ndim != ndim) return MM_ERR_SHAPE;
  for (int d = 0; d < ndim; ++d)
    if (y->shape[d] != shape[d]) return MM_ERR_SHAPE;
  if (!is_dense(y)) return MM_ERR_SHAPE;
  return MM_OK;
}

// numpy.matmul shape inference (MatMul page summary and Examples): 1-D
// promotion, right-aligned batch broadcast.  Produces the broadcast batch map
// and the matrix views of both operands.
struct MatmulPlan {
  int64_t M, N, K;
  BatchMap bm;
  MatView a, b;
  int64_t a_bshape[kMaxBatchDims], b_bshape[kMaxBatchDims];   // each operand's own size per batch dim
  int out_ndim;
  int64_t out_shape[MM_MAX_DIMS];
};

mm_status plan_matmul(const mm_tensor* A, const mm_tensor* B, MatmulPlan* p) {
  if (A->ndim < 1 || B->ndim < 1) return MM_ERR_SHAPE;
  int64_t as[MM_MAX_DIMS + 1], ast[MM_MAX_DIMS + 1], bs[MM_MAX_DIMS + 1], bst[MM_MAX_DIMS + 1];
  int an = A->ndim, bn = B->ndim;
  if (an == 1) { as[0] = 1; ast[0] = 0; as[1] = A->shape[0]; ast[1] = A->strides[0]; an = 2; }
  else { for (int d = 0; d < an; ++d) { as[d] = A->shape[d]; ast[d] = A->strides[d]; } }
  if (bn == 1) { bs[0] = B->shape[0]; bst[0] = B->strides[0]; bs[1] = 1; bst[1] = 0; bn = 2; }
  else { for (int d = 0; d < bn; ++d) { bs[d] = B->shape[d]; bst[d] = B->strides[d]; } }
  if (as[an - 1] != bs[bn - 2]) return MM_ERR_SHAPE;
  p->M = as[an - 2];
  p->K = as[an - 1];
  p->N = bs[bn - 1];
  const int nba = an - 2, nbb = bn - 2;
  const int nb = nba > nbb ? nba : nbb;
  if (nb > kMaxBatchDims) return MM_ERR_SHAPE;
  p->bm.nb = nb;
  p->bm.count = 1;
  for (int d = 0; d < nb; ++d) {
    const int da = d - (nb - nba), db = d - (nb - nbb);
    const int64_t sa = da >= 0 ? as[da] : 1, sb = db >= 0 ? bs[db] : 1;
    int64_t so;
    if (sa == sb || sb == 1) so = sa;
    else if (sa == 1) so = sb;
    else return MM_ERR_SHAPE;
    p->bm.shape[d] = so;
    p->bm.count *= so;
    p->a_bshape[d] = sa;
    p->b_bshape[d] = sb;
    p->a.bstride[d] = (sa == 1) ? 0 : ast[da];
    p->b.bstride[d] = (sb == 1) ? 0 : bst[db];
  }
  for (int d = nb; d < kMaxBatchDims; ++d) {
    p->bm.shape[d] = 1; p->a.bstride[d] = 0; p->b.bstride[d] = 0; p->a_bshape[d] = 1; p->b_bshape[d] = 1;
  }
  p->a.ptr = A->data; p->a.rs = ast[an - 2]; p->a.cs = ast[an - 1];
  p->b.ptr = B->data; p->b.rs = bst[bn - 2]; p->b.cs = bst[bn - 1];
  int k = 0;
  for (int d = 0; d < nb; ++d) p->out_shape[k++] = p->bm.shape[d];
  if (A->ndim >= 2) p->out_shape[k++] = p->M;
  if (B->ndim >= 2) p->out_shape[k++] = p->N;
  p->out_ndim = k;
  return MM_OK;
}

// View of the dense output of a matmul-shaped operator.
MatView output_view(const mm_tensor* Y, const MatmulPlan& p, int a_is_1d, int b_is_1d) {
  MatView v;
  v.ptr = Y->data;
  for (int d = 0; d < kMaxBatchDims; ++d) v.bstride[d] = d < p.bm.nb ? Y->strides[d] : 0;
  v.rs = a_is_1d ? 0 : Y->strides[p.bm.nb];
  v.cs = b_is_1d ? 0 : Y->strides[Y->ndim - 1];
  return v;
}

// Chosen path for a call, honouring the process-wide policy.
int choose(bool tensor_ok, bool tensor_pays) {
  const int pol = g_policy.load();
  if (pol == MM_PATH_SIMT) return MM_PATH_SIMT;
  if (pol == MM_PATH_TENSOR) return tensor_ok ? MM_PATH_TENSOR : -1;
  return (tensor_ok && tensor_pays) ? MM_PATH_TENSOR : MM_PATH_SIMT;
}

// Work large enough that the tensor-core kernels pay for their set-up.
bool tensor_pays(int64_t M, int64_t N, int64_t K, int64_t batch) {
  return (double)M * (double)N * (double)K * (double)batch >= 2097152.0;
}
// fp32 runs as three tf32 products on the tensor cores: it needs 8x more work
// than the 16-bit types (2^24 multiply-adds instead of 2^21) before it beats
// the CUDA-core kernel.
bool tensor_pays_dense(int dtype, int64_t M, int64_t N, int64_t K, int64_t batch) {
  if (dtype == MM_F32) return (double)M * (double)N * (double)K * (double)batch >= 8.0 * 2097152.0;
  return tensor_pays(M, N, K, batch);
}

mm_status finish(mm_status s, int path) {
  if (s == MM_OK) g_last_path = path;
  return s;
}

// MatMul and Gemm after validation: the few-row kernel where it applies (policy
// MM_PATH_AUTO, or forced by MM_PATH_VECTOR), else the tensor-core or the
// CUDA-core tiles.
// The few-row kernels pay when they stream at least 2^17 elements of B'
// (their k split and cross-CTA reduction cost a few microseconds); smaller
// products take one pass of the CUDA-core tiles.
bool few_row_pays(const GemmArgs& g) { return (double)g.N * (double)g.K * (double)g.bm.count >= 131072.0; }

mm_status run_dense(const GemmArgs& g, bool pays, cudaStream_t st) {
  const int pol = g_policy.load();
  if (pol == MM_PATH_VECTOR || (pol == MM_PATH_AUTO && vec_gemm_preferred(g) && few_row_pays(g))) {
    if (!vec_gemm_supported(g)) return MM_ERR_UNSUPPORTED;
    return finish(launch_vec_gemm(g, st), MM_PATH_VECTOR);
  }
  const int path = choose(tc_gemm_supported(g), pays);
  if (path < 0) return MM_ERR_UNSUPPORTED;
  if (path == MM_PATH_TENSOR) return finish(launch_tc_gemm(g, device_status_ptr(), st), MM_PATH_TENSOR);
  return finish(launch_simt_gemm(g, st), MM_PATH_SIMT);
}

}  // namespace

extern "C" {

const char* mm_status_string(mm_status s) {
  switch (s) {
    case MM_OK: return "MM_OK";
    case MM_ERR_INVALID_ARG: return "MM_ERR_INVALID_ARG: invalid argument";
    case MM_ERR_SHAPE: return "MM_ERR_SHAPE: shapes violate the operator's rules or the output shape/layout is wrong";
    case MM_ERR_DTYPE: return "MM_ERR_DTYPE: element type outside the operator's type constraints";
    case MM_ERR_UNSUPPORTED: return "MM_ERR_UNSUPPORTED: case not defined by the operator pages or not runnable on the forced path";
    case MM_ERR_WORKSPACE: return "MM_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case MM_ERR_CUDA: return "MM_ERR_CUDA: a CUDA call or kernel launch failed";
    case MM_ERR_TIMEOUT: return "MM_ERR_TIMEOUT: a device pipeline wait exceeded its limit";
    case MM_ERR_INDEX_RANGE: return "MM_ERR_INDEX_RANGE: a group index outside [0, G) was seen";
  }
  return "unknown mm_status";
}

const char* mm_version(void) { return "0.1.0"; }

mm_status mm_set_path_policy(int32_t policy) {
  if (policy != MM_PATH_AUTO && policy != MM_PATH_SIMT && policy != MM_PATH_TENSOR && policy != MM_PATH_VECTOR)
    return MM_ERR_INVALID_ARG;
  g_policy.store(policy);
  return MM_OK;
}

int32_t mm_last_path(void) { return g_last_path; }

mm_status mm_set_wait_limit_ns(uint64_t ns) {
  tc_set_wait_limit_ns((unsigned long long)ns);
  return MM_OK;
}

// ------------------------------------------------------------------ MatMul

mm_status mm_matmul_output_shape(const mm_tensor* A, const mm_tensor* B, int32_t* out_ndim, int64_t* out_shape) {
  if (!out_ndim || !out_shape) return MM_ERR_INVALID_ARG;
  mm_status s;
  if ((s = check_tensor(A)) != MM_OK || (s = check_tensor(B)) != MM_OK) return s;
  MatmulPlan p;
  if ((s = plan_matmul(A, B, &p)) != MM_OK) return s;
  *out_ndim = p.out_ndim;
  for (int d = 0; d < p.out_ndim; ++d) out_shape[d] = p.out_shape[d];
  return MM_OK;
}

mm_status mm_matmul(const mm_tensor* A, const mm_tensor* B, const mm_tensor* Y, void* stream) {
  mm_status s;
  if ((s = check_tensor(A)) != MM_OK || (s = check_tensor(B)) != MM_OK) return s;
  if (!is_matmul_type(A->dtype) || B->dtype != A->dtype) return MM_ERR_DTYPE;
  MatmulPlan p;
  if ((s = plan_matmul(A, B, &p)) != MM_OK) return s;
  if ((s = check_output(Y, A->dtype, p.out_ndim, p.out_shape)) != MM_OK) return s;
  if (p.M == 0 || p.N == 0 || p.bm.count == 0) return finish(MM_OK, MM_PATH_NONE);
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.dtype = A->dtype; g.M = p.M; g.N = p.N; g.K = p.K; g.bm = p.bm; g.a = p.a; g.b = p.b;
  g.c.ptr = nullptr;
  g.y = output_view(Y, p, A->ndim == 1, B->ndim == 1);
  g.alpha = 1.f; g.beta = 0.f; g.alpha_d = 1.0; g.beta_d = 0.0; g.alpha_i = 1; g.beta_i = 0;
  return run_dense(g, tensor_pays_dense(g.dtype, p.M, p.N, p.K, p.bm.count), static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ Gemm

mm_status mm_gemm_output_shape(const mm_tensor* A, const mm_tensor* B, int64_t transA, int64_t transB,
                               int32_t* out_ndim, int64_t* out_shape) {
  if (!out_ndim || !out_shape) return MM_ERR_INVALID_ARG;
  mm_status s;
  if ((s = check_tensor(A)) != MM_OK || (s = check_tensor(B)) != MM_OK) return s;
  if (A->ndim != 2 || B->ndim != 2) return MM_ERR_SHAPE;
  const int64_t M = transA ? A->shape[1] : A->shape[0], K = transA ? A->shape[0] : A->shape[1];
  const int64_t K2 = transB ? B->shape[1] : B->shape[0], N = transB ? B->shape[0] : B->shape[1];
  if (K != K2) return MM_ERR_SHAPE;
  *out_ndim = 2;
  out_shape[0] = M;
  out_shape[1] = N;
  return MM_OK;
}

mm_status mm_gemm(const mm_tensor* A, const mm_tensor* B, const mm_tensor* C, float alpha, float beta,
                  int64_t transA, int64_t transB, const mm_tensor* Y, void* stream) {
  mm_status s;
  int32_t nd;
  int64_t shp[MM_MAX_DIMS];
  if ((s = mm_gemm_output_shape(A, B, transA, transB, &nd, shp)) != MM_OK) return s;
  if (!is_matmul_type(A->dtype) || B->dtype != A->dtype) return MM_ERR_DTYPE;
  if (C && (s = check_tensor(C)) != MM_OK) return s;
  if (C && C->dtype != A->dtype) return MM_ERR_DTYPE;
  if ((s = check_output(Y, A->dtype, 2, shp)) != MM_OK) return s;
  const int64_t M = shp[0], N = shp[1];
  const int64_t K = transA ? A->shape[0] : A->shape[1];
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.dtype = A->dtype; g.M = M; g.N = N; g.K = K;
  g.bm.nb = 0; g.bm.count = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) g.bm.shape[d] = 1;
  g.a.ptr = A->data; g.a.rs = transA ? A->strides[1] : A->strides[0]; g.a.cs = transA ? A->strides[0] : A->strides[1];
  g.b.ptr = B->data; g.b.rs = transB ? B->strides[1] : B->strides[0]; g.b.cs = transB ? B->strides[0] : B->strides[1];
  g.y.ptr = Y->data; g.y.rs = Y->strides[0]; g.y.cs = Y->strides[1];
  g.c.ptr = nullptr;
  if (C) {
    // Unidirectional broadcast of C to (M, N): rank <= 2, right-aligned, each
    // dimension equal to the target or 1 (Gemm page, Inputs: C).
    if (C->ndim > 2) return MM_ERR_SHAPE;
    const int64_t tgt[2] = {M, N};
    int64_t st[2] = {0, 0};
    for (int d = 0; d < C->ndim; ++d) {
      const int td = 2 - C->ndim + d;
      if (C->shape[d] != tgt[td] && C->shape[d] != 1) return MM_ERR_SHAPE;
      st[td] = C->shape[d] == 1 ? 0 : C->strides[d];
    }
    g.c.ptr = C->data; g.c.rs = st[0]; g.c.cs = st[1];
  }
  if (is_int_type(A->dtype)) {
    if (!std::isfinite(alpha) || !std::isfinite(beta)) return MM_ERR_UNSUPPORTED;
    if (alpha == std::floor(alpha) && beta == std::floor(beta) && std::fabs(alpha) < 9.2e18f &&
        std::fabs(beta) < 9.2e18f) {
      g.alpha_i = (uint64_t)(int64_t)alpha;     // exact modulo 2^n
      g.beta_i = (uint64_t)(int64_t)beta;
    } else {
      g.int_float = 1;                          // fp64 evaluation, truncated toward zero
    }
  }
  g.alpha = alpha; g.beta = beta; g.alpha_d = (double)alpha; g.beta_d = (double)beta;
  if (M == 0 || N == 0) return finish(MM_OK, MM_PATH_NONE);
  return run_dense(g, tensor_pays_dense(g.dtype, M, N, K, 1), static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ QLinearMatMul

namespace {

// Per-row (of a) or per-column (of b) quantisation parameter view
// (QLinearMatMul - version 10, summary: scale and zero point shapes).
mm_status param_view(const mm_tensor* prm, const mm_tensor* x, const MatmulPlan& p, bool per_row, VecView* v) {
  memset(v, 0, sizeof(*v));
  v->ptr = prm->data;
  if (numel(prm) == 1) return MM_OK;   // per tensor: every stride 0
  const int nd = x->ndim;
  if (nd < 2) return MM_ERR_SHAPE;
  const int64_t len = per_row ? x->shape[nd - 2] : x->shape[nd - 1];
  if (prm->ndim == 1 && nd == 2) {
    if (prm->shape[0] != len) return MM_ERR_SHAPE;
    v->vs = prm->strides[0];
    return MM_OK;
  }
  if (prm->ndim != nd) return MM_ERR_SHAPE;
  for (int d = 0; d < nd - 2; ++d)
    if (prm->shape[d] != x->shape[d]) return MM_ERR_SHAPE;
  if (per_row) {
    if (prm->shape[nd - 2] != len || prm->shape[nd - 1] != 1) return MM_ERR_SHAPE;
    v->vs = prm->strides[nd - 2];
  } else {
    if (prm->shape[nd - 2] != 1 || prm->shape[nd - 1] != len) return MM_ERR_SHAPE;
    v->vs = prm->strides[nd - 1];
  }
  // The parameter's batch dimensions are the operand's; right-align them into
  // the broadcast batch, with stride 0 where the operand is broadcast.
  const int nbx = nd - 2;
  for (int d = 0; d < p.bm.nb; ++d) {
    const int dx = d - (p.bm.nb - nbx);
    v->bstride[d] = (dx >= 0 && x->shape[dx] != 1) ? prm->strides[dx] : 0;
  }
  return MM_OK;
}

struct QPlan {
  MatmulPlan mp;
  QLinearArgs q;
};

mm_status plan_qlinear(const mm_tensor* a, const mm_tensor* a_scale, const mm_tensor* a_zp, const mm_tensor* b,
                       const mm_tensor* b_scale, const mm_tensor* b_zp, const mm_tensor* y_scale,
                       const mm_tensor* y_zp, QPlan* qp) {
  const mm_tensor* all[8] = {a, a_scale, a_zp, b, b_scale, b_zp, y_scale, y_zp};
  mm_status s;
  for (const mm_tensor* t : all)
    if ((s = check_tensor(t)) != MM_OK) return s;
  if (!is_q8(a->dtype) || a_zp->dtype != a->dtype) return MM_ERR_DTYPE;
  if (!is_q8(b->dtype) || b_zp->dtype != b->dtype) return MM_ERR_DTYPE;
  if (!is_q8(y_zp->dtype)) return MM_ERR_DTYPE;
  for (const mm_tensor* sc : {a_scale, b_scale, y_scale})
    if (sc->dtype != MM_F32 && sc->dtype != MM_F16) return MM_ERR_DTYPE;
  auto same_shape = [](const mm_tensor* u, const mm_tensor* v) {
    if (u->ndim != v->ndim) return false;
    for (int d = 0; d < u->ndim; ++d)
      if (u->shape[d] != v->shape[d]) return false;
    return true;
  };
  if (!same_shape(a_scale, a_zp) || !same_shape(b_scale, b_zp)) return MM_ERR_SHAPE;
  if (numel(y_scale) != 1 || numel(y_zp) != 1) return MM_ERR_SHAPE;
  if ((s = plan_matmul(a, b, &qp->mp)) != MM_OK) return s;
  QLinearArgs& q = qp->q;
  memset(&q, 0, sizeof(q));
  q.M = qp->mp.M; q.N = qp->mp.N; q.K = qp->mp.K; q.bm = qp->mp.bm; q.a = qp->mp.a; q.b = qp->mp.b;
  for (int d = 0; d < kMaxBatchDims; ++d) { q.a_bshape[d] = qp->mp.a_bshape[d]; q.b_bshape[d] = qp->mp.b_bshape[d]; }
  if ((s = param_view(a_scale, a, qp->mp, true, &q.sa)) != MM_OK) return s;
  if ((s = param_view(a_zp, a, qp->mp, true, &q.za)) != MM_OK) return s;
  if ((s = param_view(b_scale, b, qp->mp, false, &q.sb)) != MM_OK) return s;
  if ((s = param_view(b_zp, b, qp->mp, false, &q.zb)) != MM_OK) return s;
  q.ys = y_scale->data; q.yz = y_zp->data;
  q.a_signed = a->dtype == MM_I8; q.b_signed = b->dtype == MM_I8; q.y_signed = y_zp->dtype == MM_I8;
  q.sa_f16 = a_scale->dtype == MM_F16; q.sb_f16 = b_scale->dtype == MM_F16; q.ys_f16 = y_scale->dtype == MM_F16;
  return MM_OK;
}

}  // namespace

mm_status mm_qlinear_matmul_workspace_size(const mm_tensor* a, const mm_tensor* b, size_t* bytes) {
  if (!bytes) return MM_ERR_INVALID_ARG;
  mm_status s;
  if ((s = check_tensor(a)) != MM_OK || (s = check_tensor(b)) != MM_OK) return s;
  if (!is_q8(a->dtype) || !is_q8(b->dtype)) return MM_ERR_DTYPE;
  MatmulPlan p;
  if ((s = plan_matmul(a, b, &p)) != MM_OK) return s;
  const int pol = g_policy.load();
  const bool want_tc = pol != MM_PATH_SIMT && (pol == MM_PATH_TENSOR || tensor_pays(p.M, p.N, p.K, p.bm.count));
  int64_t na = 1, nb = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) { na *= p.a_bshape[d]; nb *= p.b_bshape[d]; }
  *bytes = want_tc ? tc_qlinear_workspace_bytes(p.M, p.N, p.K, na, nb) : 0;
  return MM_OK;
}

mm_status mm_qlinear_matmul(const mm_tensor* a, const mm_tensor* a_scale, const mm_tensor* a_zero_point,
                            const mm_tensor* b, const mm_tensor* b_scale, const mm_tensor* b_zero_point,
                            const mm_tensor* y_scale, const mm_tensor* y_zero_point, const mm_tensor* y,
                            void* workspace, size_t workspace_bytes, void* stream) {
  QPlan qp;
  mm_status s = plan_qlinear(a, a_scale, a_zero_point, b, b_scale, b_zero_point, y_scale, y_zero_point, &qp);
  if (s != MM_OK) return s;
  if ((s = check_output(y, y_zero_point->dtype, qp.mp.out_ndim, qp.mp.out_shape)) != MM_OK) return s;
  qp.q.y = output_view(y, qp.mp, a->ndim == 1, b->ndim == 1);
  const QLinearArgs& q = qp.q;
  if (q.M == 0 || q.N == 0 || q.bm.count == 0) return finish(MM_OK, MM_PATH_NONE);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int path = choose(tc_qlinear_supported(q), tensor_pays(q.M, q.N, q.K, q.bm.count));
  if (path < 0) return MM_ERR_UNSUPPORTED;
  if (path == MM_PATH_TENSOR) {
    int64_t na = 1, nb = 1;
    for (int d = 0; d < kMaxBatchDims; ++d) { na *= q.a_bshape[d]; nb *= q.b_bshape[d]; }
    const size_t need = tc_qlinear_workspace_bytes(q.M, q.N, q.K, na, nb);
    if (need > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255)))
      return MM_ERR_WORKSPACE;
    return finish(launch_tc_qlinear(q, workspace, device_status_ptr(), st), MM_PATH_TENSOR);
  }
  return finish(launch_simt_qlinear(q, st), MM_PATH_SIMT);
}

// ------------------------------------------------------------------ GroupedMatMul

namespace {

mm_status plan_grouped(const mm_tensor* input, const mm_tensor* weights, const mm_tensor* gi,
                       const mm_tensor* bias, GroupedArgs* g) {
  mm_status s;
  if ((s = check_tensor(input)) != MM_OK || (s = check_tensor(weights)) != MM_OK || (s = check_tensor(gi)) != MM_OK)
    return s;
  if (bias && (s = check_tensor(bias)) != MM_OK) return s;
  const int dt = input->dtype;
  if (dt != MM_BF16 && dt != MM_F16 && dt != MM_F32 && dt != MM_F64) return MM_ERR_DTYPE;
  if (weights->dtype != dt || (bias && bias->dtype != dt)) return MM_ERR_DTYPE;
  if (gi->dtype != MM_I32 && gi->dtype != MM_I64) return MM_ERR_DTYPE;
  if (input->ndim != 2 || weights->ndim != 3 || gi->ndim != 2) return MM_ERR_SHAPE;
  if (weights->shape[1] != input->shape[1] || gi->shape[0] != input->shape[0]) return MM_ERR_SHAPE;
  if (bias && (bias->ndim != 2 || bias->shape[0] != weights->shape[0] || bias->shape[1] != weights->shape[2]))
    return MM_ERR_SHAPE;
  memset(g, 0, sizeof(*g));
  g->dtype = dt;
  g->ind64 = gi->dtype == MM_I64;
  g->M = input->shape[0]; g->K = input->shape[1];
  g->G = weights->shape[0]; g->N = weights->shape[2]; g->S = gi->shape[1];
  g->x = input->data; g->x_rs = input->strides[0]; g->x_cs = input->strides[1];
  g->w = weights->data; g->w_gs = weights->strides[0]; g->w_ks = weights->strides[1]; g->w_ns = weights->strides[2];
  g->gi = gi->data; g->gi_ms = gi->strides[0]; g->gi_ss = gi->strides[1];
  if (bias) { g->bias = bias->data; g->bias_gs = bias->strides[0]; g->bias_ns = bias->strides[1]; }
  return MM_OK;
}

}  // namespace

mm_status mm_grouped_matmul_workspace_size(const mm_tensor* input, const mm_tensor* weights,
                                           const mm_tensor* group_indices, size_t* bytes) {
  if (!bytes) return MM_ERR_INVALID_ARG;
  GroupedArgs g;
  mm_status s = plan_grouped(input, weights, group_indices, nullptr, &g);
  if (s != MM_OK) return s;
  const int pol = g_policy.load();
  const bool want_tc = pol != MM_PATH_SIMT &&
                       (pol == MM_PATH_TENSOR || tensor_pays(g.M * g.S, g.N, g.K, 1));
  *bytes = (want_tc && tc_grouped_supported(g)) ? tc_grouped_workspace_bytes(g) : 0;
  return MM_OK;
}

mm_status mm_grouped_matmul(const mm_tensor* input, const mm_tensor* weights, const mm_tensor* group_indices,
                            const mm_tensor* bias, const mm_tensor* output, void* workspace,
                            size_t workspace_bytes, void* stream) {
  GroupedArgs g;
  mm_status s = plan_grouped(input, weights, group_indices, bias, &g);
  if (s != MM_OK) return s;
  const int64_t oshape[3] = {g.M, g.S, g.N};
  if ((s = check_output(output, g.dtype, 3, oshape)) != MM_OK) return s;
  g.out = output->data;
  if (g.M == 0 || g.S == 0 || g.N == 0) return finish(MM_OK, MM_PATH_NONE);
  unsigned* status = device_status_ptr();
  if (!status) return MM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int path = choose(tc_grouped_supported(g), tensor_pays(g.M * g.S, g.N, g.K, 1));
  if (path < 0) return MM_ERR_UNSUPPORTED;
  if (path == MM_PATH_TENSOR) {
    const size_t need = tc_grouped_workspace_bytes(g);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
      return MM_ERR_WORKSPACE;
    return finish(launch_tc_grouped(g, workspace, status, st), MM_PATH_TENSOR);
  }
  return finish(launch_simt_grouped(g, status, st), MM_PATH_SIMT);
}

// ------------------------------------------------------------------ GroupedMatMul, weight-only quantized experts

namespace {

mm_status plan_grouped_q(const mm_tensor* input, const mm_tensor* weights_q, const mm_tensor* w_scale,
                         const mm_tensor* w_zero_point, int64_t block_size, const mm_tensor* gi,
                         const mm_tensor* bias, GroupedArgs* g) {
  mm_status s;
  if ((s = check_tensor(input)) != MM_OK || (s = check_tensor(weights_q)) != MM_OK ||
      (s = check_tensor(w_scale)) != MM_OK || (s = check_tensor(gi)) != MM_OK)
    return s;
  if (w_zero_point && (s = check_tensor(w_zero_point)) != MM_OK) return s;
  if (bias && (s = check_tensor(bias)) != MM_OK) return s;
  if (block_size < 0) return MM_ERR_INVALID_ARG;
  const int dt = input->dtype;
  if (dt != MM_BF16 && dt != MM_F16 && dt != MM_F32 && dt != MM_F64) return MM_ERR_DTYPE;
  if (!is_q8(weights_q->dtype) && !is_q4(weights_q->dtype)) return MM_ERR_DTYPE;
  if (w_scale->dtype != dt || (bias && bias->dtype != dt)) return MM_ERR_DTYPE;
  if (w_zero_point && w_zero_point->dtype != weights_q->dtype) return MM_ERR_DTYPE;
  if (gi->dtype != MM_I32 && gi->dtype != MM_I64) return MM_ERR_DTYPE;
  if (input->ndim != 2 || weights_q->ndim != 3 || gi->ndim != 2 || w_scale->ndim != 3) return MM_ERR_SHAPE;
  const int64_t G = weights_q->shape[0], K = weights_q->shape[1], N = weights_q->shape[2];
  if (K != input->shape[1] || gi->shape[0] != input->shape[0]) return MM_ERR_SHAPE;
  const int64_t block = block_size == 0 ? (K > 0 ? K : 1) : block_size;
  const int64_t kb = (K + block - 1) / block;
  if (w_scale->shape[0] != G || w_scale->shape[1] != kb || w_scale->shape[2] != N) return MM_ERR_SHAPE;
  if (w_zero_point) {
    if (w_zero_point->ndim != 3) return MM_ERR_SHAPE;
    for (int d = 0; d < 3; ++d)
      if (w_zero_point->shape[d] != w_scale->shape[d]) return MM_ERR_SHAPE;
  }
  if (bias && (bias->ndim != 2 || bias->shape[0] != G || bias->shape[1] != N)) return MM_ERR_SHAPE;
  if (is_q4(weights_q->dtype)) {
    // packed 4-bit rows start on byte boundaries: unit stride along N, N even
    // and even strides along G and K (for the zero points likewise)
    auto rows_on_bytes = [&](const mm_tensor* t) {
      return t->strides[2] == 1 && t->shape[2] % 2 == 0 && t->strides[1] % 2 == 0 && t->strides[0] % 2 == 0;
    };
    if (!rows_on_bytes(weights_q) || (w_zero_point && !rows_on_bytes(w_zero_point))) return MM_ERR_SHAPE;
  }
  memset(g, 0, sizeof(*g));
  g->dtype = dt;
  g->ind64 = gi->dtype == MM_I64;
  g->M = input->shape[0]; g->K = K; g->G = G; g->N = N; g->S = gi->shape[1];
  g->x = input->data; g->x_rs = input->strides[0]; g->x_cs = input->strides[1];
  g->w = weights_q->data;
  g->w_gs = weights_q->strides[0]; g->w_ks = weights_q->strides[1]; g->w_ns = weights_q->strides[2];
  g->gi = gi->data; g->gi_ms = gi->strides[0]; g->gi_ss = gi->strides[1];
  if (bias) { g->bias = bias->data; g->bias_gs = bias->strides[0]; g->bias_ns = bias->strides[1]; }
  switch (weights_q->dtype) {
    case MM_I8: g->wq = 1; break;
    case MM_U8: g->wq = 2; break;
    case MM_I4: g->wq = 3; break;
    default: g->wq = 4; break;
  }
  g->wsc = w_scale->data;
  g->wsc_gs = w_scale->strides[0]; g->wsc_bs = w_scale->strides[1]; g->wsc_ns = w_scale->strides[2];
  if (w_zero_point) {
    g->wzp = w_zero_point->data;
    g->wzp_gs = w_zero_point->strides[0]; g->wzp_bs = w_zero_point->strides[1]; g->wzp_ns = w_zero_point->strides[2];
  }
  g->qblock = block;
  return MM_OK;
}

}  // namespace

mm_status mm_grouped_matmul_qweights_workspace_size(const mm_tensor* input, const mm_tensor* weights_q,
                                                    const mm_tensor* w_scale, const mm_tensor* w_zero_point,
                                                    int64_t block_size, const mm_tensor* group_indices,
                                                    size_t* bytes) {
  if (!bytes) return MM_ERR_INVALID_ARG;
  GroupedArgs g;
  mm_status s = plan_grouped_q(input, weights_q, w_scale, w_zero_point, block_size, group_indices, nullptr, &g);
  if (s != MM_OK) return s;
  const int pol = g_policy.load();
  const bool want_tc = pol != MM_PATH_SIMT &&
                       (pol == MM_PATH_TENSOR || tensor_pays(g.M * g.S, g.N, g.K, 1));
  *bytes = (want_tc && tc_grouped_supported(g)) ? tc_grouped_workspace_bytes(g) : 0;
  return MM_OK;
}

mm_status mm_grouped_matmul_qweights(const mm_tensor* input, const mm_tensor* weights_q, const mm_tensor* w_scale,
                                     const mm_tensor* w_zero_point, int64_t block_size,
                                     const mm_tensor* group_indices, const mm_tensor* bias,
                                     const mm_tensor* output, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  GroupedArgs g;
  mm_status s = plan_grouped_q(input, weights_q, w_scale, w_zero_point, block_size, group_indices, bias, &g);
  if (s != MM_OK) return s;
  const int64_t oshape[3] = {g.M, g.S, g.N};
  if ((s = check_output(output, g.dtype, 3, oshape)) != MM_OK) return s;
  g.out = output->data;
  if (g.M == 0 || g.S == 0 || g.N == 0) return finish(MM_OK, MM_PATH_NONE);
  unsigned* status = device_status_ptr();
  if (!status) return MM_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int path = choose(tc_grouped_supported(g), tensor_pays(g.M * g.S, g.N, g.K, 1));
  if (path < 0) return MM_ERR_UNSUPPORTED;
  if (path == MM_PATH_TENSOR) {
    const size_t need = tc_grouped_workspace_bytes(g);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
      return MM_ERR_WORKSPACE;
    return finish(launch_tc_grouped(g, workspace, status, st), MM_PATH_TENSOR);
  }
  return finish(launch_simt_grouped(g, status, st), MM_PATH_SIMT);
}

// ------------------------------------------------------------------ GroupedMatMul without allocation
//
// Scratch for mm_grouped_matmul_noalloc: a fixed array in device memory that
// exists on every device where this library is loaded, from load until the
// process exits.  Host code may not use the symbol itself as a pointer (on the
// host it only names a stand-in object); the device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.

}  // extern "C"

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (NULL on failure).
void* noalloc_scratch_ptr() {
  static std::mutex mu;
  static void* ptrs[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" {

size_t mm_grouped_matmul_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

mm_status mm_grouped_matmul_noalloc(const mm_tensor* input, const mm_tensor* weights,
                                    const mm_tensor* group_indices, const mm_tensor* bias,
                                    const mm_tensor* output, void* stream) {
  GroupedArgs g;
  mm_status s = plan_grouped(input, weights, group_indices, bias, &g);
  if (s != MM_OK) return s;
  const int64_t oshape[3] = {g.M, g.S, g.N};
  if ((s = check_output(output, g.dtype, 3, oshape)) != MM_OK) return s;
  g.out = output->data;
  if (g.M == 0 || g.S == 0 || g.N == 0) return finish(MM_OK, MM_PATH_NONE);
  if (!tc_grouped_supported(g)) return MM_ERR_UNSUPPORTED;
  if (tc_grouped_workspace_bytes(g) > kNoAllocScratchBytes) return MM_ERR_WORKSPACE;
  unsigned* status = device_status_ptr();
  void* scratch = noalloc_scratch_ptr();
  if (!status || !scratch) return MM_ERR_CUDA;
  return finish(launch_tc_grouped(g, scratch, status, static_cast<cudaStream_t>(stream)), MM_PATH_TENSOR);
}

// ------------------------------------------------------------------ memory-stream measurement

mm_status mm_stream_probe(void* dst, const void* src, size_t bytes, int32_t mode, void* stream) {
  if (mode != kStreamWrite && mode != kStreamCopy && mode != kStreamWriteBulk) return MM_ERR_INVALID_ARG;
  if (bytes == 0) return MM_OK;
  if (!dst || (bytes & 15) || (reinterpret_cast<uintptr_t>(dst) & 15)) return MM_ERR_INVALID_ARG;
  if (mode == kStreamCopy && (!src || (reinterpret_cast<uintptr_t>(src) & 15))) return MM_ERR_INVALID_ARG;
  if (bytes > (size_t)INT64_MAX) return MM_ERR_INVALID_ARG;
  return launch_stream_probe(dst, src, (int64_t)bytes, mode, static_cast<cudaStream_t>(stream));
}

mm_status mm_alu_probe(int32_t op, void* out, int64_t iters, int64_t* multiply_adds, void* stream) {
  if (op != kAluImad && op != kAluDfma && op != kAluFfma) return MM_ERR_INVALID_ARG;
  if (iters < 0) return MM_ERR_INVALID_ARG;
  int threads = 0;
  const mm_status st = launch_alu_probe(op, nullptr, iters, &threads, static_cast<cudaStream_t>(stream));
  if (st != MM_OK) return st;
  if (multiply_adds) *multiply_adds = (int64_t)threads * kAluChains * iters;
  if (!out) return MM_OK;
  if (reinterpret_cast<uintptr_t>(out) & 7) return MM_ERR_INVALID_ARG;
  return launch_alu_probe(op, out, iters, nullptr, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ device status

mm_status mm_get_device_status(void* stream) {
  unsigned* p = device_status_ptr();
  if (!p) return MM_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MM_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MM_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MM_ERR_CUDA;
  }
  if (v & kStatusTimeout) return MM_ERR_TIMEOUT;
  if (v & kStatusIndexRange) return MM_ERR_INDEX_RANGE;
  return MM_OK;
}

}  // extern "C"
