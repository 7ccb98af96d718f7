// Plain CPU oracle for the ONNX matrix-product family, in C++
// (TEST INFRASTRUCTURE ONLY).
//
// A second, independent statement of what the operator pages define, written
// as plain loops: no BLAS, no blocking, no reordering of any sum.  It shares
// no code with the CUDA library (it includes none of its headers and is built
// separately by g++) nor with the numpy oracle beside it; the ctypes binding
// in oracle/native.py only converts arrays and raises on error codes.  Only
// tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and reference
// legs load it.
//
// Arithmetic conventions:
//  * Floating point: operands arrive widened exactly to double.  Every output
//    element is the sum over k = 0, 1, ..., K-1 of the products, each product
//    and each partial sum rounded once in double, in that order (the build
//    passes -ffp-contract=off so no multiply-add is fused).  The result is
//    left unrounded (double).
//  * Integers: operands arrive as 64-bit two's-complement bit patterns;
//    sums and products are taken modulo 2^64 (uint64_t wraps) and the result
//    is reduced modulo 2^n of the operator's type, which equals numpy's
//    wrap-around in the n-bit type whatever the order of the sum.
//  * QLinearMatMul: the accumulator is the exact integer sum (int64),
//    reduced modulo 2^32; the requantisation is a fixed sequence of float
//    operations (float is IEEE binary32 and is evaluated as such on the
//    x86-64 and AArch64 targets this is built for).
//
// Loops run over output rows in parallel (OpenMP); every output element is
// computed by one thread in the order above, so the result does not depend on
// the thread count.
//
// Each function cites the page and section it follows:
//  * MatMul (onnx-light, ai.onnx since version 13): summary -- the matrix
//    product behaves like numpy.matmul; examples for 1-D operands and
//    broadcast batch dimensions.
//  * Gemm (onnx-light, since version 13): definition, Inputs, Outputs.
//  * QLinearMatMul - version 10: summary (quantization formula, rounding,
//    saturation, scale and zero-point shapes, 32-bit accumulation).
//  * GroupedMatMul - 29: Summary, Inputs, Outputs; last paragraph of the
//    Summary for weight-only quantized experts (DequantizeLinear of the
//    weights, then GroupedMatMul).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum {
  ORC_OK = 0,
  ORC_ERR_SHAPE = 1,    // shapes violate the operator's rules
  ORC_ERR_TYPE = 2,     // element types violate the type constraints
  ORC_ERR_INDEX = 3,    // a group index outside [0, G)
  ORC_ERR_RANGE = 4,    // an integer Gemm result outside T's range (undefined)
  ORC_ERR_ARG = 5,      // invalid argument (negative size, too many dimensions, ...)
};

constexpr int kMaxDims = 16;

// ------------------------------------------------------------------ MatMul shapes
//
// numpy.matmul rules (MatMul page, summary and the examples
// test_cc_matmul_1d_1d, _1d_3d, _4d_1d, _bcast, _batch_broadcast):
//  1. a 1-D first operand [K] is read as [1, K], and that dimension is removed
//     from the result;
//  2. a 1-D second operand [K] is read as [K, 1], likewise removed;
//  3. all dimensions but the last two are batch dimensions, aligned from the
//     right (missing ones count as 1); each pair must be equal or contain a 1,
//     which is stretched;
//  4. Y[b, i, j] = sum_k A[b, i, k] * B[b, k, j] for every batch index b.
struct MatmulShape {
  int nb;                        // number of broadcast batch dimensions
  int64_t batch[kMaxDims];       // broadcast batch shape
  int64_t a_bstride[kMaxDims];   // A's stride per batch dimension, in matrices (0 where stretched)
  int64_t b_bstride[kMaxDims];
  int64_t count;                 // number of batch indices
  int64_t M, K, N;
  int out_nd;
  int64_t out[kMaxDims + 2];
};

int matmul_shape(int a_nd, const int64_t* as, int b_nd, const int64_t* bs, MatmulShape* p) {
  if (a_nd < 1 || b_nd < 1) return ORC_ERR_SHAPE;        // a 0-D operand has no matrix reading
  if (a_nd > kMaxDims || b_nd > kMaxDims) return ORC_ERR_ARG;
  for (int d = 0; d < a_nd; ++d) if (as[d] < 0) return ORC_ERR_ARG;
  for (int d = 0; d < b_nd; ++d) if (bs[d] < 0) return ORC_ERR_ARG;
  // Steps 1-2: promoted shapes.
  int64_t pa[kMaxDims + 1] = {}, pb[kMaxDims + 1] = {};
  int pan = 0, pbn = 0;
  if (a_nd == 1) { pa[0] = 1; pa[1] = as[0]; pan = 2; }
  else { for (int d = 0; d < a_nd; ++d) pa[d] = as[d]; pan = a_nd; }
  if (b_nd == 1) { pb[0] = bs[0]; pb[1] = 1; pbn = 2; }
  else { for (int d = 0; d < b_nd; ++d) pb[d] = bs[d]; pbn = b_nd; }
  p->M = pa[pan - 2];
  p->K = pa[pan - 1];
  if (pb[pbn - 2] != p->K) return ORC_ERR_SHAPE;
  p->N = pb[pbn - 1];
  // Step 3: right-aligned broadcast of the batch dimensions.
  const int na = pan - 2, nbb = pbn - 2;
  p->nb = na > nbb ? na : nbb;
  // Each operand's own batch dimensions, as strides in whole matrices.
  int64_t a_own[kMaxDims], b_own[kMaxDims];
  {
    int64_t s = 1;
    for (int d = na - 1; d >= 0; --d) { a_own[d] = s; s *= pa[d]; }
    s = 1;
    for (int d = nbb - 1; d >= 0; --d) { b_own[d] = s; s *= pb[d]; }
  }
  p->count = 1;
  for (int d = 0; d < p->nb; ++d) {
    const int da = d - (p->nb - na), db = d - (p->nb - nbb);
    const int64_t sa = da >= 0 ? pa[da] : 1, sb = db >= 0 ? pb[db] : 1;
    int64_t so;
    if (sa == sb || sb == 1) so = sa;
    else if (sa == 1) so = sb;
    else return ORC_ERR_SHAPE;
    p->batch[d] = so;
    p->a_bstride[d] = (da >= 0 && sa != 1) ? a_own[da] : 0;
    p->b_bstride[d] = (db >= 0 && sb != 1) ? b_own[db] : 0;
    p->count *= so;
  }
  int k = 0;
  for (int d = 0; d < p->nb; ++d) p->out[k++] = p->batch[d];
  if (a_nd > 1) p->out[k++] = p->M;
  if (b_nd > 1) p->out[k++] = p->N;
  p->out_nd = k;
  return ORC_OK;
}

// Matrix index of each operand for the flat batch index b (row-major over the
// broadcast batch shape).
void batch_matrices(const MatmulShape& p, int64_t b, int64_t* am, int64_t* bm) {
  int64_t ia = 0, ib = 0;
  for (int d = p.nb - 1; d >= 0; --d) {
    const int64_t i = b % p.batch[d];
    b /= p.batch[d];
    ia += i * p.a_bstride[d];
    ib += i * p.b_bstride[d];
  }
  *am = ia;
  *bm = ib;
}

int threads_or_default(int threads) {
#ifdef _OPENMP
  return threads > 0 ? threads : omp_get_max_threads();
#else
  (void)threads;
  return 1;
#endif
}

// One output row of a float product: y[j] = sum_k a[k*as] * b[k*bk + j*bj],
// summed over k in increasing order (two loop orders, the same arithmetic for
// every element: the one whose inner loop walks contiguous memory is used).
void row_f64(const double* a, int64_t as, const double* b, int64_t bk, int64_t bj, int64_t K, int64_t N,
             double* y, bool absval) {
  if (bj == 1 || bk != 1) {
    for (int64_t j = 0; j < N; ++j) y[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double av = absval ? std::fabs(a[k * as]) : a[k * as];
      const double* bp = b + k * bk;
      if (absval)
        for (int64_t j = 0; j < N; ++j) y[j] = y[j] + av * std::fabs(bp[j * bj]);
      else
        for (int64_t j = 0; j < N; ++j) y[j] = y[j] + av * bp[j * bj];
    }
  } else {
    for (int64_t j = 0; j < N; ++j) {
      const double* bp = b + j * bj;
      double s = 0.0;
      if (absval)
        for (int64_t k = 0; k < K; ++k) s = s + std::fabs(a[k * as]) * std::fabs(bp[k]);
      else
        for (int64_t k = 0; k < K; ++k) s = s + a[k * as] * bp[k];
      y[j] = s;
    }
  }
}

// The same for integers, modulo 2^64.
void row_u64(const uint64_t* a, int64_t as, const uint64_t* b, int64_t bk, int64_t bj, int64_t K, int64_t N,
             uint64_t* y) {
  for (int64_t j = 0; j < N; ++j) y[j] = 0;
  for (int64_t k = 0; k < K; ++k) {
    const uint64_t av = a[k * as];
    const uint64_t* bp = b + k * bk;
    for (int64_t j = 0; j < N; ++j) y[j] += av * bp[j * bj];
  }
}

uint64_t low_bits(uint64_t x, int bits) { return bits >= 64 ? x : (x & ((uint64_t(1) << bits) - 1)); }

// ------------------------------------------------------------------ Gemm operand and C mapping
//
// Gemm page, definition and Inputs: A' = transpose(A) if transA else A,
// A of shape (M, K) or (K, M); likewise B' from B of shape (K, N) or (N, K);
// C optional and unidirectionally broadcastable to (M, N): read as numpy
// broadcasting in which only C is stretched (rank <= 2, right-aligned, each
// dimension equal to the target or 1).
struct GemmShape {
  int64_t M, K, N;
  int64_t a_rs, a_cs, b_rs, b_cs;   // element strides of A' and B' (row, column)
  int64_t c_rs, c_cs;               // element strides of stretched C (0 along stretched dims)
};

int gemm_shape(int64_t a0, int64_t a1, int64_t b0, int64_t b1, int trans_a, int trans_b, int c_nd,
               const int64_t* cs, GemmShape* g) {
  if (a0 < 0 || a1 < 0 || b0 < 0 || b1 < 0) return ORC_ERR_ARG;
  g->M = trans_a ? a1 : a0;
  g->K = trans_a ? a0 : a1;
  const int64_t k2 = trans_b ? b1 : b0;
  g->N = trans_b ? b0 : b1;
  if (g->K != k2) return ORC_ERR_SHAPE;
  // A stored (a0, a1) row-major: A'[i, k] = A[i, k] or A[k, i].
  g->a_rs = trans_a ? 1 : a1;
  g->a_cs = trans_a ? a1 : 1;
  g->b_rs = trans_b ? 1 : b1;
  g->b_cs = trans_b ? b1 : 1;
  g->c_rs = g->c_cs = 0;
  if (c_nd < 0) return ORC_OK;                      // C absent
  if (c_nd > 2) return ORC_ERR_SHAPE;
  const int64_t tgt[2] = {g->M, g->N};
  int64_t st[2] = {0, 0};
  int64_t s = 1;
  for (int d = c_nd - 1; d >= 0; --d) {
    const int td = 2 - c_nd + d;
    if (cs[d] != tgt[td] && cs[d] != 1) return ORC_ERR_SHAPE;
    st[td] = cs[d] == 1 ? 0 : s;
    s *= cs[d];
  }
  g->c_rs = st[0];
  g->c_cs = st[1];
  return ORC_OK;
}

// alpha (a float attribute) as an integer modulo 2^64, when it is integral.
bool integral_mod64(float x, uint64_t* out) {
  if (!std::isfinite(x) || x != std::floor(x)) return false;
  const double ax = std::fabs((double)x);
  uint64_t m;
  if (ax < 9223372036854775808.0) {
    m = (uint64_t)(int64_t)ax;
  } else {
    // |x| = mant * 2^e with a 24-bit integer mant: reduce modulo 2^64.
    int e2 = 0;
    const double f = std::frexp(ax, &e2);            // ax = f * 2^e2, f in [0.5, 1)
    const uint64_t mant = (uint64_t)std::ldexp(f, 24);
    const int sh = e2 - 24;
    m = sh >= 64 ? 0 : (mant << sh);
  }
  *out = x < 0 ? (uint64_t)0 - m : m;
  return true;
}

// ------------------------------------------------------------------ float rounding to a type
//
// Round x to the nearest value of a binary format with p significant bits and
// minimum normal exponent emin (ties to even), from the format's definition:
// the spacing of representable values around x is 2^(max(floor(log2|x|), emin)
// - (p - 1)); values beyond the largest finite one become infinities.
double round_format(double x, int p, int emin, double max_finite) {
  if (!std::isfinite(x) || x == 0.0) return x;
  int e2 = 0;
  std::frexp(x, &e2);                                // |x| in [2^(e2-1), 2^e2)
  int ex = e2 - 1;
  if (ex < emin) ex = emin;
  const double quantum = std::ldexp(1.0, ex - (p - 1));
  const double r = std::nearbyint(x / quantum) * quantum;
  if (std::fabs(r) > max_finite) return x < 0 ? -INFINITY : INFINITY;
  return r;
}

double round_to_type(double x, int t) {
  switch (t) {
    case 0: return round_format(x, 8, -126, std::ldexp(255.0, 120));       // bfloat16
    case 1: return round_format(x, 11, -14, 65504.0);                      // float16
    case 2: return (double)(float)x;                                        // float
    default: return x;                                                      // double
  }
}

}  // namespace

extern "C" {

int orc_num_threads(int threads) { return threads_or_default(threads); }

// ------------------------------------------------------------------ MatMul

int orc_matmul_shape(int a_nd, const int64_t* a_shape, int b_nd, const int64_t* b_shape, int* out_nd,
                     int64_t* out_shape) {
  MatmulShape p;
  const int s = matmul_shape(a_nd, a_shape, b_nd, b_shape, &p);
  if (s != ORC_OK) return s;
  *out_nd = p.out_nd;
  for (int d = 0; d < p.out_nd; ++d) out_shape[d] = p.out[d];
  return ORC_OK;
}

// Y = A @ B for float operands (dense row-major, widened to double); with
// absval, Y = |A| @ |B| (the per-element error-bound denominator).
int orc_matmul_f64(int a_nd, const int64_t* a_shape, const double* A, int b_nd, const int64_t* b_shape,
                   const double* B, double* Y, int absval, int threads) {
  MatmulShape p;
  const int s = matmul_shape(a_nd, a_shape, b_nd, b_shape, &p);
  if (s != ORC_OK) return s;
  const int64_t rows = p.count * p.M, M = p.M, K = p.K, N = p.N;
  const int nt = threads_or_default(threads);
  (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t am, bm;
    batch_matrices(p, r / M, &am, &bm);
    const int64_t i = r % M;
    row_f64(A + am * M * K + i * K, 1, B + bm * K * N, N, 1, K, N, Y + r * N, absval != 0);
  }
  return ORC_OK;
}

// Integer MatMul: operands are 64-bit two's-complement bit patterns of
// n-bit values; Y holds the low n bits of the exact result.
int orc_matmul_u64(int a_nd, const int64_t* a_shape, const uint64_t* A, int b_nd, const int64_t* b_shape,
                   const uint64_t* B, uint64_t* Y, int bits, int threads) {
  MatmulShape p;
  const int s = matmul_shape(a_nd, a_shape, b_nd, b_shape, &p);
  if (s != ORC_OK) return s;
  const int64_t rows = p.count * p.M, M = p.M, K = p.K, N = p.N;
  const int nt = threads_or_default(threads);
  (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t am, bm;
    batch_matrices(p, r / M, &am, &bm);
    uint64_t* y = Y + r * N;
    row_u64(A + am * M * K + (r % M) * K, 1, B + bm * K * N, N, 1, K, N, y);
    for (int64_t j = 0; j < N; ++j) y[j] = low_bits(y[j], bits);
  }
  return ORC_OK;
}

// ------------------------------------------------------------------ Gemm

int orc_gemm_shape(int64_t a0, int64_t a1, int64_t b0, int64_t b1, int trans_a, int trans_b, int c_nd,
                   const int64_t* c_shape, int64_t* M, int64_t* N) {
  GemmShape g;
  const int s = gemm_shape(a0, a1, b0, b1, trans_a, trans_b, c_nd, c_shape, &g);
  if (s != ORC_OK) return s;
  *M = g.M;
  *N = g.N;
  return ORC_OK;
}

// Float Gemm: Y = alpha * (A' @ B') + beta * C, each product, the row sums and
// the final sum rounded in double (alpha and beta are float attributes,
// widened exactly).  C is NULL when absent (c_nd < 0).  With absval,
// Y = |alpha| * (|A'| @ |B'|) + |beta| * |C|: the error-bound denominator.
int orc_gemm_f64(int64_t a0, int64_t a1, const double* A, int64_t b0, int64_t b1, const double* B, int c_nd,
                 const int64_t* c_shape, const double* C, double alpha, double beta, int trans_a, int trans_b,
                 double* Y, int absval, int threads) {
  GemmShape g;
  const int s = gemm_shape(a0, a1, b0, b1, trans_a, trans_b, C ? c_nd : -1, c_shape, &g);
  if (s != ORC_OK) return s;
  double al = (double)(float)alpha, be = (double)(float)beta;
  if (absval) { al = std::fabs(al); be = std::fabs(be); }
  const int nt = threads_or_default(threads);
  (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int64_t i = 0; i < g.M; ++i) {
    double* y = Y + i * g.N;
    row_f64(A + i * g.a_rs, g.a_cs, B, g.b_rs, g.b_cs, g.K, g.N, y, absval != 0);
    for (int64_t j = 0; j < g.N; ++j) {
      double v = al * y[j];
      if (C) {
        const double c = C[i * g.c_rs + j * g.c_cs];
        v = v + be * (absval ? std::fabs(c) : c);
      }
      y[j] = v;
    }
  }
  return ORC_OK;
}

// Integer Gemm (T of `bits` bits, signed or not).  The page does not say how a
// real-valued alpha * acc + beta * C becomes a T.  With integral alpha and
// beta, Y = alpha * acc + beta * C exactly modulo 2^n.  Otherwise acc, the
// product A' @ B' taken modulo 2^n as a T value, is rounded to double; then
// r = alpha * acc + beta * C in double (each product rounded, then the sum)
// is truncated toward zero; a result outside T's range is undefined and
// returns ORC_ERR_RANGE.
int orc_gemm_u64(int64_t a0, int64_t a1, const uint64_t* A, int64_t b0, int64_t b1, const uint64_t* B, int c_nd,
                 const int64_t* c_shape, const uint64_t* C, double alpha, double beta, int trans_a, int trans_b,
                 uint64_t* Y, int bits, int is_signed, int threads) {
  GemmShape g;
  const int s = gemm_shape(a0, a1, b0, b1, trans_a, trans_b, C ? c_nd : -1, c_shape, &g);
  if (s != ORC_OK) return s;
  const float af = (float)alpha, bf = (float)beta;
  uint64_t ai = 0, bi = 0;
  const bool integral = integral_mod64(af, &ai) && integral_mod64(bf, &bi);
  const int nt = threads_or_default(threads);
  (void)nt;
  int err = ORC_OK;
  const double lo = is_signed ? -std::ldexp(1.0, bits - 1) : 0.0;
  const double hi = is_signed ? std::ldexp(1.0, bits - 1) : std::ldexp(1.0, bits);
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int64_t i = 0; i < g.M; ++i) {
    uint64_t* y = Y + i * g.N;
    row_u64(A + i * g.a_rs, g.a_cs, B, g.b_rs, g.b_cs, g.K, g.N, y);
    for (int64_t j = 0; j < g.N; ++j) {
      const uint64_t acc = low_bits(y[j], bits);
      const uint64_t c = C ? C[i * g.c_rs + j * g.c_cs] : 0;
      if (integral) {
        y[j] = low_bits(ai * acc + (C ? bi * c : 0), bits);
        continue;
      }
      // The wrapped accumulator and C as T values (sign-extended when signed).
      auto as_double = [&](uint64_t v) {
        if (is_signed) {
          const uint64_t sign = uint64_t(1) << (bits - 1);
          const int64_t sv = (int64_t)((v ^ sign) - sign);
          return (double)sv;
        }
        return (double)v;
      };
      double r = (double)af * as_double(acc);
      if (C) r = r + (double)bf * as_double(low_bits(c, bits));
      const double t = std::trunc(r);
      if (!(t >= lo && t < hi)) {
#pragma omp atomic write
        err = ORC_ERR_RANGE;
        y[j] = 0;
        continue;
      }
      y[j] = low_bits(is_signed ? (uint64_t)(int64_t)t : (uint64_t)t, bits);
    }
  }
  return err;
}

// ------------------------------------------------------------------ QLinearMatMul
//
// QLinearMatMul - version 10, summary: acc = sum_k (a - a_zero_point) *
// (b - b_zero_point), exact, reduced to int32 (the page allows overflow only
// in the 32-bit accumulation); y = saturate(round(x / y_scale) + y_zero_point)
// with round-half-to-even, x the real-valued product a_scale * b_scale * acc.
// Readings: x / y_scale is evaluated in float as s = a_scale * b_scale;
// v = float(acc) * s; q = v / y_scale; r = rint(q); t = r + y_zero_point;
// then clamped with fmin/fmax (a NaN saturates to the low end).  A scale and
// its zero point are per tensor (one element), per row of a (M elements:
// [M] for 2-D a, or a.shape[:-1] + [1]) or per column of b (N elements: [N]
// for 2-D b, or b.shape[:-2] + [1, N]); the page's "K elements" for the
// per-column vector cannot index the columns of the result.

namespace {

// Index rule of one quantisation parameter: per tensor (unit = 0), or one
// value per row of the operand's flat row list (a: batch-matrix * M + m) or
// per column (b: batch-matrix * N + n).
int param_kind(int p_nd, const int64_t* ps, int x_nd, const int64_t* xs, bool per_row, int* kind) {
  int64_t numel = 1;
  for (int d = 0; d < p_nd; ++d) numel *= ps[d];
  if (numel == 1) { *kind = 0; return ORC_OK; }
  if (x_nd < 2) return ORC_ERR_SHAPE;
  const int64_t len = per_row ? xs[x_nd - 2] : xs[x_nd - 1];
  if (p_nd == 1 && x_nd == 2) {
    if (ps[0] != len) return ORC_ERR_SHAPE;
    *kind = 1;
    return ORC_OK;
  }
  if (p_nd != x_nd) return ORC_ERR_SHAPE;
  for (int d = 0; d < x_nd - 2; ++d)
    if (ps[d] != xs[d]) return ORC_ERR_SHAPE;
  if (per_row) {
    if (ps[x_nd - 2] != len || ps[x_nd - 1] != 1) return ORC_ERR_SHAPE;
  } else {
    if (ps[x_nd - 2] != 1 || ps[x_nd - 1] != len) return ORC_ERR_SHAPE;
  }
  *kind = 1;
  return ORC_OK;
}

bool same_shape(int n1, const int64_t* s1, int n2, const int64_t* s2) {
  if (n1 != n2) return false;
  for (int d = 0; d < n1; ++d)
    if (s1[d] != s2[d]) return false;
  return true;
}

float requant_one(int32_t acc, float sa, float sb, float ys, int32_t yz, float qmin, float qmax) {
  const float s = sa * sb;
  const float v = (float)acc * s;
  const float q = v / ys;
  const float r = std::nearbyint(q);       // the default rounding mode: to nearest, ties to even
  const float t = r + (float)yz;
  return std::fmin(std::fmax(t, qmin), qmax);
}

}  // namespace

// The requantisation step alone, element by element (n elements).
int orc_requantize(int64_t n, const int32_t* acc, const float* sa, const float* sb, float ys, int32_t yz,
                   int y_unsigned, int32_t* y) {
  const float qmin = y_unsigned ? 0.f : -128.f, qmax = y_unsigned ? 255.f : 127.f;
  for (int64_t i = 0; i < n; ++i) y[i] = (int32_t)requant_one(acc[i], sa[i], sb[i], ys, yz, qmin, qmax);
  return ORC_OK;
}

// Types are 0 = int8, 1 = uint8 (anything else: ORC_ERR_TYPE).  a, b and the
// zero points arrive widened to int32, the scales as float (float16 scales
// widened exactly).  y receives the saturated values as int32.
int orc_qlinear_matmul(int a_nd, const int64_t* a_shape, const int32_t* a, int a_type,
                       int sa_nd, const int64_t* sa_shape, const float* sa,
                       int za_nd, const int64_t* za_shape, const int32_t* za, int za_type,
                       int b_nd, const int64_t* b_shape, const int32_t* b, int b_type,
                       int sb_nd, const int64_t* sb_shape, const float* sb,
                       int zb_nd, const int64_t* zb_shape, const int32_t* zb, int zb_type,
                       int64_t ys_numel, const float* ys, int64_t yz_numel, const int32_t* yz, int y_type,
                       int32_t* y, int threads) {
  if ((a_type != 0 && a_type != 1) || (b_type != 0 && b_type != 1) || (y_type != 0 && y_type != 1))
    return ORC_ERR_TYPE;
  if (za_type != a_type || zb_type != b_type) return ORC_ERR_TYPE;
  if (!same_shape(sa_nd, sa_shape, za_nd, za_shape) || !same_shape(sb_nd, sb_shape, zb_nd, zb_shape))
    return ORC_ERR_SHAPE;
  if (ys_numel != 1 || yz_numel != 1) return ORC_ERR_SHAPE;
  MatmulShape p;
  int s = matmul_shape(a_nd, a_shape, b_nd, b_shape, &p);
  if (s != ORC_OK) return s;
  int ka = 0, kb = 0;
  if ((s = param_kind(sa_nd, sa_shape, a_nd, a_shape, true, &ka)) != ORC_OK) return s;
  if ((s = param_kind(sb_nd, sb_shape, b_nd, b_shape, false, &kb)) != ORC_OK) return s;
  const int64_t rows = p.count * p.M, M = p.M, K = p.K, N = p.N;
  const float qmin = y_type ? 0.f : -128.f, qmax = y_type ? 255.f : 127.f;
  const float y_scale = ys[0];
  const int32_t y_zp = yz[0];
  const int nt = threads_or_default(threads);
  (void)nt;
#pragma omp parallel num_threads(nt)
  {
    std::vector<int64_t> acc((size_t)N);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      int64_t am, bm;
      batch_matrices(p, r / M, &am, &bm);
      const int64_t m = r % M;
      const int64_t ia = ka ? am * M + m : 0;           // a's parameters for this row
      const int32_t* arow = a + am * M * K + m * K;
      const int32_t* bmat = b + bm * K * N;
      const int32_t* zbrow = zb + (kb ? bm * N : 0);
      for (int64_t n = 0; n < N; ++n) acc[n] = 0;
      for (int64_t k = 0; k < K; ++k) {
        const int64_t av = (int64_t)arow[k] - (int64_t)za[ia];
        const int32_t* brow = bmat + k * N;
        for (int64_t n = 0; n < N; ++n) acc[n] += av * ((int64_t)brow[n] - (int64_t)zbrow[kb ? n : 0]);
      }
      const float* sbrow = sb + (kb ? bm * N : 0);
      for (int64_t n = 0; n < N; ++n) {
        const int32_t a32 = (int32_t)(uint32_t)(uint64_t)acc[n];      // modulo 2^32
        y[r * N + n] = (int32_t)requant_one(a32, sa[ia], sbrow[kb ? n : 0], y_scale, y_zp, qmin, qmax);
      }
    }
  }
  return ORC_OK;
}

// ------------------------------------------------------------------ GroupedMatMul
//
// GroupedMatMul - 29, Summary, Inputs, Outputs: input [M, K], weights
// [G, K, N], group_indices [M, S] (int32 or int64: ind_type 0 or 1), bias
// [G, N] (optional: b_nd < 0); output [M, S, N].
int orc_grouped_shape(int x_nd, const int64_t* xs, int w_nd, const int64_t* ws, int gi_nd, const int64_t* gs,
                      int ind_type, int b_nd, const int64_t* bs, int64_t* dims /* M, K, G, N, S */) {
  if (x_nd != 2 || w_nd != 3 || gi_nd != 2) return ORC_ERR_SHAPE;
  if (ind_type != 0 && ind_type != 1) return ORC_ERR_TYPE;
  if (ws[1] != xs[1] || gs[0] != xs[0]) return ORC_ERR_SHAPE;
  if (b_nd >= 0 && (b_nd != 2 || bs[0] != ws[0] || bs[1] != ws[2])) return ORC_ERR_SHAPE;
  dims[0] = xs[0]; dims[1] = xs[1]; dims[2] = ws[0]; dims[3] = ws[2]; dims[4] = gs[1];
  for (int d = 0; d < 5; ++d) if (dims[d] < 0) return ORC_ERR_ARG;
  return ORC_OK;
}

// output[m, i] = input[m] @ weights[g] (+ bias[g]) with g = group_indices[m, i];
// every index must lie in [0, G) (the page leaves anything else undefined:
// ORC_ERR_INDEX, nothing is computed).  The page defines the result through
// Gather / Expand / MatMul; the loop below is the same mathematics per output
// row.  The bias is added to the finished row sum.  With absval the result is
// |input| @ |weights[g]| + |bias[g]|, the error-bound denominator.
int orc_grouped_matmul_f64(int64_t M, int64_t K, int64_t G, int64_t N, int64_t S, const double* x,
                           const double* w, const int64_t* gi, const double* bias, double* out, int absval,
                           int threads) {
  if (M < 0 || K < 0 || G < 0 || N < 0 || S < 0) return ORC_ERR_ARG;
  for (int64_t r = 0; r < M * S; ++r)
    if (gi[r] < 0 || gi[r] >= G) return ORC_ERR_INDEX;
  const int nt = threads_or_default(threads);
  (void)nt;
#pragma omp parallel for schedule(static) num_threads(nt)
  for (int64_t r = 0; r < M * S; ++r) {
    const int64_t m = r / S, g = gi[r];
    double* y = out + r * N;
    row_f64(x + m * K, 1, w + g * K * N, N, 1, K, N, y, absval != 0);
    if (bias)
      for (int64_t n = 0; n < N; ++n) y[n] = y[n] + (absval ? std::fabs(bias[g * N + n]) : bias[g * N + n]);
  }
  return ORC_OK;
}

// DequantizeLinear of the weights (the Summary's last paragraph names it
// without defining it; reading): q [G, K, N] of int8 (q_type 0) or uint8 (1);
// scale and zero point of one shape [G, Kb, N], Kb = ceil(K / block) (block 0
// means K); the zero point has q's type, or is absent (zp_nd < 0: 0);
// W[g, k, n] = T((q[g, k, n] - zp[g, k / block, n]) * scale[g, k / block, n]),
// the difference an exact integer and the product rounded once to T
// (t: 0 bfloat16, 1 float16, 2 float, 3 double; the scale values are T's,
// passed as double).
int orc_dequantize_linear(int q_nd, const int64_t* qs, const int32_t* q, int q_type, int s_nd, const int64_t* ss,
                          const double* scale, int zp_nd, const int64_t* zs, const int32_t* zp, int zp_type,
                          int64_t block, int t, double* W) {
  if (q_nd != 3 || (q_type != 0 && q_type != 1)) return ORC_ERR_TYPE;
  if (t < 0 || t > 3) return ORC_ERR_TYPE;
  if (zp_nd >= 0 && zp_type != q_type) return ORC_ERR_TYPE;
  const int64_t G = qs[0], K = qs[1], N = qs[2];
  if (block < 0) return ORC_ERR_ARG;
  const int64_t bl = block == 0 ? (K > 0 ? K : 1) : block;
  const int64_t kb = (K + bl - 1) / bl;
  if (s_nd != 3 || ss[0] != G || ss[1] != kb || ss[2] != N) return ORC_ERR_SHAPE;
  if (zp_nd >= 0 && !same_shape(zp_nd, zs, s_nd, ss)) return ORC_ERR_SHAPE;
  for (int64_t g = 0; g < G; ++g)
    for (int64_t k = 0; k < K; ++k)
      for (int64_t n = 0; n < N; ++n) {
        const int64_t pi = (g * kb + k / bl) * N + n;
        const int64_t diff = (int64_t)q[(g * K + k) * N + n] - (zp_nd >= 0 ? (int64_t)zp[pi] : 0);
        W[(g * K + k) * N + n] = round_to_type((double)diff * scale[pi], t);
      }
  return ORC_OK;
}

// Rounding of double values to a type (the rule of orc_dequantize_linear).
int orc_round_to_type(int64_t n, const double* x, int t, double* y) {
  if (t < 0 || t > 3) return ORC_ERR_TYPE;
  for (int64_t i = 0; i < n; ++i) y[i] = round_to_type(x[i], t);
  return ORC_OK;
}

}  // extern "C"
