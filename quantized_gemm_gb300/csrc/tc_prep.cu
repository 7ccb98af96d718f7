// Front ends of the tensor-core path for QLinearMatMul and GroupedMatMul: the
// kernels that prepare operands in the caller's workspace, then the launch of
// the shared tcgen05 GEMM (tc_gemm.cu).
//
// QLinearMatMul (QLinearMatMul - version 10, summary): acc = sum_k (a - a_zp)(b - b_zp).
//   GB300 has no int8 tensor-core instruction (tcgen05 kind::i8 does not exist
//   on sm_103a), so each operand is rewritten once, exactly, in f16 (shifted
//   into [-128, 127]) together with its row or column sums; the GEMM runs on
//   the f16 pipe with segment-exact fp32 accumulation and an int32 epilogue
//   that applies the zero points.
//
// GroupedMatMul (GroupedMatMul - 29, summary): rows (m, i) are routed to their
//   group on the device: a histogram of group_indices, an exclusive scan into
//   per-group row offsets and per-group tile ranges, and a scatter that writes
//   each row's output index and copies input[m] into a group-ordered row
//   buffer.  The GEMM then multiplies each group's contiguous rows by
//   weights[g] in place (the [M*S, K, N] selected weights are never formed) and
//   scatters results to output[m, i, :].
#include <cstring>

#include "tc.h"
#include "tc_internal.h"

namespace qg {
namespace {

constexpr int64_t kAlign = 256;

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ QLinear: operands to f16 + sums
//
// Each operand is rewritten once as x' = x - c (c = 128 for uint8, 0 for
// int8), so x' lies in [-128, 127] for both types and is exact in f16.  The
// zero points are not applied here: with za' = za - c_a and zb' = zb - c_b,
//   sum_k (a - za)(b - zb) = sum_k a'b' - zb' * rs - za' * cs + K * za' * zb'
// where rs[m] = sum_k a'[m, k] and cs[n] = sum_k b'[k, n]; the GEMM epilogue
// applies this (int32, wrapping).  Products |a'b'| <= 2^14 let 1024-deep
// segments accumulate exactly in fp32 (|sum| <= 2^24).

struct ShiftArgs {
  const uint8_t* src;
  int is_signed;                       // int8 (shift 0) or uint8 (shift 128)
  int nb;
  int64_t own_shape[kMaxBatchDims];    // operand's own batch shape (1 where broadcast)
  int64_t src_bstride[kMaxBatchDims];
  int64_t src_rs, src_cs;
  int64_t rows, cols, ld, count;       // dst: [count, rows, ld] f16
  __half* dst;
  int32_t* sums;                       // a: row sums [count, rows]; b: column sums [count, cols]
};

__device__ __forceinline__ int64_t own_offset(const ShiftArgs& p, int64_t mat) {
  int64_t off = 0;
  for (int d = p.nb - 1; d >= 0; --d) {
    const int64_t i = mat % p.own_shape[d];
    mat /= p.own_shape[d];
    off += i * p.src_bstride[d];
  }
  return off;
}

// Loads are issued kBatch at a time before any is used: the f16 stores could
// alias the uint8 source as far as the compiler knows, so without this each
// 16-byte load would wait for the previous chunk's store (one DRAM round trip
// per chunk).
constexpr int kBatch = 4;

// Whether the 16 bytes of a row at column c0 can be read as one aligned vector.
__device__ __forceinline__ bool vec16_ok(const ShiftArgs& p, const uint8_t* srow, int64_t c0) {
  return p.src_cs == 1 && c0 + 16 <= p.cols && ((reinterpret_cast<uintptr_t>(srow + c0) & 15) == 0);
}

// x = the 16 bytes of u moved into [-128, 127] (int8 as is, uint8 minus 128).
__device__ __forceinline__ void decode16(const uint4& u, int is_signed, int (&x)[16]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b = (w[q] >> (8 * e)) & 0xFFu;
      x[4 * q + e] = is_signed ? (int)(int8_t)b : (int)b - 128;
    }
}

// The same for a piece that is not a full aligned vector (zeros beyond `cols`).
__device__ __forceinline__ void load16_scalar(const ShiftArgs& p, const uint8_t* srow, int64_t c0, int (&x)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    int v = 0;
    if (c0 + e < p.cols) {
      const uint8_t b = __ldg(srow + (c0 + e) * p.src_cs);
      v = p.is_signed ? (int)(int8_t)b : (int)b - 128;
    }
    x[e] = v;
  }
}

// Stores 16 f16 values at dst (16-byte aligned); the second half only if it
// starts inside the padded row (ld).
__device__ __forceinline__ void store16_f16(__half* dst, const int (&x)[16], int64_t c0, int64_t ld) {
  uint32_t w[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    __half2 h = __floats2half2_rn((float)x[2 * e], (float)x[2 * e + 1]);   // exact: |x| <= 128
    w[e] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  if (c0 + 8 < ld) d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// a: one warp converts one row (matrix `mat`, row r) and writes its exact sum.
__device__ __forceinline__ void shift_row(const ShiftArgs& p, int64_t wr, int lane) {
  const int64_t mat = wr / p.rows, r = wr - mat * p.rows;
  const uint8_t* srow = p.src + own_offset(p, mat) + r * p.src_rs;
  __half* drow = p.dst + wr * p.ld;
  uint32_t sum = 0;   // modulo 2^32, like every term of the int32 accumulator
  for (int64_t cb = (int64_t)lane * 16; cb < p.cols; cb += 512 * kBatch) {
    uint4 raw[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t c0 = cb + 512 * u;
      raw[u] = vec16_ok(p, srow, c0) ? __ldg(reinterpret_cast<const uint4*>(srow + c0)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t c0 = cb + 512 * u;
      if (c0 >= p.cols) break;
      int x[16];
      if (vec16_ok(p, srow, c0)) decode16(raw[u], p.is_signed, x);
      else load16_scalar(p, srow, c0, x);
#pragma unroll
      for (int e = 0; e < 16; ++e) sum += (uint32_t)x[e];
      store16_f16(drow + c0, x, c0, p.ld);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) p.sums[wr] = (int32_t)sum;
}

// b: one warp converts a strip of 256 columns (8 per lane) over a band of
// kStripRows rows, reading kBatch consecutive rows at a time (each load of the
// warp is 256 contiguous bytes of a row), and adds its partial column sums to
// the column sums (which start at zero) with one atomic add per column.
constexpr int kStripRows = 64;

// x = 8 bytes moved into [-128, 127]; zeros beyond `cols`.  Vector loads need
// a unit column stride and an 8-byte aligned, complete piece.
__device__ __forceinline__ bool vec8_ok(const ShiftArgs& p, const uint8_t* srow, int64_t c0) {
  return p.src_cs == 1 && c0 + 8 <= p.cols && ((reinterpret_cast<uintptr_t>(srow + c0) & 7) == 0);
}

__device__ __forceinline__ void decode8(const uint2& u, int is_signed, int (&x)[8]) {
  const uint32_t w[2] = {u.x, u.y};
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b = (w[q] >> (8 * e)) & 0xFFu;
      x[4 * q + e] = is_signed ? (int)(int8_t)b : (int)b - 128;
    }
}

__device__ __forceinline__ void shift_strip(const ShiftArgs& p, int64_t unit, int lane) {
  const int64_t strips = (p.cols + 255) / 256;
  const int64_t bands = (p.rows + kStripRows - 1) / kStripRows;
  const int64_t mat = unit / (strips * bands);
  const int64_t rest = unit - mat * strips * bands;
  const int64_t band = rest / strips, strip = rest - band * strips;
  const int64_t c0 = strip * 256 + (int64_t)lane * 8;
  if (c0 >= p.cols) return;
  const uint8_t* base = p.src + own_offset(p, mat);
  __half* dbase = p.dst + mat * p.rows * p.ld + c0;
  const int64_t r0 = band * kStripRows, r1 = min(p.rows, r0 + kStripRows);
  uint32_t part[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) part[e] = 0;
  for (int64_t rb = r0; rb < r1; rb += kBatch) {
    uint2 raw[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const uint8_t* srow = base + (rb + u) * p.src_rs;
      raw[u] = (rb + u < r1 && vec8_ok(p, srow, c0)) ? __ldg(reinterpret_cast<const uint2*>(srow + c0))
                                                     : make_uint2(0, 0);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t r = rb + u;
      if (r >= r1) break;
      const uint8_t* srow = base + r * p.src_rs;
      int x[8];
      if (vec8_ok(p, srow, c0)) {
        decode8(raw[u], p.is_signed, x);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          int v = 0;
          if (c0 + e < p.cols) {
            const uint8_t b = __ldg(srow + (c0 + e) * p.src_cs);
            v = p.is_signed ? (int)(int8_t)b : (int)b - 128;
          }
          x[e] = v;
        }
      }
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        part[2 * e] += (uint32_t)x[2 * e];
        part[2 * e + 1] += (uint32_t)x[2 * e + 1];
        __half2 h = __floats2half2_rn((float)x[2 * e], (float)x[2 * e + 1]);   // exact: |x| <= 128
        w[e] = *reinterpret_cast<uint32_t*>(&h);
      }
      // 8 columns from c0 < cols end within the row padded to ld = round8(cols)
      *reinterpret_cast<uint4*>(dbase + r * p.ld) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  unsigned* sums = reinterpret_cast<unsigned*>(p.sums) + mat * p.cols;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (c0 + e < p.cols) atomicAdd(sums + c0 + e, part[e]);
}

// Both operands in one launch, one warp per unit: units [0, b_units) are b's
// column strips (the larger units, taken first), the rest a's rows.  One
// launch lets b's work fill the gaps of a's and leaves no second, partly
// filled last wave.  Four blocks per SM cap a thread at 64 registers (no
// spills); unbounded, the strip path took 153.
__global__ void __launch_bounds__(256, 4) shift_kernel(const ShiftArgs pa, const ShiftArgs pb, const int64_t b_units) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t total = b_units + pa.count * pa.rows;
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < total; u += warps) {
    if (u < b_units) shift_strip(pb, u, lane);
    else shift_row(pa, u - b_units, lane);
  }
}

struct QLayout {
  int64_t a_count, b_count, kp, np;
  size_t a_bytes, b_bytes, rs_bytes, cs_bytes;
};

QLayout qlayout(int64_t M, int64_t N, int64_t K, int64_t a_count, int64_t b_count) {
  QLayout l;
  l.a_count = a_count;
  l.b_count = b_count;
  l.kp = round_up(K, 8);
  l.np = round_up(N, 8);
  l.a_bytes = (size_t)round_up(a_count * M * l.kp * 2, kAlign);
  l.b_bytes = (size_t)round_up(b_count * K * l.np * 2, kAlign);
  l.rs_bytes = (size_t)round_up(a_count * M * 4, kAlign);
  l.cs_bytes = (size_t)round_up(b_count * N * 4, kAlign);
  return l;
}

int64_t own_count(const int64_t* shape) {
  int64_t n = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) n *= shape[d];
  return n;
}

// Element strides, over the broadcast batch, of a dense [own batch..., rows, ld]
// copy of an operand whose own batch shape is `own` (0 where broadcast).
void dense_batch_strides(const BatchMap& bm, const int64_t* own, int64_t matrix_elems, int64_t* out) {
  int64_t acc = matrix_elems;
  for (int d = kMaxBatchDims - 1; d >= 0; --d) {
    out[d] = (d < bm.nb && own[d] > 1) ? acc : 0;
    if (d < bm.nb) acc *= own[d];
  }
}

bool plan_qlinear(const QLinearArgs& q, const QLayout& l, void* ws, bool pair, OperandPlan* a, OperandPlan* b) {
  if (q.M < 2 || q.N < 2 || q.K < 1) return false;
  if (q.M > 0x7fffffffLL || q.N > 0x7fffffffLL || q.K > 0x7fffffffLL) return false;
  if (q.y.cs != 1) return false;
  // Tensor maps are only encoded once the workspace address is known; before
  // that a 256-aligned stand-in address checks the layout rules.
  char* base = ws ? static_cast<char*>(ws) : reinterpret_cast<char*>(kAlign);
  int64_t abs_[kMaxBatchDims], bbs[kMaxBatchDims];
  dense_batch_strides(q.bm, q.a_bshape, q.M * l.kp, abs_);
  dense_batch_strides(q.bm, q.b_bshape, q.K * l.np, bbs);
  if (!plan_operand(base, MM_F16, q.M, q.K, l.kp, 1, q.bm, abs_, kTileM, a)) return false;
  if (!plan_operand(base + l.a_bytes, MM_F16, q.N, q.K, 1, l.np, q.bm, bbs, pair ? kTileN / 2 : kTileN, b))
    return false;
  return true;
}

}  // namespace

size_t tc_qlinear_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t a_count, int64_t b_count) {
  const QLayout l = qlayout(M, N, K, a_count, b_count);
  return l.a_bytes + l.b_bytes + l.rs_bytes + l.cs_bytes;
}

bool tc_qlinear_supported(const QLinearArgs& q) {
  const QLayout l = qlayout(q.M, q.N, q.K, own_count(q.a_bshape), own_count(q.b_bshape));
  OperandPlan a, b;
  return plan_qlinear(q, l, nullptr, false, &a, &b);
}

mm_status launch_tc_qlinear(const QLinearArgs& q, void* ws, unsigned* status, cudaStream_t stream) {
  const QLayout l = qlayout(q.M, q.N, q.K, own_count(q.a_bshape), own_count(q.b_bshape));
  OperandPlan a, b;
  if (!ws || !status || !plan_qlinear(q, l, ws, false, &a, &b)) return MM_ERR_UNSUPPORTED;
  char* base = static_cast<char*>(ws);
  __half* a16 = reinterpret_cast<__half*>(base);
  __half* b16 = reinterpret_cast<__half*>(base + l.a_bytes);
  int32_t* rs = reinterpret_cast<int32_t*>(base + l.a_bytes + l.b_bytes);
  int32_t* cs = reinterpret_cast<int32_t*>(base + l.a_bytes + l.b_bytes + l.rs_bytes);

  // 1. a' = a - c_a with row sums, b' = b - c_b with column sums, as exact f16.
  ShiftArgs sa;
  memset(&sa, 0, sizeof(sa));
  sa.src = static_cast<const uint8_t*>(q.a.ptr); sa.is_signed = q.a_signed; sa.nb = q.bm.nb;
  sa.src_rs = q.a.rs; sa.src_cs = q.a.cs;
  sa.rows = q.M; sa.cols = q.K; sa.ld = l.kp; sa.count = l.a_count; sa.dst = a16; sa.sums = rs;
  ShiftArgs sb = sa;
  sb.src = static_cast<const uint8_t*>(q.b.ptr); sb.is_signed = q.b_signed;
  sb.src_rs = q.b.rs; sb.src_cs = q.b.cs;
  sb.rows = q.K; sb.cols = q.N; sb.ld = l.np; sb.count = l.b_count; sb.dst = b16; sb.sums = cs;
  for (int d = 0; d < kMaxBatchDims; ++d) {
    sa.own_shape[d] = d < q.bm.nb ? q.a_bshape[d] : 1;
    sa.src_bstride[d] = q.a.bstride[d];
    sb.own_shape[d] = d < q.bm.nb ? q.b_bshape[d] : 1;
    sb.src_bstride[d] = q.b.bstride[d];
  }
  if (cudaMemsetAsync(cs, 0, (size_t)(l.b_count * q.N * 4), stream) != cudaSuccess) return MM_ERR_CUDA;
  const int64_t b_units = l.b_count * ((q.N + 255) / 256) * ((q.K + kStripRows - 1) / kStripRows);
  const int64_t blocks = (b_units + l.a_count * q.M + 7) / 8;
  launch_pdl(shift_kernel, dim3((unsigned)(blocks < 8 * 152 * 8 ? blocks : 8 * 152 * 8)), dim3(256), 0, stream, sa, sb,
             b_units);
  if (cudaGetLastError() != cudaSuccess) return MM_ERR_CUDA;

  // 2. The f16 GEMM with 1024-deep exact segments and the zero-point-correcting,
  //    requantising epilogue.
  TcParams p;
  init_params(&p);
  p.M = q.M; p.N = q.N; p.K = q.K;
  p.bm = q.bm;
  p.kb_per_seg = 1024 / kTileK;
  p.y = const_cast<void*>(q.y.ptr);
  for (int d = 0; d < kMaxBatchDims; ++d) p.y_bstride[d] = q.y.bstride[d];
  p.y_rs = q.y.rs;
  p.y_vec = (reinterpret_cast<uintptr_t>(q.y.ptr) % 16 == 0) && (q.y.rs % 16 == 0);
  for (int d = 0; d < q.bm.nb; ++d) p.y_vec = p.y_vec && (q.y.bstride[d] % 16 == 0);
  p.sa = q.sa; p.sb = q.sb; p.za = q.za; p.zb = q.zb; p.ys = q.ys; p.yz = q.yz;
  p.sa_f16 = q.sa_f16; p.sb_f16 = q.sb_f16; p.ys_f16 = q.ys_f16; p.y_signed = q.y_signed;
  p.a_signed = q.a_signed; p.b_signed = q.b_signed;
  p.q_rs = rs; p.q_cs = cs;
  p.status = status;
  // Single CTAs: this product is bound by its epilogue (exact int32 segment
  // sums and requantisation), which CTA pairs do not shorten.
  p.idesc = make_idesc(1, a.mn_major, b.mn_major, false);
  return launch_tc(kQLinear, false, a, b, p, stream);
}

// ------------------------------------------------------------------ GroupedMatMul: routing

namespace {

struct GLayout {
  int64_t kp;
  size_t off_count, off_cursor, off_offset, off_tiles, off_rowlist, off_x, total;
};

GLayout glayout(int64_t M, int64_t S, int64_t G, int64_t K, int elem) {
  GLayout l;
  l.kp = round_up(K, 8);
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o = (size_t)round_up((int64_t)(o + bytes), kAlign); return at; };
  l.off_count = take((size_t)G * 4);
  l.off_cursor = take((size_t)G * 4);
  l.off_offset = take((size_t)(G + 1) * 4);
  l.off_tiles = take((size_t)(G + 1) * 4);
  l.off_rowlist = take((size_t)(M * S) * 4);
  l.off_x = take((size_t)(M * S) * (size_t)l.kp * (size_t)elem);
  l.total = o;
  return l;
}

__device__ __forceinline__ int64_t load_index(const void* gi, int64_t off, int ind64) {
  return ind64 ? static_cast<const int64_t*>(gi)[off] : (int64_t) static_cast<const int32_t*>(gi)[off];
}

// Up to kHistGroups groups are counted in a shared-memory histogram per block
// (lanes of a warp that pick the same group add once, by popcount), then added
// to the global counts; more groups count with global atomics directly.
constexpr int kHistGroups = 4096;

__global__ void __launch_bounds__(256) route_count_kernel(const void* gi, int ind64, int64_t gi_ms, int64_t gi_ss,
                                                          int64_t M, int64_t S, int64_t G, int32_t* count,
                                                          unsigned* status) {
  pdl_wait();
  __shared__ int32_t hist[kHistGroups];
  const int64_t total = M * S;
  const bool shared_hist = G <= kHistGroups;
  if (shared_hist) {
    for (int g = threadIdx.x; g < G; g += blockDim.x) hist[g] = 0;
    __syncthreads();
  }
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // Every lane of a warp runs the same number of iterations (the loop bound is
  // rounded up to whole warps), so the warp-wide match below is well defined.
  const int64_t total_w = (total + 31) / 32 * 32;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total_w; e += stride) {
    int64_t g = -1;
    bool valid = false;
    if (e < total) {
      const int64_t m = e / S, i = e - m * S;
      g = load_index(gi, m * gi_ms + i * gi_ss, ind64);
      valid = g >= 0 && g < G;
      if (!valid) atomicOr(status, kStatusIndexRange);
    }
    if (shared_hist) {
      const int key = valid ? (int)g : -1;
      const unsigned same = __match_any_sync(0xffffffffu, key);
      if (valid && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(hist + key, __popc(same));
    } else if (valid) {
      atomicAdd(count + g, 1);
    }
  }
  if (shared_hist) {
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += blockDim.x)
      if (hist[g]) atomicAdd(count + g, hist[g]);
  }
}

// Inclusive sum of v over the threads of the block, in thread order (warp
// shuffles, then one warp over the per-warp totals); `part` holds 32 values.
__device__ __forceinline__ int64_t block_inclusive_sum(int64_t v, int64_t* part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) part[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < (int)(blockDim.x >> 5) ? part[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    part[lane] = w;
  }
  __syncthreads();
  const int64_t r = v + (warp > 0 ? part[warp - 1] : 0);
  __syncthreads();   // part may be reused by the caller
  return r;
}

// One block: offset[g] = sum_{h<g} count[h]; tile_start[g] = sum_{h<g} ceil(count[h]/tile_rows) * nt.
__global__ void __launch_bounds__(1024) route_scan_kernel(const int32_t* count, int64_t G, int64_t nt,
                                                          int tile_rows, int32_t* offset, int32_t* tile_start) {
  pdl_wait();
  __shared__ int64_t part[32];
  const int t = threadIdx.x, T = blockDim.x;
  const int64_t per = (G + T - 1) / T;
  const int64_t lo = min(G, (int64_t)t * per), hi = min(G, lo + per);
  int64_t rows = 0, tiles = 0;
  for (int64_t g = lo; g < hi; ++g) {
    rows += count[g];
    tiles += (count[g] + tile_rows - 1) / tile_rows * nt;
  }
  // Exclusive prefix of this thread's range.
  rows = block_inclusive_sum(rows, part) - rows;
  tiles = block_inclusive_sum(tiles, part) - tiles;
  for (int64_t g = lo; g < hi; ++g) {
    offset[g] = (int32_t)rows;
    tile_start[g] = (int32_t)tiles;
    rows += count[g];
    tiles += (count[g] + tile_rows - 1) / tile_rows * nt;
  }
  if (hi == G && lo < hi) {
    offset[G] = (int32_t)rows;
    tile_start[G] = (int32_t)tiles;
  }
  if (G == 0 && t == 0) {
    offset[0] = 0;
    tile_start[0] = 0;
  }
}

// One block per routed row (m, i): claim a slot in the group's row range,
// record the output row, copy input[m] into the group-ordered buffer.  Rows
// with an invalid index are written as zeros instead (never reading weights).
template <typename T>
__global__ void __launch_bounds__(128) route_scatter_kernel(const GroupedArgs g, const int32_t* offset,
                                                            int32_t* cursor, int32_t* rowlist, T* xperm,
                                                            int64_t kp) {
  pdl_wait();
  __shared__ int64_t s_pos;
  const int64_t total = g.M * g.S;
  const T* X = static_cast<const T*>(g.x);
  T* Out = static_cast<T*>(g.out);
  for (int64_t e = blockIdx.x; e < total; e += gridDim.x) {
    const int64_t m = e / g.S, i = e - m * g.S;
    const int64_t grp = load_index(g.gi, m * g.gi_ms + i * g.gi_ss, g.ind64);
    __syncthreads();
    if (threadIdx.x == 0) s_pos = (grp >= 0 && grp < g.G) ? (int64_t)offset[grp] + atomicAdd(cursor + grp, 1) : -1;
    __syncthreads();
    const int64_t pos = s_pos;
    if (pos < 0) {
      for (int64_t n = threadIdx.x; n < g.N; n += blockDim.x) Out[e * g.N + n] = T(0.f);
      continue;
    }
    if (threadIdx.x == 0) rowlist[pos] = (int32_t)e;
    const T* src = X + m * g.x_rs;
    T* dst = xperm + pos * kp;
    const bool vec = g.x_cs == 1 && ((reinterpret_cast<uintptr_t>(src) & 15) == 0) && (g.K % 8 == 0);
    if (vec) {
      for (int64_t k = threadIdx.x * 8; k < g.K; k += blockDim.x * 8)
        *reinterpret_cast<uint4*>(dst + k) = *reinterpret_cast<const uint4*>(src + k);
    } else {
      for (int64_t k = threadIdx.x; k < g.K; k += blockDim.x) dst[k] = src[k * g.x_cs];
    }
  }
}

bool plan_grouped_b(const GroupedArgs& g, bool pair, OperandPlan* b) {
  BatchMap bm;
  memset(&bm, 0, sizeof(bm));
  bm.nb = 1;
  bm.shape[0] = g.G;
  bm.count = g.G;
  for (int d = 1; d < kMaxBatchDims; ++d) bm.shape[d] = 1;
  int64_t bs[kMaxBatchDims] = {g.w_gs, 0, 0, 0, 0, 0};
  if (!plan_operand(g.w, g.dtype, g.N, g.K, g.w_ns, g.w_ks, bm, bs, pair ? kTileN / 2 : kTileN, b)) return false;
  // Tile coordinates address weights[g] directly as batch coordinate g.
  return g.G <= 1 || b->bc[0] == 1;
}

// Byte stride of a dimension of extent `count` for a plain tensor map: the
// given stride, or (a dimension of extent 1 is never stepped) any valid one.
int64_t map_stride(int64_t stride_bytes, int64_t count, int64_t fallback) {
  return count == 1 ? (fallback + 15) / 16 * 16 : stride_bytes;
}

// Weight-only quantized experts: the weights (boxes of 128 columns x 64 k)
// and the scale and zero-point rows (boxes of 128 columns x 1 row) as plain
// tensor maps indexed (n, k or k-block, g).  The maps of 4-bit weights and
// zero points address bytes (two columns each): boxes of 64 bytes.
bool plan_grouped_q(const GroupedArgs& g, OperandPlan* b, OperandPlan* sm, OperandPlan* zm) {
  if (g.wq == 0 || g.w_ns != 1 || g.wsc_ns != 1 || (g.wzp && g.wzp_ns != 1)) return false;
  if (!(g.qblock >= g.K || g.qblock % kTileK == 0)) return false;
  const int64_t kb = (g.K + g.qblock - 1) / g.qblock;
  const int64_t per = g.wq >= 3 ? 2 : 1;   // elements per byte
  const int64_t nb = g.N / per;             // bytes per row (N is even for 4-bit)
  const int box = 128 / (int)per;
  if (!plan_plain_3d(g.w, 1, nb, g.K, g.G, map_stride(g.w_ks / per, g.K, nb),
                     map_stride(g.w_gs / per, g.G, g.w_ks / per * g.K), box, 64, b))
    return false;
  const int64_t sbs = map_stride(g.wsc_bs * 2, kb, g.N * 2);
  if (!plan_plain_3d(g.wsc, 2, g.N, kb, g.G, sbs, map_stride(g.wsc_gs * 2, g.G, sbs * kb), 128, 1, sm)) return false;
  if (g.wzp) {
    const int64_t zbs = map_stride(g.wzp_bs / per, kb, nb);
    if (!plan_plain_3d(g.wzp, 1, nb, kb, g.G, zbs, map_stride(g.wzp_gs / per, g.G, zbs * kb), box, 1, zm)) return false;
  }
  return true;
}

}  // namespace

size_t tc_grouped_workspace_bytes(const GroupedArgs& g) {
  return glayout(g.M, g.S, g.G, g.K, g.dtype == MM_F64 ? 8 : g.dtype == MM_F32 ? 4 : 2).total;
}

bool tc_grouped_supported(const GroupedArgs& g) {
  if (g.dtype != MM_BF16 && g.dtype != MM_F16) return false;
  if (g.N < 8 || g.K < 1 || g.G < 1) return false;
  if (g.M * g.S > 0x7fffffffLL || g.G > 0x7fffffffLL || g.N > 0x7fffffffLL || g.K > 0x7fffffffLL) return false;
  // an upper bound on the tile count must fit the int32 tile table
  const int64_t nt = (g.N + kTileN - 1) / kTileN;
  if ((g.M * g.S / kTileM + g.G + 1) * nt > 0x7fffffffLL) return false;
  OperandPlan b, sm, zm;
  if (g.wq) return plan_grouped_q(g, &b, &sm, &zm) && grouped_q_pairs_available();
  return plan_grouped_b(g, false, &b);
}

mm_status launch_tc_grouped(const GroupedArgs& g, void* ws, unsigned* status, cudaStream_t stream) {
  OperandPlan a, b, sm, zm;
  // CTA pairs (256-row tiles) when groups are large enough, and always for
  // quantized weights; the routing scan counts tiles of the same height.
  const bool pair = g.wq ? true : use_grouped_pair(g.M * g.S, g.G, g.K);
  if (!ws || !status) return MM_ERR_UNSUPPORTED;
  if (g.wq ? !plan_grouped_q(g, &b, &sm, &zm) : !plan_grouped_b(g, pair, &b)) return MM_ERR_UNSUPPORTED;
  const GLayout l = glayout(g.M, g.S, g.G, g.K, 2);
  char* base = static_cast<char*>(ws);
  int32_t* count = reinterpret_cast<int32_t*>(base + l.off_count);
  int32_t* cursor = reinterpret_cast<int32_t*>(base + l.off_cursor);
  int32_t* offset = reinterpret_cast<int32_t*>(base + l.off_offset);
  int32_t* tile_start = reinterpret_cast<int32_t*>(base + l.off_tiles);
  int32_t* rowlist = reinterpret_cast<int32_t*>(base + l.off_rowlist);
  void* xperm = base + l.off_x;
  const int64_t rows = g.M * g.S;
  const int64_t nt = (g.N + kTileN - 1) / kTileN;

  BatchMap bm1;
  memset(&bm1, 0, sizeof(bm1));
  bm1.nb = 0;
  bm1.count = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) bm1.shape[d] = 1;
  int64_t zero[kMaxBatchDims] = {0, 0, 0, 0, 0, 0};
  if (!plan_operand(xperm, g.dtype, rows, g.K, l.kp, 1, bm1, zero, kTileM, &a)) return MM_ERR_UNSUPPORTED;
  // Pairs run each group's last row tile, when it has at most 128 rows, as
  // one M = 128 MMA fed by 64 rows of A per CTA (a 64-row box of the same rows).
  OperandPlan a_tail;
  const bool tail = pair && !g.wq && plan_operand(xperm, g.dtype, rows, g.K, l.kp, 1, bm1, zero, kTileM / 2, &a_tail);

  if (cudaMemsetAsync(count, 0, l.off_offset - l.off_count, stream) != cudaSuccess) return MM_ERR_CUDA;
  const int64_t cb = (rows + 255) / 256;
  launch_pdl(route_count_kernel, dim3((unsigned)(cb < 4096 ? cb : 4096)), dim3(256), 0, stream, g.gi, g.ind64, g.gi_ms,
             g.gi_ss, g.M, g.S, g.G, count, status);
  launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, stream, (const int32_t*)count, g.G, nt,
             pair ? 2 * kTileM : kTileM, offset, tile_start);
  const unsigned sgrid = (unsigned)(rows < 65536 ? rows : 65536);
  if (g.dtype == MM_BF16)
    launch_pdl(route_scatter_kernel<__nv_bfloat16>, dim3(sgrid), dim3(128), 0, stream, g, (const int32_t*)offset,
               cursor, rowlist, static_cast<__nv_bfloat16*>(xperm), l.kp);
  else
    launch_pdl(route_scatter_kernel<__half>, dim3(sgrid), dim3(128), 0, stream, g, (const int32_t*)offset, cursor,
               rowlist, static_cast<__half*>(xperm), l.kp);
  if (cudaGetLastError() != cudaSuccess) return MM_ERR_CUDA;

  TcParams p;
  init_params(&p);
  p.M = rows; p.N = g.N; p.K = g.K;
  p.nt = nt;
  p.idesc = make_idesc(g.dtype == MM_F16, a.mn_major, b.mn_major, pair);
  if (tail) {
    p.pair_tail = 1;
    p.idesc_tail = make_idesc_rows(g.dtype == MM_F16, a.mn_major, b.mn_major, kTileM);
  }
  if (g.wq) {
    p.w_signed = g.wq == 1 || g.wq == 3;
    p.w4 = g.wq >= 3;
    p.wzp_present = g.wzp != nullptr;
    p.kb_per_q = g.qblock >= g.K ? (1 << 30) : (int)(g.qblock / kTileK);
  }
  p.out_f16 = g.dtype == MM_F16;
  p.y = g.out;
  p.y_rs = g.N;
  p.y_vec = (reinterpret_cast<uintptr_t>(g.out) % 16 == 0) && (g.N % 8 == 0);
  if (g.bias) {
    p.c = g.bias;
    p.beta = 1.f;
    p.c_gs = g.bias_gs;
    p.c_cs = g.bias_ns;
    p.c_vec = g.bias_ns == 1 && (reinterpret_cast<uintptr_t>(g.bias) % 16 == 0) && (g.bias_gs % 8 == 0);
  }
  p.g_count = count; p.g_offset = offset; p.g_tile_start = tile_start; p.g_rowlist = rowlist;
  p.G = (int)g.G;
  p.status = status;
  // The tile count is known only on the device: one persistent CTA (pair) per SM (pair).
  if (g.wq) return launch_tc(kGroupedQ, true, a, b, p, stream, &sm, g.wzp ? &zm : nullptr);
  return launch_tc(kGrouped, pair, a, b, p, stream, tail ? &a_tail : nullptr);
}

}  // namespace qg
