// CUDA-core kernels: every element type and every stride pattern.
//
// These run the types that have no tensor-core path on GB300 (f32 via FFMA --
// never TF32 --, f64, and the 32/64-bit integer types, which wrap modulo 2^n),
// and any bf16/f16 or 8-bit call whose layout the tensor-core kernels do not
// take.  A block computes a 64 x 64 output tile with 256 threads (4 x 4
// outputs each, strided by 16 so shared-memory reads are conflict-free and
// global stores are coalesced along the row); K is staged through shared
// memory 16 at a time with plain strided loads.
//
// Products with 1 to 4 rows of A' (bf16, f16, f32) have their own kernels,
// which read B' once at memory speed: vec_gemm_kernel for K-major B' and
// vec_mn_kernel for MN-major B' (see "few-row products" below).
#include <atomic>
#include <cstring>

#include <cooperative_groups.h>

#include "kernels.h"

namespace qg {
namespace {

namespace cg = cooperative_groups;

constexpr int kTile = 64;
constexpr int kTk = 16;
constexpr int kThreads = 256;

template <typename T> struct Arith;
template <> struct Arith<__nv_bfloat16> {
  using acc = float;
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ __nv_bfloat16 store(float v) { return __float2bfloat16_rn(v); }
};
template <> struct Arith<__half> {
  using acc = float;
  static __device__ __forceinline__ float load(const __half* p) { return __half2float(*p); }
  static __device__ __forceinline__ __half store(float v) { return __float2half_rn(v); }
};
template <> struct Arith<float> {
  using acc = float;
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ float store(float v) { return v; }
};
template <> struct Arith<double> {
  using acc = double;
  static __device__ __forceinline__ double load(const double* p) { return *p; }
  static __device__ __forceinline__ double store(double v) { return v; }
};
// Integers accumulate in the unsigned type of the same width: wrap-around
// modulo 2^n is then well defined and equals numpy's result.
template <> struct Arith<int32_t> {
  using acc = uint32_t;
  static __device__ __forceinline__ uint32_t load(const int32_t* p) { return (uint32_t)*p; }
  static __device__ __forceinline__ int32_t store(uint32_t v) { return (int32_t)v; }
};
template <> struct Arith<uint32_t> {
  using acc = uint32_t;
  static __device__ __forceinline__ uint32_t load(const uint32_t* p) { return *p; }
  static __device__ __forceinline__ uint32_t store(uint32_t v) { return v; }
};
template <> struct Arith<int64_t> {
  using acc = uint64_t;
  static __device__ __forceinline__ uint64_t load(const int64_t* p) { return (uint64_t)*p; }
  static __device__ __forceinline__ int64_t store(uint64_t v) { return (int64_t)v; }
};
template <> struct Arith<uint64_t> {
  using acc = uint64_t;
  static __device__ __forceinline__ uint64_t load(const uint64_t* p) { return *p; }
  static __device__ __forceinline__ uint64_t store(uint64_t v) { return v; }
};

template <typename A> __device__ __forceinline__ A mac(A acc, A x, A y) { return acc + x * y; }
template <> __device__ __forceinline__ float mac<float>(float acc, float x, float y) { return __fmaf_rn(x, y, acc); }
template <> __device__ __forceinline__ double mac<double>(double acc, double x, double y) { return __fma_rn(x, y, acc); }

// y = alpha*acc + beta*c in the accumulator type.
template <typename T> struct Epi {
  using acc = typename Arith<T>::acc;
  static __device__ __forceinline__ acc apply(const GemmArgs& p, acc v, const T* c) {
    acc r = (acc)p.alpha * v;
    if (c) r = __fmaf_rn(p.beta, Arith<T>::load(c), r);
    return r;
  }
};
template <> struct Epi<double> {
  static __device__ __forceinline__ double apply(const GemmArgs& p, double v, const double* c) {
    double r = p.alpha_d * v;
    if (c) r = __fma_rn(p.beta_d, *c, r);
    return r;
  }
};
// Integer T.  Integral alpha and beta: exact modulo 2^n.  Otherwise (a reading
// of the Gemm page, which leaves this open): the accumulator taken as a T value
// and C widened to fp64, r = (alpha*acc) + (beta*c) with each product and the
// sum rounded once in fp64, then truncated toward zero; the hardware's
// round-toward-zero conversions saturate values outside T's range.
template <typename T> __device__ __forceinline__ double int_to_f64(T x);
template <> __device__ __forceinline__ double int_to_f64<int32_t>(int32_t x) { return (double)x; }
template <> __device__ __forceinline__ double int_to_f64<uint32_t>(uint32_t x) { return (double)x; }
template <> __device__ __forceinline__ double int_to_f64<int64_t>(int64_t x) { return __ll2double_rn(x); }
template <> __device__ __forceinline__ double int_to_f64<uint64_t>(uint64_t x) { return __ull2double_rn(x); }
template <typename T> __device__ __forceinline__ T f64_to_int_rz(double x);
template <> __device__ __forceinline__ int32_t f64_to_int_rz<int32_t>(double x) { return __double2int_rz(x); }
template <> __device__ __forceinline__ uint32_t f64_to_int_rz<uint32_t>(double x) { return __double2uint_rz(x); }
template <> __device__ __forceinline__ int64_t f64_to_int_rz<int64_t>(double x) { return __double2ll_rz(x); }
template <> __device__ __forceinline__ uint64_t f64_to_int_rz<uint64_t>(double x) { return __double2ull_rz(x); }

template <typename T, typename U> struct EpiInt {
  static __device__ __forceinline__ U apply(const GemmArgs& p, U v, const T* c) {
    if (p.int_float) {
      double r = __dmul_rn(p.alpha_d, int_to_f64<T>((T)v));
      if (c) r = __dadd_rn(r, __dmul_rn(p.beta_d, int_to_f64<T>(*c)));
      return (U)f64_to_int_rz<T>(r);
    }
    U r = (U)p.alpha_i * v;
    if (c) r += (U)p.beta_i * Arith<T>::load(c);
    return r;
  }
};
template <> struct Epi<int32_t> : EpiInt<int32_t, uint32_t> {};
template <> struct Epi<uint32_t> : EpiInt<uint32_t, uint32_t> {};
template <> struct Epi<int64_t> : EpiInt<int64_t, uint64_t> {};
template <> struct Epi<uint64_t> : EpiInt<uint64_t, uint64_t> {};

// ------------------------------------------------------------------ tiled CUDA-core GEMM

// A block of 256 threads (16 x 16) computes a (16*TM) x (16*TN) output tile,
// TM x TN outputs per thread.  A thread's rows are ty*RM + i in each of the
// tile's TM/RM row bands (RM = 16 bytes of accumulators), and likewise its
// columns, so that each step over k reads its A and B values from shared
// memory as 16-byte vectors (conflict-free: the 16 threads of a half-warp read
// 256 consecutive bytes of B, the two halves the same words of A) and the
// output rows are written 16 bytes per thread, 256 bytes per half-warp.
//
// K goes through shared memory in slabs of KS, double-buffered: the global
// loads of slab s+1 are issued before slab s is multiplied, so a small product
// pays the memory latency about once instead of once per slab.  An operand
// that is contiguous along one of its dimensions, with 16-byte aligned rows and
// batches, is read 16 bytes per thread (along k, or along m / n); any other
// layout element by element with its strides.
// Slab depth: 16 for the 8 x 8 tiles, deeper for the small tiles (every
// thread still loads 8 32-bit or 4 64-bit values a slab), so that a small
// product (K = 64 for 2 x 2 tiles) is a single slab: one memory latency.
template <int TM, int ACC_BYTES>
constexpr int slab_depth() { return TM >= 8 ? 16 : TM == 4 ? (ACC_BYTES == 8 ? 16 : 32) : (ACC_BYTES == 8 ? 32 : 64); }

enum SimtLoad { kLoadScalar = 0, kLoadVecK = 1, kLoadVecMN = 2 };

// One operand of the tile as the kernel reads it: R "rows" (m of A, n of B),
// row stride rs and k stride ks (elements), the load mode, and for the
// element-by-element mode whether consecutive threads go along k (k is the
// smaller stride) or along the rows.
struct SimtOperand {
  int mode, along_k;
};

template <typename T, int R, int kSlab>
struct SlabLoad {
  using Acc = typename Arith<T>::acc;
  static constexpr int V = 16 / (int)sizeof(T);               // elements per 16-byte vector
  static constexpr int NE = R * kSlab / kThreads;              // elements per thread (scalar mode)
  static constexpr int NV = R * kSlab / V;                     // vectors per slab
  static constexpr int NVT = (NV + kThreads - 1) / kThreads;   // vectors per thread
  static_assert(NE * sizeof(T) <= NVT * 16, "scalar-mode elements fit the vector registers");
  // The loaded values as stored in memory: NVT vectors, or (scalar mode) NE
  // elements packed in the same registers; converted when written to shared memory.
  uint4 v[NVT];

  // Global -> registers for the slab at k0 of the operand at `base` (rows r0..).
  __device__ __forceinline__ void load(const T* base, int64_t rs, int64_t ks, int64_t r0, int64_t rows, int64_t k0,
                                       int64_t K, SimtOperand op, int tid) {
    if (op.mode == kLoadScalar) {
#pragma unroll
      for (int u = 0; u < NE; ++u) {
        const int idx = tid + u * kThreads;
        const int r = op.along_k ? idx / kSlab : idx % R, k = op.along_k ? idx % kSlab : idx / R;
        const int64_t gr = r0 + r, gk = k0 + k;
        reinterpret_cast<T*>(v)[u] = (gr < rows && gk < K) ? base[gr * rs + gk * ks] : T(0);
      }
      return;
    }
#pragma unroll
    for (int u = 0; u < NVT; ++u) {
      const int idx = tid + u * kThreads;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (idx >= NV) continue;
      int64_t gr, gk;
      bool full;
      if (op.mode == kLoadVecK) {
        gr = r0 + idx / (kSlab / V);
        gk = k0 + (int64_t)(idx % (kSlab / V)) * V;
        full = gr < rows && gk + V <= K;
        if (!full && gr < rows) {        // the k tail: element by element
          T* t = reinterpret_cast<T*>(&v[u]);
          for (int c = 0; c < V; ++c)
            if (gk + c < K) t[c] = base[gr * rs + (gk + c) * ks];
        }
      } else {
        gk = k0 + idx / (R / V);
        gr = r0 + (int64_t)(idx % (R / V)) * V;
        full = gk < K && gr + V <= rows;
        if (!full && gk < K) {           // the row tail
          T* t = reinterpret_cast<T*>(&v[u]);
          for (int c = 0; c < V; ++c)
            if (gr + c < rows) t[c] = base[(gr + c) * rs + gk * ks];
        }
      }
      if (full) v[u] = __ldg(reinterpret_cast<const uint4*>(base + gr * rs + gk * ks));
    }
  }

  // Registers -> shared memory slab S[k][r] (row pitch P).
  template <int P>
  __device__ __forceinline__ void store(Acc (*S)[P], SimtOperand op, int tid) const {
    if (op.mode == kLoadScalar) {
#pragma unroll
      for (int u = 0; u < NE; ++u) {
        const int idx = tid + u * kThreads;
        const int r = op.along_k ? idx / kSlab : idx % R, k = op.along_k ? idx % kSlab : idx / R;
        S[k][r] = Arith<T>::load(reinterpret_cast<const T*>(v) + u);
      }
      return;
    }
#pragma unroll
    for (int u = 0; u < NVT; ++u) {
      const int idx = tid + u * kThreads;
      if (idx >= NV) continue;
      const T* t = reinterpret_cast<const T*>(&v[u]);
      if (op.mode == kLoadVecK) {
        const int r = idx / (kSlab / V), k = (idx % (kSlab / V)) * V;
#pragma unroll
        for (int c = 0; c < V; ++c) S[k + c][r] = Arith<T>::load(t + c);
      } else {
        const int k = idx / (R / V), r = (idx % (R / V)) * V;
#pragma unroll
        for (int c = 0; c < V; ++c) S[k][r + c] = Arith<T>::load(t + c);
      }
    }
  }
};

// RM consecutive accumulators from shared memory (RM * sizeof(Acc) = 16 bytes,
// or fewer for small tiles).
template <typename Acc, int RM>
__device__ __forceinline__ void lds_vec(const Acc* src, Acc (&dst)[RM]) {
  if constexpr (RM * sizeof(Acc) == 16) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    memcpy(dst, &u, 16);
  } else if constexpr (RM * sizeof(Acc) == 8) {
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    memcpy(dst, &u, 8);
  } else {
#pragma unroll
    for (int i = 0; i < RM; ++i) dst[i] = src[i];
  }
}

// Two blocks per SM (at most 128 registers a thread) except for the 8 x 8
// tiles, whose 64 accumulators would then spill.
template <typename T, int TM, int TN>
__global__ void __launch_bounds__(kThreads, TM == 8 ? 1 : 2)
    simt_gemm_kernel(const GemmArgs p, SimtOperand opa, SimtOperand opb) {
  pdl_begin();
  using Acc = typename Arith<T>::acc;
  constexpr int RM = (16 / (int)sizeof(Acc)) < TM ? 16 / (int)sizeof(Acc) : TM;   // rows per band
  constexpr int RN = (16 / (int)sizeof(Acc)) < TN ? 16 / (int)sizeof(Acc) : TN;
  constexpr int BMt = 16 * TM, BNt = 16 * TN;
  constexpr int PA = BMt + 16 / (int)sizeof(Acc), PB = BNt + 16 / (int)sizeof(Acc);   // padded row pitch
  constexpr int kSlab = slab_depth<TM, (int)sizeof(Acc)>();
  __shared__ __align__(16) Acc As[2][kSlab][PA];
  __shared__ __align__(16) Acc Bs[2][kSlab][PB];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int64_t n0 = (int64_t)blockIdx.x * BNt;
  const int64_t mtiles = (p.M + BMt - 1) / BMt;
  const T* A = static_cast<const T*>(p.a.ptr);
  const T* B = static_cast<const T*>(p.b.ptr);
  const T* C = static_cast<const T*>(p.c.ptr);
  T* Y = static_cast<T*>(const_cast<void*>(p.y.ptr));
  const int nslab = (int)((p.K + kSlab - 1) / kSlab);
  SlabLoad<T, BMt, kSlab> la;
  SlabLoad<T, BNt, kSlab> lb;

  for (int64_t bt = blockIdx.z; bt < p.bm.count; bt += gridDim.z) {
    const T* Ab = A + batch_offset(p.bm, p.a.bstride, bt);
    const T* Bb = B + batch_offset(p.bm, p.b.bstride, bt);
    const T* Cb = C ? C + batch_offset(p.bm, p.c.bstride, bt) : nullptr;
    T* Yb = Y + batch_offset(p.bm, p.y.bstride, bt);
    for (int64_t mt = blockIdx.y; mt < mtiles; mt += gridDim.y) {
      const int64_t m0 = mt * BMt;
      Acc acc[TM][TN];
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = Acc(0);
      if (nslab > 0) {
        la.load(Ab, p.a.rs, p.a.cs, m0, p.M, 0, p.K, opa, tid);
        lb.load(Bb, p.b.cs, p.b.rs, n0, p.N, 0, p.K, opb, tid);
        __syncthreads();   // the previous tile's last reads of buffer 0 are done
        la.store(As[0], opa, tid);
        lb.store(Bs[0], opb, tid);
        __syncthreads();
      }
      for (int s = 0; s < nslab; ++s) {
        const int buf = s & 1;
        if (s + 1 < nslab) {
          la.load(Ab, p.a.rs, p.a.cs, m0, p.M, (int64_t)(s + 1) * kSlab, p.K, opa, tid);
          lb.load(Bb, p.b.cs, p.b.rs, n0, p.N, (int64_t)(s + 1) * kSlab, p.K, opb, tid);
        }
#pragma unroll
        for (int kk = 0; kk < kSlab; ++kk) {
          Acc av[TM], bv[TN];
#pragma unroll
          for (int g = 0; g < TM / RM; ++g) {
            Acc t[RM];
            lds_vec<Acc, RM>(&As[buf][kk][g * 16 * RM + ty * RM], t);
#pragma unroll
            for (int i = 0; i < RM; ++i) av[g * RM + i] = t[i];
          }
#pragma unroll
          for (int g = 0; g < TN / RN; ++g) {
            Acc t[RN];
            lds_vec<Acc, RN>(&Bs[buf][kk][g * 16 * RN + tx * RN], t);
#pragma unroll
            for (int j = 0; j < RN; ++j) bv[g * RN + j] = t[j];
          }
#pragma unroll
          for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = mac<Acc>(acc[i][j], av[i], bv[j]);
        }
        if (s + 1 < nslab) {
          la.store(As[buf ^ 1], opa, tid);
          lb.store(Bs[buf ^ 1], opb, tid);
        }
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const int64_t gm = m0 + (i / RM) * 16 * RM + ty * RM + (i % RM);
        if (gm >= p.M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          const int64_t gn = n0 + (j / RN) * 16 * RN + tx * RN + (j % RN);
          if (gn >= p.N) continue;
          const T* c = Cb ? Cb + gm * p.c.rs + gn * p.c.cs : nullptr;
          Yb[gm * p.y.rs + gn * p.y.cs] = Arith<T>::store(Epi<T>::apply(p, acc[i][j], c));
        }
      }
    }
  }
}

// ------------------------------------------------------------------ few-row products

// With at most 4 rows of A' a product reads each element of B' once and does
// 1 to 4 multiply-adds with it: one pass over B' at memory speed.  This kernel
// takes B' K-major (column n of B' contiguous in k, as for weights stored
// [N, K]) and A' with k contiguous.  A warp owns a few adjacent columns; each
// lane loads 16-byte pieces (8 values of k; 4 for fp32) of every column, a
// round of several pieces of each before it uses any, and the same pieces of
// the rows of A' (read by every warp: they stay in L1, while the stream over
// B' bypasses it), and accumulates in fp32 (FFMA, never TF32).  The lanes'
// partial sums are added with shuffles.  The launch gives every warp the same
// number of column groups, so no warp is left streaming alone at the end.
constexpr int kVecWarps = 4;   // warps per block

// Columns per warp, pieces per column in a round, and whether the pieces of
// A' are loaded as they are used (L1 hits) instead of with the round: the
// fastest of 8 shapes timed on 1, 2 and 4 x 8192 x 8192 bf16 products.
template <int MT> struct VecShape {
  static constexpr int cols = MT == 4 ? 4 : 2;
  static constexpr int steps = MT == 4 ? 8 : 16;
  static constexpr bool a_late = MT < 4;
};

// One 16-byte piece of B', read once: not kept in L1.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// acc + the dot product of two 16-byte pieces of T values, in fp32.
template <typename T> __device__ __forceinline__ float dot16(float acc, uint4 a, uint4 b);
template <> __device__ __forceinline__ float dot16<__nv_bfloat16>(float acc, uint4 a, uint4 b) {
  const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {   // a bf16 value is the upper half of its fp32 pattern
    acc = __fmaf_rn(__uint_as_float(x[j] << 16), __uint_as_float(y[j] << 16), acc);
    acc = __fmaf_rn(__uint_as_float(x[j] & 0xffff0000u), __uint_as_float(y[j] & 0xffff0000u), acc);
  }
  return acc;
}
template <> __device__ __forceinline__ float dot16<__half>(float acc, uint4 a, uint4 b) {
  const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 hx, hy;
    memcpy(&hx, &x[j], 4);
    memcpy(&hy, &y[j], 4);
    const float2 fx = __half22float2(hx), fy = __half22float2(hy);
    acc = __fmaf_rn(fx.x, fy.x, acc);
    acc = __fmaf_rn(fx.y, fy.y, acc);
  }
  return acc;
}
// The values of a 16-byte piece as fp32.
template <typename T> __device__ __forceinline__ void unpack16(uint4 u, float (&f)[16 / sizeof(T)]);
template <> __device__ __forceinline__ void unpack16<__nv_bfloat16>(uint4 u, float (&f)[8]) {
  const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(x[j] << 16);
    f[2 * j + 1] = __uint_as_float(x[j] & 0xffff0000u);
  }
}
template <> __device__ __forceinline__ void unpack16<__half>(uint4 u, float (&f)[8]) {
  const uint32_t x[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 h;
    memcpy(&h, &x[j], 4);
    const float2 v = __half22float2(h);
    f[2 * j] = v.x;
    f[2 * j + 1] = v.y;
  }
}
template <> __device__ __forceinline__ void unpack16<float>(uint4 u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}

template <> __device__ __forceinline__ float dot16<float>(float acc, uint4 a, uint4 b) {
  acc = __fmaf_rn(__uint_as_float(a.x), __uint_as_float(b.x), acc);
  acc = __fmaf_rn(__uint_as_float(a.y), __uint_as_float(b.y), acc);
  acc = __fmaf_rn(__uint_as_float(a.z), __uint_as_float(b.z), acc);
  return __fmaf_rn(__uint_as_float(a.w), __uint_as_float(b.w), acc);
}

// Warp w takes the column groups t = w, w + warps, ... of groups x batches
// (group t: batch t / groups, columns kVecCols * (t % groups) + 0 .. kVecCols - 1).
template <typename T, int MT>
__global__ void __launch_bounds__(kVecWarps * 32) vec_gemm_kernel(const GemmArgs p, int64_t groups, int64_t tasks,
                                                                  int64_t warps) {
  pdl_begin();
  constexpr int kVecCols = VecShape<MT>::cols;
  constexpr int U = VecShape<MT>::steps;
  constexpr int kPiece = 16 / (int)sizeof(T);   // values of k in a 16-byte piece
  constexpr int kStep = 32 * kPiece;            // values of k a warp covers per piece
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * kVecWarps + (threadIdx.x >> 5);
  if (w >= warps) return;
  const T* A = static_cast<const T*>(p.a.ptr);
  const T* B = static_cast<const T*>(p.b.ptr);
  const T* C = static_cast<const T*>(p.c.ptr);
  T* Y = static_cast<T*>(const_cast<void*>(p.y.ptr));
  const int64_t kmain = p.K / (kStep * U) * (kStep * U);
  for (int64_t t = w; t < tasks; t += warps) {
    const int64_t bt = t / groups, n0 = (t - bt * groups) * kVecCols;
    const T* Ab = A + batch_offset(p.bm, p.a.bstride, bt);
    const T* Bb = B + batch_offset(p.bm, p.b.bstride, bt);
    const T* col[kVecCols];
#pragma unroll
    for (int r = 0; r < kVecCols; ++r) col[r] = Bb + (n0 + r < p.N ? n0 + r : p.N - 1) * p.b.cs;   // past N: never stored
    const T* row[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) row[m] = Ab + (m < p.M ? m : p.M - 1) * p.a.rs;
    float acc[MT][kVecCols];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < kVecCols; ++r) acc[m][r] = 0.f;

    // Every lane runs the same number of these rounds: U pieces per column.
    for (int64_t k0 = (int64_t)kPiece * lane; k0 < kmain; k0 += kStep * U) {
      uint4 bv[U][kVecCols];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < kVecCols; ++r) bv[u][r] = ld_stream(col[r] + k0 + u * kStep);
      if constexpr (VecShape<MT>::a_late) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(row[m] + k0 + u * kStep));
#pragma unroll
            for (int r = 0; r < kVecCols; ++r) acc[m][r] = dot16<T>(acc[m][r], a, bv[u][r]);
          }
      } else {
        uint4 av[U][MT];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int m = 0; m < MT; ++m) av[u][m] = __ldg(reinterpret_cast<const uint4*>(row[m] + k0 + u * kStep));
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < kVecCols; ++r) acc[m][r] = dot16<T>(acc[m][r], av[u][m], bv[u][r]);
      }
    }
    // The rest of k: whole pieces, then a ragged last piece value by value.
    for (int64_t k = kmain + (int64_t)kPiece * lane; k < p.K; k += kStep) {
      if (k + kPiece <= p.K) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const uint4 a = __ldg(reinterpret_cast<const uint4*>(row[m] + k));
#pragma unroll
          for (int r = 0; r < kVecCols; ++r) acc[m][r] = dot16<T>(acc[m][r], a, ld_stream(col[r] + k));
        }
      } else {
        for (int64_t j = k; j < p.K; ++j)
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < kVecCols; ++r)
              acc[m][r] = __fmaf_rn(Arith<T>::load(row[m] + j), Arith<T>::load(col[r] + j), acc[m][r]);
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < kVecCols; ++r)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[m][r] += __shfl_xor_sync(0xffffffffu, acc[m][r], o);
    // Lane kVecCols * m + r stores output (m, n0 + r).
    const T* Cb = C ? C + batch_offset(p.bm, p.c.bstride, bt) : nullptr;
    T* Yb = Y + batch_offset(p.bm, p.y.bstride, bt);
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int r = 0; r < kVecCols; ++r) {
        const int64_t n = n0 + r;
        if (lane == kVecCols * m + r && m < p.M && n < p.N) {
          const T* c = Cb ? Cb + m * p.c.rs + n * p.c.cs : nullptr;
          Yb[m * p.y.rs + n * p.y.cs] = Arith<T>::store(Epi<T>::apply(p, acc[m][r], c));
        }
      }
  }
}

// B' MN-major (n contiguous: B stored [K, N], MatMul's usual layout).  A
// cluster of kMnSplit CTAs owns 32 pieces of adjacent columns (256 columns of
// bf16/f16, 128 of fp32) of one batch: CTA c of the cluster takes the c-th
// slice of k, its warp w the rows w, w + kMnWarps, ... of that slice, and each
// lane one 16-byte piece of every such row, kMnRounds rows loaded before any is
// used.  A' (any strides) is read value by value: every lane of a warp reads
// the same value, one broadcast load.  The warps' fp32 partial sums go to
// shared memory and the leader CTA adds all the cluster's, in a fixed order,
// through distributed shared memory, then applies alpha, beta and C.
constexpr int kMnSplit = 8;    // CTAs per cluster: slices of k
constexpr int kMnWarps = 8;    // warps per CTA
constexpr int kMnRounds = 8;   // rows of B' per warp in flight

template <typename T, int MT>
__global__ void __cluster_dims__(kMnSplit, 1, 1) __launch_bounds__(kMnWarps * 32)
    vec_mn_kernel(const GemmArgs p) {
  pdl_begin();
  constexpr int kPiece = 16 / (int)sizeof(T);
  constexpr int kSpan = 32 * kPiece;   // columns of a cluster
  __shared__ __align__(16) float part[kMnWarps][MT][kSpan];
  cg::cluster_group cluster = cg::this_cluster();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned crank = cluster.block_rank();
  const int64_t n0 = (int64_t)blockIdx.y * kSpan + (int64_t)lane * kPiece;   // this lane's first column
  const int nvalid = n0 >= p.N ? 0 : (int)min((int64_t)kPiece, p.N - n0);
  const int64_t kslice = (p.K + kMnSplit - 1) / kMnSplit;
  const int64_t kbeg = (int64_t)crank * kslice, kend = min(p.K, kbeg + kslice);
  const T* A = static_cast<const T*>(p.a.ptr);
  const T* B = static_cast<const T*>(p.b.ptr);
  const T* C = static_cast<const T*>(p.c.ptr);
  T* Y = static_cast<T*>(const_cast<void*>(p.y.ptr));
  for (int64_t bt = blockIdx.z; bt < p.bm.count; bt += gridDim.z) {
    const T* Ab = A + batch_offset(p.bm, p.a.bstride, bt);
    const T* bcol = B + batch_offset(p.bm, p.b.bstride, bt) + (nvalid > 0 ? n0 : 0);
    const T* row[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) row[m] = Ab + (m < p.M ? m : p.M - 1) * p.a.rs;
    float acc[MT][kPiece];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < kPiece; ++j) acc[m][j] = 0.f;
    // The piece of row k of B' (columns past N read as zero).
    auto piece = [&](int64_t k) -> uint4 {
      if (nvalid == kPiece) return ld_stream(bcol + k * p.b.rs);
      T v[kPiece];
#pragma unroll
      for (int j = 0; j < kPiece; ++j) v[j] = j < nvalid ? bcol[k * p.b.rs + j] : T(0.f);
      uint4 u;
      memcpy(&u, v, 16);
      return u;
    };
    auto use = [&](int64_t k, uint4 b) {
      float f[kPiece];
      unpack16<T>(b, f);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const float a = Arith<T>::load(row[m] + k * p.a.cs);
#pragma unroll
        for (int j = 0; j < kPiece; ++j) acc[m][j] = __fmaf_rn(a, f[j], acc[m][j]);
      }
    };
    int64_t k = kbeg + warp;
    for (; k + (int64_t)(kMnRounds - 1) * kMnWarps < kend; k += (int64_t)kMnRounds * kMnWarps) {
      uint4 bv[kMnRounds];
#pragma unroll
      for (int u = 0; u < kMnRounds; ++u) bv[u] = piece(k + (int64_t)u * kMnWarps);
#pragma unroll
      for (int u = 0; u < kMnRounds; ++u) use(k + (int64_t)u * kMnWarps, bv[u]);
    }
    for (; k < kend; k += kMnWarps) use(k, piece(k));
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < kPiece; ++j) part[warp][m][lane * kPiece + j] = acc[m][j];
    cluster.sync();   // every CTA's partial sums visible to the leader
    if (crank == 0) {
      const T* Cb = C ? C + batch_offset(p.bm, p.c.bstride, bt) : nullptr;
      T* Yb = Y + batch_offset(p.bm, p.y.bstride, bt);
      for (int e = threadIdx.x; e < MT * kSpan; e += kMnWarps * 32) {
        const int m = e / kSpan, c = e - m * kSpan;
        const int64_t n = (int64_t)blockIdx.y * kSpan + c;
        float sum = 0.f;
        for (int r = 0; r < kMnSplit; ++r) {
          const float* rp = cluster.map_shared_rank(&part[0][0][0], r);
#pragma unroll
          for (int w = 0; w < kMnWarps; ++w) sum += rp[(w * MT + m) * kSpan + c];
        }
        if (m < p.M && n < p.N) {
          const T* cp = Cb ? Cb + m * p.c.rs + n * p.c.cs : nullptr;
          Yb[m * p.y.rs + n * p.y.cs] = Arith<T>::store(Epi<T>::apply(p, sum, cp));
        }
      }
    }
    cluster.sync();   // the leader has read every CTA's shared memory
  }
}

int device_sm_count() {
  static std::atomic<int> counts[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  int c = counts[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) return 0;
    counts[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

template <typename T, int MT>
mm_status launch_vec(const GemmArgs& p, cudaStream_t stream) {
  static std::atomic<int> resident{0};   // blocks of this kernel one SM holds
  int per_sm = resident.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vec_gemm_kernel<T, MT>, kVecWarps * 32, 0) !=
            cudaSuccess || per_sm <= 0)
      return MM_ERR_CUDA;
    resident.store(per_sm, std::memory_order_relaxed);
  }
  const int sms = device_sm_count();
  if (sms <= 0) return MM_ERR_CUDA;
  const int64_t groups = (p.N + VecShape<MT>::cols - 1) / VecShape<MT>::cols;
  const int64_t tasks = groups * p.bm.count;
  const int64_t wmax = (int64_t)sms * per_sm * kVecWarps;
  const int64_t rounds = (tasks + wmax - 1) / wmax;
  const int64_t warps = (tasks + rounds - 1) / rounds;   // every warp runs rounds or rounds - 1 groups
  const int64_t blocks = (warps + kVecWarps - 1) / kVecWarps;
  launch_pdl(vec_gemm_kernel<T, MT>, dim3((unsigned)blocks), dim3(kVecWarps * 32), 0, stream, p, groups, tasks, warps);
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

template <typename T, int MT>
mm_status launch_vec_mn(const GemmArgs& p, cudaStream_t stream) {
  constexpr int kSpan = 32 * (16 / (int)sizeof(T));
  const int64_t spans = (p.N + kSpan - 1) / kSpan;
  const unsigned gz = (unsigned)(p.bm.count < 65535 ? p.bm.count : 65535);
  launch_pdl(vec_mn_kernel<T, MT>, dim3(kMnSplit, (unsigned)spans, gz), dim3(kMnWarps * 32), 0, stream, p);
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

// K-major B' (vec_gemm_kernel): k contiguous in both operands, 16-byte
// aligned columns of B' and rows of A'.
bool vec_kmajor(const GemmArgs& p) {
  const int64_t v = p.dtype == MM_F32 ? 4 : 8;   // values in 16 bytes
  if (p.b.rs != 1 || p.a.cs != 1) return false;
  if (reinterpret_cast<uintptr_t>(p.b.ptr) % 16 || reinterpret_cast<uintptr_t>(p.a.ptr) % 16) return false;
  if ((p.N > 1 && p.b.cs % v) || (p.M > 1 && p.a.rs % v)) return false;
  for (int d = 0; d < p.bm.nb; ++d)
    if (p.bm.shape[d] > 1 && (p.b.bstride[d] % v || p.a.bstride[d] % v)) return false;
  return p.N <= (int64_t(1) << 40) / (p.bm.count > 0 ? p.bm.count : 1);   // column groups x batches in range
}

// MN-major B' (vec_mn_kernel): n contiguous in B', 16-byte aligned rows of B';
// A' any strides.
bool vec_mnmajor(const GemmArgs& p) {
  const int64_t v = p.dtype == MM_F32 ? 4 : 8;
  if (p.b.cs != 1 || reinterpret_cast<uintptr_t>(p.b.ptr) % 16) return false;
  if (p.K > 1 && p.b.rs % v) return false;
  for (int d = 0; d < p.bm.nb; ++d)
    if (p.bm.shape[d] > 1 && p.b.bstride[d] % v) return false;
  return (p.N + 32 * v - 1) / (32 * v) <= 65535;   // column spans: grid y
}

template <typename T>
mm_status launch_vec_t(const GemmArgs& p, cudaStream_t stream) {
  if (vec_kmajor(p)) {
    if (p.M == 1) return launch_vec<T, 1>(p, stream);
    if (p.M == 2) return launch_vec<T, 2>(p, stream);
    return launch_vec<T, 4>(p, stream);
  }
  if (p.M == 1) return launch_vec_mn<T, 1>(p, stream);
  if (p.M == 2) return launch_vec_mn<T, 2>(p, stream);
  return launch_vec_mn<T, 4>(p, stream);
}

// ------------------------------------------------------------------ QLinear

__device__ __forceinline__ int load_q(const void* base, int64_t off, int is_signed) {
  const uint8_t u = static_cast<const uint8_t*>(base)[off];
  return is_signed ? (int)(int8_t)u : (int)u;
}
__device__ __forceinline__ float load_scale(const void* base, int64_t off, int is_f16) {
  return is_f16 ? __half2float(static_cast<const __half*>(base)[off]) : static_cast<const float*>(base)[off];
}

__global__ void __launch_bounds__(kThreads) simt_qlinear_kernel(const QLinearArgs p) {
  pdl_begin();
  __shared__ int As[kTk][kTile + 1];
  __shared__ int Bs[kTk][kTile + 1];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int64_t n0 = (int64_t)blockIdx.x * kTile;
  const int64_t mtiles = (p.M + kTile - 1) / kTile;
  const float qmin = p.y_signed ? -128.f : 0.f, qmax = p.y_signed ? 127.f : 255.f;
  const float ys = load_scale(p.ys, 0, p.ys_f16);
  const float yz = (float)load_q(p.yz, 0, p.y_signed);
  uint8_t* Y = static_cast<uint8_t*>(const_cast<void*>(p.y.ptr));

  for (int64_t bt = blockIdx.z; bt < p.bm.count; bt += gridDim.z) {
    const int64_t aoff = batch_offset(p.bm, p.a.bstride, bt);
    const int64_t boff = batch_offset(p.bm, p.b.bstride, bt);
    const int64_t yoff = batch_offset(p.bm, p.y.bstride, bt);
    const int64_t saoff = batch_offset(p.bm, p.sa.bstride, bt), zaoff = batch_offset(p.bm, p.za.bstride, bt);
    const int64_t sboff = batch_offset(p.bm, p.sb.bstride, bt), zboff = batch_offset(p.bm, p.zb.bstride, bt);
    for (int64_t mt = blockIdx.y; mt < mtiles; mt += gridDim.y) {
      const int64_t m0 = mt * kTile;
      uint32_t acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0u;
      for (int64_t k0 = 0; k0 < p.K; k0 += kTk) {
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
          const int e = tid + e4 * kThreads;
          const int ar = e / kTk, ak = e % kTk;
          const int64_t gm = m0 + ar, gk = k0 + ak;
          As[ak][ar] = (gm < p.M && gk < p.K)
                           ? load_q(p.a.ptr, aoff + gm * p.a.rs + gk * p.a.cs, p.a_signed) -
                                 load_q(p.za.ptr, zaoff + gm * p.za.vs, p.a_signed)
                           : 0;
          const int bk = e / kTile, bn = e % kTile;
          const int64_t hk = k0 + bk, hn = n0 + bn;
          Bs[bk][bn] = (hk < p.K && hn < p.N)
                           ? load_q(p.b.ptr, boff + hk * p.b.rs + hn * p.b.cs, p.b_signed) -
                                 load_q(p.zb.ptr, zboff + hn * p.zb.vs, p.b_signed)
                           : 0;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kTk; ++kk) {
          uint32_t av[4], bv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) av[i] = (uint32_t)As[kk][ty + 16 * i];
#pragma unroll
          for (int j = 0; j < 4; ++j) bv[j] = (uint32_t)Bs[kk][tx + 16 * j];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] += av[i] * bv[j];   // wraps modulo 2^32
        }
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t gm = m0 + ty + 16 * i;
        if (gm >= p.M) continue;
        const float sa = load_scale(p.sa.ptr, saoff + gm * p.sa.vs, p.sa_f16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t gn = n0 + tx + 16 * j;
          if (gn >= p.N) continue;
          const float sb = load_scale(p.sb.ptr, sboff + gn * p.sb.vs, p.sb_f16);
          const float t = requant_f32((int32_t)acc[i][j], sa, sb, ys, yz, qmin, qmax);
          Y[yoff + gm * p.y.rs + gn * p.y.cs] = (uint8_t)(int)t;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ GroupedMatMul

// Quantized value at element offset e: int8 (wq 1), uint8 (2), or a 4-bit
// int4 (3) / uint4 (4) packed two per byte, element e in the low nibble of
// byte e / 2 when e is even and in its high nibble when e is odd.
__device__ __forceinline__ int load_qweight(const void* base, int64_t e, int wq) {
  const uint8_t* b = static_cast<const uint8_t*>(base);
  if (wq <= 2) return wq == 1 ? (int)(int8_t)b[e] : (int)b[e];
  const int nib = (b[e >> 1] >> ((e & 1) * 4)) & 15;
  return wq == 3 ? nib - ((nib & 8) << 1) : nib;
}

// Weight (g, k, n) of weight-only quantized experts: T((q - zp) * scale), the
// difference exact, the product exact in the accumulator type for a bf16 or
// f16 scale (at most 9 + 11 significant bits) and rounded once for f32/f64;
// then rounded once to T (GroupedMatMul - 29, Summary: DequantizeLinear of
// the weights).
template <typename T>
__device__ __forceinline__ typename Arith<T>::acc dequant_weight(const GroupedArgs& p, int64_t g, int64_t k,
                                                                 int64_t n) {
  using Acc = typename Arith<T>::acc;
  const int64_t kq = k / p.qblock;
  int d = load_qweight(p.w, g * p.w_gs + k * p.w_ks + n * p.w_ns, p.wq);
  if (p.wzp) d -= load_qweight(p.wzp, g * p.wzp_gs + kq * p.wzp_bs + n * p.wzp_ns, p.wq);
  const Acc sc = Arith<T>::load(static_cast<const T*>(p.wsc) + g * p.wsc_gs + kq * p.wsc_bs + n * p.wsc_ns);
  const T w = Arith<T>::store((Acc)d * sc);
  return Arith<T>::load(&w);
}

template <typename T, bool QW>
__global__ void __launch_bounds__(kThreads) simt_grouped_kernel(const GroupedArgs p, unsigned* status) {
  pdl_begin();
  using Acc = typename Arith<T>::acc;
  constexpr int kChunk = 1024;
  __shared__ Acc xs[kChunk];
  const T* X = static_cast<const T*>(p.x);
  const T* W = static_cast<const T*>(p.w);
  const T* Bias = static_cast<const T*>(p.bias);
  T* Out = static_cast<T*>(p.out);
  const int64_t rows = p.M * p.S;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    const int64_t m = r / p.S, i = r % p.S;
    const int64_t goff = m * p.gi_ms + i * p.gi_ss;
    const int64_t g = p.ind64 ? static_cast<const int64_t*>(p.gi)[goff]
                              : (int64_t) static_cast<const int32_t*>(p.gi)[goff];
    const int64_t n = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (g < 0 || g >= p.G) {   // invalid input: never read weights[g]; zero row, flag it
      if (n < p.N) Out[r * p.N + n] = Arith<T>::store(Acc(0));
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, kStatusIndexRange);
      continue;
    }
    Acc acc = Acc(0);
    for (int64_t k0 = 0; k0 < p.K; k0 += kChunk) {
      const int kc = (int)((p.K - k0) < kChunk ? (p.K - k0) : kChunk);
      __syncthreads();
      for (int k = threadIdx.x; k < kc; k += kThreads) xs[k] = Arith<T>::load(X + m * p.x_rs + (k0 + k) * p.x_cs);
      __syncthreads();
      if (n < p.N) {
        if (QW) {
          for (int k = 0; k < kc; ++k) acc = mac<Acc>(acc, xs[k], dequant_weight<T>(p, g, k0 + k, n));
        } else {
          const T* wcol = W + g * p.w_gs + n * p.w_ns + k0 * p.w_ks;
          for (int k = 0; k < kc; ++k) acc = mac<Acc>(acc, xs[k], Arith<T>::load(wcol + k * p.w_ks));
        }
      }
    }
    if (n < p.N) {
      if (Bias) acc = acc + Arith<T>::load(Bias + g * p.bias_gs + n * p.bias_ns);
      Out[r * p.N + n] = Arith<T>::store(acc);
    }
  }
}

template <typename T>
void launch_grouped(const GroupedArgs& p, unsigned* status, dim3 grid, cudaStream_t stream) {
  if (p.wq) launch_pdl(simt_grouped_kernel<T, true>, grid, dim3(kThreads), 0, stream, p, status);
  else launch_pdl(simt_grouped_kernel<T, false>, grid, dim3(kThreads), 0, stream, p, status);
}

dim3 tile_grid(int64_t M, int64_t N, int64_t batch) {
  const int64_t nt = (N + kTile - 1) / kTile, mt = (M + kTile - 1) / kTile;
  return dim3((unsigned)nt, (unsigned)(mt < 65535 ? mt : 65535), (unsigned)(batch < 65535 ? batch : 65535));
}

// How the tiled kernel reads an operand with `rows` rows (stride rs) and k
// stride ks: 16-byte vectors along whichever dimension is contiguous when the
// base, the other stride and every batch stride keep the vectors aligned;
// otherwise element by element, consecutive threads along the smaller stride.
SimtOperand simt_operand(const void* ptr, int elem, int64_t rs, int64_t ks, const BatchMap& bm,
                         const int64_t* bstride) {
  const int64_t v = 16 / elem;
  bool aligned = (reinterpret_cast<uintptr_t>(ptr) % 16) == 0;
  for (int d = 0; d < bm.nb; ++d) aligned = aligned && (bm.shape[d] <= 1 || bstride[d] % v == 0);
  SimtOperand op;
  op.along_k = (ks < 0 ? -ks : ks) <= (rs < 0 ? -rs : rs);
  if (aligned && ks == 1 && rs % v == 0) op.mode = kLoadVecK;
  else if (aligned && rs == 1 && ks % v == 0) op.mode = kLoadVecMN;
  else op.mode = kLoadScalar;
  return op;
}

template <typename T, int TM>
mm_status launch_tile_cfg(const GemmArgs& p, cudaStream_t stream) {
  constexpr int BT = 16 * TM;
  const int64_t nt = (p.N + BT - 1) / BT, mt = (p.M + BT - 1) / BT;
  if (nt > 0x7fffffff) return MM_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)nt, (unsigned)(mt < 65535 ? mt : 65535),
                  (unsigned)(p.bm.count < 65535 ? p.bm.count : 65535));
  const SimtOperand oa = simt_operand(p.a.ptr, (int)sizeof(T), p.a.rs, p.a.cs, p.bm, p.a.bstride);
  const SimtOperand ob = simt_operand(p.b.ptr, (int)sizeof(T), p.b.cs, p.b.rs, p.bm, p.b.bstride);
  launch_pdl(simt_gemm_kernel<T, TM, TM>, grid, dim3(kThreads), 0, stream, p, oa, ob);
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

// The largest tile that still gives every SM a block: 128 x 128 (8 x 8 per
// thread) for 32- and 16-bit types, 64 x 64 for 64-bit ones, down to 32 x 32
// for small products, which are bound by latency rather than arithmetic.
template <typename T>
mm_status launch_tiles(const GemmArgs& p, cudaStream_t stream) {
  const int64_t sms = sm_count_public();
  auto tiles = [&](int64_t bt) { return ((p.M + bt - 1) / bt) * ((p.N + bt - 1) / bt) * p.bm.count; };
  if constexpr (sizeof(typename Arith<T>::acc) == 8) {
    if (tiles(64) >= sms) return launch_tile_cfg<T, 4>(p, stream);
    return launch_tile_cfg<T, 2>(p, stream);
  } else {
    if (tiles(128) >= sms) return launch_tile_cfg<T, 8>(p, stream);
    if (tiles(64) >= sms) return launch_tile_cfg<T, 4>(p, stream);
    return launch_tile_cfg<T, 2>(p, stream);
  }
}

}  // namespace

mm_status launch_simt_gemm(const GemmArgs& p, cudaStream_t stream) {
  if (p.M == 0 || p.N == 0 || p.bm.count == 0) return MM_OK;
  switch (p.dtype) {
    case MM_BF16: return launch_tiles<__nv_bfloat16>(p, stream);
    case MM_F16: return launch_tiles<__half>(p, stream);
    case MM_F32: return launch_tiles<float>(p, stream);
    case MM_F64: return launch_tiles<double>(p, stream);
    case MM_I32: return launch_tiles<int32_t>(p, stream);
    case MM_I64: return launch_tiles<int64_t>(p, stream);
    case MM_U32: return launch_tiles<uint32_t>(p, stream);
    case MM_U64: return launch_tiles<uint64_t>(p, stream);
    default: return MM_ERR_DTYPE;
  }
}

bool vec_gemm_supported(const GemmArgs& p) {
  if (p.dtype != MM_BF16 && p.dtype != MM_F16 && p.dtype != MM_F32) return false;
  if (p.M < 1 || p.M > kVecMaxRows || p.N < 1 || p.K < 1) return false;
  return vec_kmajor(p) || vec_mnmajor(p);
}

// With 3 or 4 rows of 16-bit values against MN-major B' the tensor-core
// kernel is as fast (8192 x 8192) or faster (4096 x 14336): the planner keeps
// those there.
bool vec_gemm_preferred(const GemmArgs& p) {
  return vec_gemm_supported(p) && (vec_kmajor(p) || p.dtype == MM_F32 || p.M <= 2);
}

mm_status launch_vec_gemm(const GemmArgs& p, cudaStream_t stream) {
  if (p.M == 0 || p.N == 0 || p.bm.count == 0) return MM_OK;
  switch (p.dtype) {
    case MM_BF16: return launch_vec_t<__nv_bfloat16>(p, stream);
    case MM_F16: return launch_vec_t<__half>(p, stream);
    case MM_F32: return launch_vec_t<float>(p, stream);
    default: return MM_ERR_DTYPE;
  }
}

mm_status launch_simt_qlinear(const QLinearArgs& p, cudaStream_t stream) {
  if (p.M == 0 || p.N == 0 || p.bm.count == 0) return MM_OK;
  if ((p.N + kTile - 1) / kTile > 0x7fffffff) return MM_ERR_UNSUPPORTED;
  launch_pdl(simt_qlinear_kernel, tile_grid(p.M, p.N, p.bm.count), dim3(kThreads), 0, stream, p);
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

mm_status launch_simt_grouped(const GroupedArgs& p, unsigned* status, cudaStream_t stream) {
  const int64_t rows = p.M * p.S;
  if (rows == 0 || p.N == 0) return MM_OK;
  const int64_t nb = (p.N + kThreads - 1) / kThreads;
  if (nb > 0x7fffffff) return MM_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)nb, (unsigned)(rows < 65535 ? rows : 65535));
  switch (p.dtype) {
    case MM_BF16: launch_grouped<__nv_bfloat16>(p, status, grid, stream); break;
    case MM_F16: launch_grouped<__half>(p, status, grid, stream); break;
    case MM_F32: launch_grouped<float>(p, status, grid, stream); break;
    case MM_F64: launch_grouped<double>(p, status, grid, stream); break;
    default: return MM_ERR_DTYPE;
  }
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

}  // namespace qg
