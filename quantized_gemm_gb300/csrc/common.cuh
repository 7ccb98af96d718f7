// Internal types shared by the host planner and the CUDA kernels.
//
// An operand of any operator is described as a batch of 2-D matrices: a
// broadcast batch shape (BatchMap, row-major, shared by all operands of one
// call) plus, per operand, one element stride per batch dimension (0 where the
// operand is broadcast) and the element strides of its two matrix dimensions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "mm.h"

namespace qg {

constexpr int kMaxBatchDims = MM_MAX_DIMS - 2;

struct BatchMap {
  int nb;                          // number of batch dimensions
  int64_t shape[kMaxBatchDims];    // broadcast batch shape
  int64_t count;                   // product of shape (1 when nb == 0)
};

struct MatView {                   // X[b, r, c] = ptr[boff(b) + r*rs + c*cs]
  const void* ptr;
  int64_t bstride[kMaxBatchDims];
  int64_t rs, cs;
};

struct VecView {                   // per-row / per-column parameter: ptr[boff(b) + i*vs]
  const void* ptr;
  int64_t bstride[kMaxBatchDims];
  int64_t vs;
};

// Division of a 32-bit unsigned integer by an invariant divisor 1 <= d < 2^31
// with one multiply-high and a shift (Granlund & Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, unsigned case):
// l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, and for every n < 2^32
// n / d = (mulhi(m, n) + n) >> l, the sum taken in 64 bits.
struct FastDiv {
  uint32_t d, mul, shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  f.shift = l;
  f.mul = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
  return f;
}

__host__ __device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  const uint32_t t = (uint32_t)(((uint64_t)n * f.mul) >> 32);
  return (uint32_t)(((uint64_t)t + n) >> f.shift);
}

// Device status word bits (see mm_get_device_status).
enum : unsigned { kStatusIndexRange = 1u, kStatusTimeout = 2u };

// Element offset of flattened batch index b for an operand with strides bstride.
__host__ __device__ __forceinline__ int64_t batch_offset(const BatchMap& bm, const int64_t* bstride,
                                                         int64_t b) {
  int64_t off = 0;
  for (int d = bm.nb - 1; d >= 0; --d) {
    const int64_t n = bm.shape[d];
    off += (b % n) * bstride[d];
    b /= n;
  }
  return off;
}

// QLinearMatMul requantisation of one int32 accumulator: each step is one
// correctly rounded IEEE fp32 operation, in the order
//   s = a_scale*b_scale; v = float(acc)*s; q = v/y_scale; r = rint(q) (ties to even);
//   t = r + y_zero_point; saturate with fmin/fmax to [qmin, qmax].
// (QLinearMatMul - version 10: quantization formula and rounding sentence.)
__device__ __forceinline__ float requant_f32(int32_t acc, float sa, float sb, float ys, float yzp,
                                             float qmin, float qmax) {
  const float s = __fmul_rn(sa, sb);
  const float v = __fmul_rn(__int2float_rn(acc), s);
  const float q = __fdiv_rn(v, ys);
  const float r = rintf(q);
  const float t = __fadd_rn(r, yzp);
  return fminf(fmaxf(t, qmin), qmax);
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization (launch_pdl) and calls pdl_wait()
// before its first access to global memory: it waits there until the kernels
// it depends on on its stream have completed and their memory is visible, so
// that its launch and set-up overlap the end of the previous kernel.
// pdl_trigger() lets the next kernel on the stream be launched before this
// one ends (otherwise that happens as this grid completes).  Short SIMT
// kernels and the large dense tensor-core products trigger right after their
// wait; the operand preparation kernels and the few-row, QLinear and grouped
// products do not, since the next kernel's blocks, resident early, measured
// slower there.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
  pdl_wait();
  pdl_trigger();
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace qg
