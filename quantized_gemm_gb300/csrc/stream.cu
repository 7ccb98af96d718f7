// Streaming kernels that measure the memory roofline this library's kernels
// are judged against (and, at the end, the arithmetic-rate probe of the
// CUDA-core instructions the tiled GEMM uses): a write-only stream (the bound of a product whose
// traffic is almost all output, such as a batched product with a 128-deep k)
// and a copy.  They are measurement helpers, not operator steps.
//
// Every kernel is persistent (a few CTAs per SM, grid-stride over the
// buffer) and moves 16-byte vectors:
//  * kWrite: st.global.v4 of a constant, 4 vectors in flight per thread;
//  * kCopy: ld.global.nc.L1::no_allocate.v4 then st.global.v4, 4 in flight;
//  * kWriteBulk: one thread per CTA issues cp.async.bulk stores of a zeroed
//    32 KiB shared-memory buffer (the TMA's untiled bulk store) to successive
//    chunks, keeping at most 16 bulk groups pending.
#include <cstdint>

#include "kernels.h"

namespace qg {
namespace {

constexpr int kStreamThreads = 256;
constexpr int kBulkChunk = 32 * 1024;

__global__ void __launch_bounds__(kStreamThreads) write_stream_kernel(uint4* dst, int64_t nvec) {
  const uint4 v = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[i + u * stride] = v;
  }
  for (; i < nvec; i += stride) dst[i] = v;
}

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kStreamThreads) copy_stream_kernel(uint4* dst, const uint4* src, int64_t nvec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ld_nc(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < nvec; i += stride) dst[i] = ld_nc(src + i);
}

__global__ void __launch_bounds__(32) write_bulk_kernel(char* dst, int64_t bytes) {
  __shared__ __align__(128) uint4 buf[kBulkChunk / 16];
  for (int i = threadIdx.x; i < kBulkChunk / 16; i += 32) buf[i] = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if (threadIdx.x != 0) return;
  const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(buf);
  const int64_t nchunks = (bytes + kBulkChunk - 1) / kBulkChunk;
  for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const int64_t off = c * kBulkChunk;
    const uint32_t n = (uint32_t)(bytes - off < kBulkChunk ? bytes - off : kBulkChunk);
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst + off), "r"(sbuf), "r"(n) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 16;" ::: "memory");
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// kAluChains independent chains x = x * a + c per thread, `iters` steps each,
// in the instruction being measured (inline PTX, so each step is one
// mad.lo.u32 / fma.rn.f64 / fma.rn.f32); the chains' sum is stored so that
// nothing is dead.  a and c come from the caller's arguments.
template <int OP>
__global__ void __launch_bounds__(kAluThreads) alu_probe_kernel(void* out, int64_t iters, uint32_t seed) {
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
  if constexpr (OP == kAluImad) {
    uint32_t x[kAluChains];
    const uint32_t a = seed | 1u, c = seed ^ 0x9e3779b9u;
#pragma unroll
    for (int j = 0; j < kAluChains; ++j) x[j] = tid + j;
#pragma unroll 4
    for (int64_t i = 0; i < iters; ++i)
#pragma unroll
      for (int j = 0; j < kAluChains; ++j) asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(x[j]) : "r"(a), "r"(c));
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < kAluChains; ++j) s += x[j];
    static_cast<uint32_t*>(out)[tid] = s;
  } else if constexpr (OP == kAluDfma) {
    double x[kAluChains];
    const double a = 1.0 - (double)(seed & 0xff) * 0x1p-40, c = 0x1p-30;
#pragma unroll
    for (int j = 0; j < kAluChains; ++j) x[j] = (double)(tid + j);
#pragma unroll 4
    for (int64_t i = 0; i < iters; ++i)
#pragma unroll
      for (int j = 0; j < kAluChains; ++j) asm volatile("fma.rn.f64 %0, %0, %1, %2;" : "+d"(x[j]) : "d"(a), "d"(c));
    double s = 0;
#pragma unroll
    for (int j = 0; j < kAluChains; ++j) s += x[j];
    static_cast<double*>(out)[tid] = s;
  } else {
    float x[kAluChains];
    const float a = 1.0f - (float)(seed & 0xff) * 0x1p-20f, c = 0x1p-12f;
#pragma unroll
    for (int j = 0; j < kAluChains; ++j) x[j] = (float)(tid + j);
#pragma unroll 4
    for (int64_t i = 0; i < iters; ++i)
#pragma unroll
      for (int j = 0; j < kAluChains; ++j) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x[j]) : "f"(a), "f"(c));
    float s = 0;
#pragma unroll
    for (int j = 0; j < kAluChains; ++j) s += x[j];
    static_cast<float*>(out)[tid] = s;
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

mm_status launch_stream_probe(void* dst, const void* src, int64_t bytes, int mode, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return MM_ERR_CUDA;
  const int64_t nvec = bytes / 16;
  switch (mode) {
    case kStreamWrite:
      write_stream_kernel<<<sms * 4, kStreamThreads, 0, stream>>>(static_cast<uint4*>(dst), nvec);
      break;
    case kStreamCopy:
      copy_stream_kernel<<<sms * 4, kStreamThreads, 0, stream>>>(static_cast<uint4*>(dst),
                                                                 static_cast<const uint4*>(src), nvec);
      break;
    case kStreamWriteBulk:
      write_bulk_kernel<<<sms * 4, 32, 0, stream>>>(static_cast<char*>(dst), bytes);
      break;
    default:
      return MM_ERR_INVALID_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

mm_status launch_alu_probe(int op, void* out, int64_t iters, int* threads_out, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return MM_ERR_CUDA;
  const int blocks = sms * kAluBlocksPerSm;
  if (threads_out) *threads_out = blocks * kAluThreads;
  if (!out) return MM_OK;
  const uint32_t seed = (uint32_t)(iters * 2654435761u);
  switch (op) {
    case kAluImad: alu_probe_kernel<kAluImad><<<blocks, kAluThreads, 0, stream>>>(out, iters, seed); break;
    case kAluDfma: alu_probe_kernel<kAluDfma><<<blocks, kAluThreads, 0, stream>>>(out, iters, seed); break;
    case kAluFfma: alu_probe_kernel<kAluFfma><<<blocks, kAluThreads, 0, stream>>>(out, iters, seed); break;
    default: return MM_ERR_INVALID_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}

}  // namespace qg
