// Launchers implemented by the kernel translation units and called by the
// C-ABI layer (api.cu).  Every launcher enqueues work on `stream` and returns
// MM_OK or MM_ERR_CUDA; arguments have been validated by the caller.
#pragma once

#include "common.cuh"

namespace qg {

// MatMul and Gemm: Y[b] = alpha * A[b] @ B[b] + beta * C (C broadcast view).
struct GemmArgs {
  int dtype;                 // mm_dtype shared by A, B, C, Y
  int64_t M, N, K;
  BatchMap bm;
  MatView a;                 // rows M, cols K
  MatView b;                 // rows K, cols N
  MatView c;                 // rows M, cols N (strides 0 where broadcast); ptr null = absent
  MatView y;                 // rows M, cols N, dense
  float alpha, beta;         // float types
  double alpha_d, beta_d;    // f64
  uint64_t alpha_i, beta_i;  // integer types: two's complement of the integral values
  // Integer types with a non-integral alpha or beta: y = trunc(alpha*acc + beta*c)
  // evaluated in fp64 (each product, then the sum, rounded once), saturated to T.
  int int_float;
};

// QLinearMatMul.
struct QLinearArgs {
  int64_t M, N, K;
  BatchMap bm;
  MatView a, b, y;           // a: rows M cols K; b: rows K cols N; y dense
  int64_t a_bshape[kMaxBatchDims], b_bshape[kMaxBatchDims];  // operands' own batch sizes (1 = broadcast)
  VecView sa, za;            // indexed by row m (vs = 0 for per-tensor)
  VecView sb, zb;            // indexed by column n
  const void* ys;            // y_scale (one element)
  const void* yz;            // y_zero_point (one element)
  int a_signed, b_signed, y_signed;
  int sa_f16, sb_f16, ys_f16;
};

// GroupedMatMul.
struct GroupedArgs {
  int dtype;                 // T
  int ind64;                 // Tind is int64
  int64_t M, K, N, G, S;
  const void* x;   int64_t x_rs, x_cs;
  const void* w;   int64_t w_gs, w_ks, w_ns;
  const void* gi;  int64_t gi_ms, gi_ss;
  const void* bias; int64_t bias_gs, bias_ns;   // bias null = absent
  void* out;                 // dense [M, S, N]
  // Weight-only quantized experts: w holds int8 (wq == 1), uint8 (2), int4
  // (3) or uint4 (4) values and the weights are W = T((w - zero_point) *
  // scale), scale and zero point [G, Kb, N] indexed by (g, k / qblock, n).
  // 4-bit values are packed two per byte (element offset e: the low nibble
  // of byte e / 2 when e is even, else its high nibble; strides in elements).
  // wq == 0: w is T.
  int wq;
  const void* wsc; int64_t wsc_gs, wsc_bs, wsc_ns;   // scale, type T
  const void* wzp; int64_t wzp_gs, wzp_bs, wzp_ns;   // zero point (null = 0), type of w
  int64_t qblock;
};

mm_status launch_simt_gemm(const GemmArgs& args, cudaStream_t stream);
// Multiprocessors of the current device (cached per device).
int sm_count_public();
// Products with at most kVecMaxRows rows of A' (bf16, f16, f32): one pass over
// B' on the CUDA cores, for K-major B' (k contiguous in A' and B', 16-byte
// aligned rows of A' and columns of B') and for MN-major B' (n contiguous,
// 16-byte aligned rows of B'; A' any strides).  vec_gemm_supported says
// whether launch_vec_gemm takes the call, vec_gemm_preferred whether the
// planner should send it there.
constexpr int kVecMaxRows = 4;
bool vec_gemm_supported(const GemmArgs& args);
bool vec_gemm_preferred(const GemmArgs& args);
mm_status launch_vec_gemm(const GemmArgs& args, cudaStream_t stream);
mm_status launch_simt_qlinear(const QLinearArgs& args, cudaStream_t stream);
mm_status launch_simt_grouped(const GroupedArgs& args, unsigned* status, cudaStream_t stream);

// Streaming measurement kernels (stream.cu): bytes is a multiple of 16 and the
// buffers are 16-byte aligned (checked by the caller).
enum { kStreamWrite = 0, kStreamCopy = 1, kStreamWriteBulk = 2 };
// Arithmetic-rate probe: dependent multiply-add chains of one instruction.
enum { kAluImad = 0, kAluDfma = 1, kAluFfma = 2 };
constexpr int kAluChains = 16;     // independent chains per thread
constexpr int kAluThreads = 256;   // threads per block
constexpr int kAluBlocksPerSm = 4;
mm_status launch_alu_probe(int op, void* out, int64_t iters, int* threads_out, cudaStream_t stream);
mm_status launch_stream_probe(void* dst, const void* src, int64_t bytes, int mode, cudaStream_t stream);

}  // namespace qg
