/*
 * mm.h -- C ABI of the GB300 (sm_103a) library for the ONNX matrix-product
 * operator family: MatMul, Gemm, QLinearMatMul and GroupedMatMul.
 *
 * Every entry point takes plain pointers and sizes; no C++ or framework type
 * crosses this boundary.  All computation runs in this library's own CUDA
 * kernels on the caller's stream; there is no CPU fallback.
 *
 * Conventions shared by all entry points
 * --------------------------------------
 * Tensors.  An mm_tensor names caller-owned DEVICE memory (`data`), an element
 *   type, a rank (0..MM_MAX_DIMS), a shape and per-dimension strides counted in
 *   ELEMENTS (not bytes).  Input strides may be any non-negative values,
 *   including 0 (a broadcast view).  Output tensors (Y, y, output) must be
 *   dense row-major (strides equal to the suffix products of the shape) and
 *   must not overlap any input.
 * Shapes.  Outputs are preallocated by the caller with exactly the shape and
 *   type the operator infers (the *_output_shape helpers compute it); any other
 *   shape returns MM_ERR_SHAPE and any other type MM_ERR_DTYPE.
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Calls are asynchronous: the return value reports host-side
 *   validation and launch errors only.  mm_matmul, mm_gemm, mm_qlinear_matmul
 *   and mm_grouped_matmul enqueue only kernels and asynchronous memsets, so
 *   once one call has run on the device (it caches per-device properties)
 *   they can be captured in a CUDA graph and replayed.  Device-side conditions (an out-of-range
 *   group index, a pipeline wait that timed out) are recorded in a per-device
 *   status word read with mm_get_device_status().  Every kernel is launched
 *   with programmatic stream serialization: it may be scheduled while the
 *   previous kernel on the stream is finishing, and waits for that kernel to
 *   complete (and its memory to be visible) before its first global-memory
 *   access, so stream order is kept for any work before or after a call.
 * Memory.  The library never allocates device memory.  Operators whose fast
 *   path needs scratch space (QLinearMatMul, GroupedMatMul) take a
 *   caller-provided workspace whose size is given by the matching
 *   *_workspace_size function; the workspace must be 256-byte aligned.
 * Threads.  Entry points may be called from several host threads; calls that
 *   share a workspace must be ordered on one stream.
 */
#ifndef QGEMM_GB300_MM_H
#define QGEMM_GB300_MM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MM_MAX_DIMS 8

typedef enum mm_status {
  MM_OK = 0,
  MM_ERR_INVALID_ARG = 1,  /* NULL pointer, rank out of range, negative size or stride, bad attribute */
  MM_ERR_SHAPE = 2,        /* shapes violate the operator's rules, or the output has the wrong shape/layout */
  MM_ERR_DTYPE = 3,        /* an element type outside the operator's type constraints */
  MM_ERR_UNSUPPORTED = 4,  /* a case the pages leave undefined, or a forced path that cannot run it */
  MM_ERR_WORKSPACE = 5,    /* workspace NULL, too small or not 256-byte aligned */
  MM_ERR_CUDA = 6,         /* a CUDA runtime call or kernel launch failed */
  MM_ERR_TIMEOUT = 7,      /* device side: a pipeline wait exceeded its limit and the kernel gave up */
  MM_ERR_INDEX_RANGE = 8   /* device side: a GroupedMatMul index outside [0, G) was seen */
} mm_status;

typedef enum mm_dtype {
  MM_BF16 = 0, MM_F16 = 1, MM_F32 = 2, MM_F64 = 3,
  MM_I32 = 4, MM_I64 = 5, MM_U32 = 6, MM_U64 = 7,
  MM_I8 = 8, MM_U8 = 9,
  /* 4-bit integers ([-8, 7] and [0, 15]), packed two per byte: the element
   * at element offset e = sum_d index[d] * strides[d] is the low nibble of
   * byte e / 2 of `data` when e is even and its high nibble when e is odd.
   * Accepted only as the weights and zero points of
   * mm_grouped_matmul_qweights (quantized experts stored with 4 bits). */
  MM_I4 = 10, MM_U4 = 11
} mm_dtype;

typedef struct mm_tensor {
  void* data;                      /* device pointer, caller-owned */
  int32_t dtype;                   /* an mm_dtype value */
  int32_t ndim;                    /* 0 .. MM_MAX_DIMS */
  int64_t shape[MM_MAX_DIMS];
  int64_t strides[MM_MAX_DIMS];    /* in elements */
} mm_tensor;

/* Which kernel family runs a call (see mm_set_path_policy / mm_last_path). */
typedef enum mm_path {
  MM_PATH_AUTO = 0,    /* policy only: let the planner choose */
  MM_PATH_SIMT = 1,    /* CUDA-core kernels (every type, every stride pattern) */
  MM_PATH_TENSOR = 2,  /* tcgen05 tensor-core kernels (bf16/f16, fp32 as three tf32 products, 8-bit quantized operands) */
  MM_PATH_NONE = 3,    /* result only: no kernel was needed (an empty output) */
  MM_PATH_VECTOR = 4   /* MatMul/Gemm with 1 to 4 rows of A' (bf16/f16/f32) and B' either K-major (k
                          contiguous in A' and B', 16-byte aligned rows of A' and columns of B') or
                          MN-major (n contiguous, 16-byte aligned rows of B'): one pass over B' on the
                          CUDA cores */
} mm_path;

/* Human-readable name of a status code; never NULL. */
const char* mm_status_string(mm_status status);

/* Library version string, e.g. "0.1.0". */
const char* mm_version(void);

/* Process-wide planner policy (MM_PATH_AUTO by default).  MM_PATH_SIMT forces
 * the CUDA-core tile kernels; MM_PATH_TENSOR forces the tensor-core kernels and
 * makes calls they cannot run return MM_ERR_UNSUPPORTED.  MM_PATH_VECTOR forces
 * the few-row kernel for MatMul and Gemm (MM_ERR_UNSUPPORTED where it does not
 * apply) and acts as MM_PATH_AUTO for the other operators.  Under
 * MM_PATH_AUTO the few-row kernels take every MatMul/Gemm call they can run
 * that streams at least 2^17 elements of B' (N * K * batch), except 3 or 4
 * rows of bf16/f16 against MN-major B' (the tensor cores are as fast there);
 * smaller ones run on the CUDA-core tiles.
 * Meant for tests and measurements.  Returns MM_ERR_INVALID_ARG for an unknown
 * value. */
mm_status mm_set_path_policy(int32_t policy);

/* The mm_path taken by the most recent successful compute call made on the
 * calling host thread (MM_PATH_NONE before any). */
int32_t mm_last_path(void);

/* Failure detection.  Every wait of the tensor-core kernels' pipeline
 * (shared-memory stages, TMEM accumulators) gives up after this many
 * nanoseconds; the kernel then records MM_ERR_TIMEOUT in the device status,
 * lets its in-flight copies and MMAs land (those final waits keep a fixed 2 s
 * limit), releases its tensor memory and exits, leaving the CUDA context
 * usable.  Default 2e9 ns; 0 restores the default.  Applies to calls made
 * after it returns; meant for tests and diagnosis. */
mm_status mm_set_wait_limit_ns(uint64_t ns);

/* ---------------------------------------------------------------- MatMul
 * MatMul (onnx-light operator page, ai.onnx MatMul since version 13; summary
 * and Examples): Y = A @ B with numpy.matmul semantics.  A 1-D A is promoted to
 * [1, K] and a 1-D B to [K, 1], the promoted dimension being removed from Y;
 * leading (batch) dimensions are right-aligned and broadcast (each pair equal
 * or containing a 1).  T is one of bf16, f16, f32, f64, i32, i64, u32, u64 and
 * is shared by A, B and Y.
 * Arithmetic: bf16/f16 and f32 accumulate in fp32, f64 in fp64, then one
 * round-to-nearest-even conversion to T; integer types wrap modulo 2^n.  f32
 * never uses plain TF32: small or strided f32 products use FFMA, large ones
 * with a unit-stride matrix dimension per operand use three tf32 tensor-core
 * products (each operand split into tf32 high and low parts; relative error
 * about 3 * 2^-22 per product, within the fp32 bound).  K = 0 gives zeros. */
mm_status mm_matmul_output_shape(const mm_tensor* A, const mm_tensor* B,
                                 int32_t* out_ndim, int64_t* out_shape /* [MM_MAX_DIMS] */);
mm_status mm_matmul(const mm_tensor* A, const mm_tensor* B, const mm_tensor* Y, void* stream);

/* ---------------------------------------------------------------- Gemm
 * Gemm (onnx-light operator page, ai.onnx Gemm since version 13; definition
 * and Inputs/Outputs): Y = alpha * A' * B' + beta * C, A' = A^T if transA != 0
 * else A (A is (M,K) or (K,M)), B' = B^T if transB != 0 else B (B is (K,N) or
 * (N,K)), Y is (M,N).  C is optional (NULL = absent = scalar 0) and
 * unidirectionally broadcastable to (M,N): rank <= 2, right-aligned, each
 * dimension equal to the target or 1.  ONNX defaults are alpha = beta = 1,
 * transA = transB = 0.  Float T: y = alpha*acc + beta*c evaluated in fp32
 * (fp64 for f64), rounded once to T.  Integer T (the page does not say how
 * a real-valued result becomes a T): with integral alpha and beta, Y is exact
 * modulo 2^n; otherwise acc = A'B' wraps modulo 2^n to a T value, then
 * r = alpha*acc + beta*C is evaluated in fp64 (each product rounded, then the
 * sum) and truncated toward zero; results outside T's range are undefined
 * (this library saturates them).  Non-finite alpha or beta with an integer T
 * returns MM_ERR_UNSUPPORTED. */
mm_status mm_gemm_output_shape(const mm_tensor* A, const mm_tensor* B, int64_t transA, int64_t transB,
                               int32_t* out_ndim, int64_t* out_shape /* [MM_MAX_DIMS] */);
mm_status mm_gemm(const mm_tensor* A, const mm_tensor* B, const mm_tensor* C /* NULL = absent */,
                  float alpha, float beta, int64_t transA, int64_t transB,
                  const mm_tensor* Y, void* stream);

/* ---------------------------------------------------------------- QLinearMatMul
 * QLinearMatMul - version 10 (onnx-light operator page source; summary,
 * Inputs, Type Constraints): numpy.matmul of 8-bit operands with
 *   acc = sum_k (a - a_zero_point) * (b - b_zero_point)   exact, wrapped to int32,
 *   y   = saturate(round_half_even(x / y_scale) + y_zero_point),
 * where x is evaluated in IEEE fp32 as  s = a_scale*b_scale; v = float(acc)*s;
 * q = v / y_scale  (each a correctly rounded fp32 operation, in this order) and
 * saturate clamps to [-128,127] (int8) or [0,255] (uint8).  Results are
 * bit-exact with that definition.
 * Types: a/a_zero_point share T1, b/b_zero_point share T2, y/y_zero_point share
 * T3, each MM_I8 or MM_U8; scales are MM_F32 (MM_F16 is also accepted and is
 * widened exactly to fp32).
 * Parameter shapes: a scale and its zero point have the same shape.  One
 * element = per tensor.  Per row of a: [M] (2-D a) or a.shape[:-1] + [1].
 * Per column of b: [N] (2-D b) or b.shape[:-2] + [1, N].  y_scale and
 * y_zero_point are per tensor.  Scales and zero points are device tensors.
 * The output shape is mm_matmul_output_shape(a, b).
 * Workspace: mm_qlinear_matmul_workspace_size() bytes (0 when the planner uses
 * the CUDA-core kernel, which needs none). */
mm_status mm_qlinear_matmul_workspace_size(const mm_tensor* a, const mm_tensor* b, size_t* bytes);
mm_status mm_qlinear_matmul(const mm_tensor* a, const mm_tensor* a_scale, const mm_tensor* a_zero_point,
                            const mm_tensor* b, const mm_tensor* b_scale, const mm_tensor* b_zero_point,
                            const mm_tensor* y_scale, const mm_tensor* y_zero_point,
                            const mm_tensor* y, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- GroupedMatMul
 * GroupedMatMul - 29 (onnx.ai operator page; Summary, Inputs, Outputs, Type
 * Constraints): input [M,K], weights [G,K,N], group_indices [M,S] (MM_I32 or
 * MM_I64), optional bias [G,N] (NULL = absent), output [M,S,N]:
 *   output[m,i,:] = input[m,:] @ weights[g,:,:] (+ bias[g,:]),  g = group_indices[m,i].
 * T is bf16, f16, f32 or f64.  The selected weights are never materialised:
 * rows are routed to their group on the device and each group's rows are
 * multiplied by weights[g] in place.  Accumulation as for MatMul; the bias is
 * added to the accumulator before the single rounding to T.
 * Indices outside [0, G) are invalid input (undefined on the page).  Here the
 * kernels never read out of bounds for them: the affected output rows are
 * written as zeros and MM_ERR_INDEX_RANGE is recorded in the device status.
 * Workspace: mm_grouped_matmul_workspace_size() bytes. */
mm_status mm_grouped_matmul_workspace_size(const mm_tensor* input, const mm_tensor* weights,
                                           const mm_tensor* group_indices, size_t* bytes);
mm_status mm_grouped_matmul(const mm_tensor* input, const mm_tensor* weights,
                            const mm_tensor* group_indices, const mm_tensor* bias /* NULL = absent */,
                            const mm_tensor* output, void* workspace, size_t workspace_bytes,
                            void* stream);

/* ---------------------------------------------------------------- GroupedMatMul, weight-only quantized experts
 * GroupedMatMul - 29 (onnx.ai operator page), Summary, last paragraph: experts
 * whose weights are stored quantized are expressed as DequantizeLinear of the
 * weights followed by GroupedMatMul, and a runtime may fuse the two so that
 * the dequantized [G, K, N] weights are never formed.  This entry point is
 * that fusion:
 *   W[g,k,n] = T((weights_q[g,k,n] - w_zero_point[g,k/B,n]) * w_scale[g,k/B,n])
 *   output[m,i,:] = input[m,:] @ W[g,:,:] (+ bias[g,:]),  g = group_indices[m,i],
 * with B = block_size (0 means K: one scale per group and output column).
 * The pages name DequantizeLinear without defining it; this is the reading
 * used: the difference is an exact integer and the product is rounded once to
 * T (nearest, ties to even), so W is exactly what a separate dequantization to
 * T would store; the product with W then accumulates as in mm_grouped_matmul.
 *   input [M,K] (T = bf16, f16, f32 or f64); weights_q [G,K,N] MM_I8, MM_U8,
 *   MM_I4 or MM_U4; w_scale [G, ceil(K/B), N] of type T; w_zero_point NULL
 *   (zero) or of the type of weights_q and the shape of w_scale; 4-bit
 *   weights and zero points need a unit stride along N, N even and even
 *   strides along G and K (rows start on byte boundaries; otherwise
 *   MM_ERR_SHAPE); group_indices [M,S] MM_I32 or
 *   MM_I64; bias NULL or [G,N] of type T; output dense [M,S,N] of type T.
 *   block_size < 0 returns MM_ERR_INVALID_ARG.  Invalid group indices as for
 *   mm_grouped_matmul (zero rows, MM_ERR_INDEX_RANGE in the device status).
 * The tensor-core path (bf16/f16; weights, scales and zero points with a
 * unit-stride N dimension and 16-byte aligned rows; B a multiple of 64 or
 * B >= K) keeps the weights 8- or 4-bit in memory: each k-block is loaded
 * as stored and converted in shared memory just before the tensor cores
 * read it.
 * Workspace: mm_grouped_matmul_qweights_workspace_size() bytes. */
mm_status mm_grouped_matmul_qweights_workspace_size(const mm_tensor* input, const mm_tensor* weights_q,
                                                    const mm_tensor* w_scale, const mm_tensor* w_zero_point,
                                                    int64_t block_size, const mm_tensor* group_indices,
                                                    size_t* bytes);
mm_status mm_grouped_matmul_qweights(const mm_tensor* input, const mm_tensor* weights_q, const mm_tensor* w_scale,
                                     const mm_tensor* w_zero_point /* NULL = 0 */, int64_t block_size,
                                     const mm_tensor* group_indices, const mm_tensor* bias /* NULL = absent */,
                                     const mm_tensor* output, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* ---------------------------------------------------------------- GroupedMatMul without allocation
 * This entry point has no counterpart in the operator pages; it exists for
 * callers that cannot allocate device memory at call time: code whose device
 * memory is fixed when it starts (a serving loop or plugin that must not call
 * cudaMalloc, which can block and synchronise the device, or that runs inside
 * a host framework owning every allocation).  mm_grouped_matmul needs a
 * caller-provided workspace; this variant computes the same result with the
 * same tensor-core kernels but takes its scratch from a fixed array of
 * mm_grouped_matmul_noalloc_max_scratch() bytes (16 MiB) that the library
 * holds in device memory on every GPU where it is loaded, until the process
 * exits.  It calls no cudaMalloc, cudaFree or allocating library routine.
 *   Arguments, layout and result: as mm_grouped_matmul, without the workspace.
 *   Limits: bf16/f16 operands whose layout the tensor-core kernels take
 *   (otherwise MM_ERR_UNSUPPORTED; f32/f64 callers can use mm_grouped_matmul,
 *   whose CUDA-core path needs no workspace), and a problem whose scratch
 *   (mm_grouped_matmul_workspace_size() under the tensor-core policy: the
 *   routing tables plus M*S rows of K elements) fits the array; larger
 *   problems return MM_ERR_WORKSPACE.
 *   Path: always the tensor-core routing and GEMM kernels, whatever
 *   mm_set_path_policy says (the CUDA-core path needs no scratch at all).
 *   The first call on a device looks up the array's device address (a CUDA
 *   runtime query, no allocation); make that first call before any stream
 *   capture.  The address is then cached for the device's ordinal for the rest
 *   of the process, so it does not survive cudaDeviceReset (nor does the
 *   device-status word's, which every entry point caches the same way): do not
 *   call the library on a device after resetting it.  Every call on a device
 *   shares the one array and each call resets
 *   what it needs, so calls whose GPU work overlaps (different streams, or
 *   other host threads) race on it and must be ordered by the caller. */
size_t mm_grouped_matmul_noalloc_max_scratch(void);
mm_status mm_grouped_matmul_noalloc(const mm_tensor* input, const mm_tensor* weights,
                                    const mm_tensor* group_indices, const mm_tensor* bias /* NULL = absent */,
                                    const mm_tensor* output, void* stream);

/* ---------------------------------------------------------------- memory-stream measurement
 * Not an operator (the pages have no counterpart): the streaming kernels that
 * measure the HBM roofline a memory-bound product is compared with.
 *   mode 0: write `bytes` of a constant to dst (16-byte vector stores);
 *   mode 1: copy `bytes` from src to dst (16-byte vector loads and stores);
 *   mode 2: write `bytes` with bulk (TMA) stores from shared memory.
 * dst (and src for mode 1) are device memory owned by the caller, 16-byte
 * aligned; bytes is a multiple of 16 (otherwise MM_ERR_INVALID_ARG).  The
 * call is asynchronous on `stream`; time it with events on that stream. */
mm_status mm_stream_probe(void* dst, const void* src, size_t bytes, int32_t mode, void* stream);

/* ---------------------------------------------------------------- arithmetic-rate measurement
 * Not an operator (the pages have no counterpart): the peak rate of the
 * CUDA-core multiply-add that the tiled kernels use for the types without a
 * tensor-core path, against which they are compared.
 *   op 0: mad.lo.u32 (int32 / uint32 GEMMs), op 1: fma.rn.f64 (f64),
 *   op 2: fma.rn.f32 (f32 on the CUDA cores).
 * Every thread of a grid of 4 blocks of 256 threads per SM runs 16
 * independent chains of `iters` dependent multiply-adds.  *multiply_adds (if not NULL)
 * receives the total count (ops = 2 x that); out, device memory owned by the
 * caller, 8-byte aligned, must hold one 8-byte value per thread (at most
 * 4 * 256 * SMs values); with out NULL only the count is returned.  The call
 * is asynchronous on `stream`; time it with events on that stream.
 * Returns MM_ERR_INVALID_ARG for an unknown op, iters < 0 or a misaligned out. */
mm_status mm_alu_probe(int32_t op, void* out, int64_t iters, int64_t* multiply_adds, void* stream);

/* ---------------------------------------------------------------- device status
 * Synchronises `stream`, then returns and clears the device-side status of the
 * current device: MM_OK, MM_ERR_INDEX_RANGE or MM_ERR_TIMEOUT (the first set,
 * in that order of precedence: TIMEOUT over INDEX_RANGE), or MM_ERR_CUDA if the
 * synchronisation itself failed. */
mm_status mm_get_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_GB300_MM_H */
