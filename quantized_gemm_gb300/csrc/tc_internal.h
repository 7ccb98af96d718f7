// Internal interface of the tcgen05 GEMM (tc_gemm.cu) used by the operator
// front ends (MatMul/Gemm in tc_gemm.cu, QLinearMatMul and GroupedMatMul in
// tc_prep.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace qg {

constexpr int kTileM = 128;   // UMMA M (TMEM lanes)
constexpr int kTileN = 256;   // UMMA N (TMEM columns per accumulator)
constexpr int kTileK = 64;    // one 128-byte swizzle row of 16-bit elements

// kGroupedQ: GroupedMatMul whose weights arrive as int8/uint8 with scales and
// zero points (DequantizeLinear fused into the mainloop; CTA pairs only).
// kTF32: fp32 MatMul / Gemm as three tf32 products (hi*hi + hi*lo + lo*hi of
// each operand's split x = hi + lo, split in shared memory by converter warps).
// kSkinny: dense bf16/f16 products with at most 64 rows and few tiles (a
// vector or a few rows against a wide B'): 256-column tiles whose k-blocks
// are split across the `split` CTAs of a cluster; each CTA keeps its fp32
// partial sums in shared memory and reduces a slice of the columns over
// distributed shared memory, so that every SM streams its own share of B'.
enum TcMode { kDense = 0, kGrouped = 1, kQLinear = 2, kGroupedQ = 3, kTF32 = 4, kSkinny = 5 };

struct TcParams {
  int64_t M, N, K;
  int64_t mt, nt, tiles;                       // tile counts (dense / qlinear)
  BatchMap bm;
  // 32-bit tile decoding (filled by launch_tc): divisors by the tiles per
  // batch, per raster band and (last band) the band height, and by each batch
  // dimension; tile indices are < 2^31.
  FastDiv fd_per_batch, fd_band, fd_last_h;
  uint32_t last_band;
  FastDiv fd_bshape[kMaxBatchDims];
  int64_t a_bc[kMaxBatchDims], b_bc[kMaxBatchDims];   // batch index -> TMA batch coordinate
  int a_mn, b_mn;                              // operand is MN-major in shared memory
  int num_kb, kb_per_seg;                      // k-blocks; k-blocks per accumulation segment
  int split;                                   // kSkinny: CTAs of a cluster that split one tile's k-blocks
  uint32_t idesc;                              // tcgen05 instruction descriptor
  // CTA pairs: a pair tile with at most 128 valid rows (the last row tile of
  // a group, or of a dense product) runs as one M = 128 cta_group::2 MMA
  // (idesc_tail) whose A rows (64 per CTA) come from the second A map.
  int pair_tail;
  uint32_t idesc_tail;
  // output: dense/qlinear y + boff(batch) + m*y_rs + n; grouped y + out_row*y_rs + n
  void* y;
  int64_t y_bstride[kMaxBatchDims];
  int64_t y_rs;
  int y_vec, out_f16, out_f32;
  // 16-bit dense outputs: y_tma set when the epilogue writes each warp's
  // output as 32 x 32 boxes with TMA tensor stores (the map is the kernel's
  // fourth tensor map); y_bc maps a batch index to the map's batch coordinate.
  int y_tma;
  int64_t y_bc[kMaxBatchDims];
  // float epilogue: v = alpha*acc + beta*C
  float alpha, beta;
  const void* c;
  int64_t c_bstride[kMaxBatchDims];
  int64_t c_rs, c_cs, c_gs;                    // c_gs: grouped bias row stride per group
  int c_vec;
  // QLinear epilogue: zero-point correction from the operand sums, then requantisation
  VecView sa, sb, za, zb;
  const void* ys;
  const void* yz;
  int sa_f16, sb_f16, ys_f16, y_signed;
  int a_signed, b_signed;                      // uint8 operands were shifted by -128
  const int32_t* q_rs;                         // [a matrices, M] row sums of a'
  const int32_t* q_cs;                         // [b matrices, N] column sums of b'
  // GroupedMatMul routing tables (device, in the workspace)
  const int32_t* g_count;
  const int32_t* g_offset;
  const int32_t* g_tile_start;
  const int32_t* g_rowlist;
  int G;
  // kGroupedQ: weights are int8 (w_signed) or uint8, or with w4 int4
  // (w_signed) or uint4 packed two per byte (the even column in the low
  // nibble); a scale row (and, when wzp_present, a zero-point row of the
  // weights' type) applies to kb_per_q consecutive k-blocks.
  int w_signed, w4, wzp_present, kb_per_q;
  unsigned* status;
  unsigned long long timeout_ns;    // limit of each pipeline wait
  unsigned long long teardown_ns;   // limit of the waits that let in-flight copies and MMAs land
};

struct OperandPlan {
  CUtensorMap map;
  int mn_major;
  int64_t bc[kMaxBatchDims];
};

bool plan_operand(const void* ptr, int dtype, int64_t mn_len, int64_t k_len, int64_t mn_stride, int64_t k_stride,
                  const BatchMap& bm, const int64_t* bstride, int box_mn, OperandPlan* out);
// A plain (unswizzled) 3-D tensor map over elements of elem_bytes bytes:
// dims d0 (contiguous) x d1 x d2, byte strides s1 and s2, box box0 x box1 x 1.
bool plan_plain_3d(const void* ptr, int elem_bytes, int64_t d0, int64_t d1, int64_t d2, int64_t s1, int64_t s2,
                   int box0, int box1, OperandPlan* out);
uint32_t make_idesc(int f16, int a_mn, int b_mn, bool pair);
// The same with an explicit MMA height (128 or 256 rows).
uint32_t make_idesc_rows(int f16, int a_mn, int b_mn, uint32_t m);
// The same with an explicit MMA width (16..256 columns, a multiple of 16).
uint32_t make_idesc_mn(int f16, int a_mn, int b_mn, uint32_t m, uint32_t n);
uint32_t make_idesc_tf32(bool pair);
void init_params(TcParams* p);
// Fills the tile bookkeeping and launches tc_gemm_kernel: one CTA per SM, or
// (pair) 2-CTA clusters computing 256-row tiles with cta_group::2 MMAs.
// Returns MM_ERR_UNSUPPORTED when pairs cannot be placed.
// kGroupedQ also takes the scale and zero-point maps (s, z); for kDense and
// kGrouped pairs with p.pair_tail set, s is A's map with a 64-row box.
mm_status launch_tc(int mode, bool pair, const OperandPlan& a, const OperandPlan& b, TcParams& p,
                    cudaStream_t stream, const OperandPlan* s = nullptr, const OperandPlan* z = nullptr);
// Whether an M x K problem uses CTA pairs.
bool use_pair(int64_t M, int64_t K);
bool use_grouped_pair(int64_t rows, int64_t G, int64_t K);
// Whether the fused-dequantisation kernel's CTA pairs can be resident.
bool grouped_q_pairs_available();
int sm_count_public();

}  // namespace qg
