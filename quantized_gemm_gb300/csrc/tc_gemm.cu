// tcgen05 tensor-core GEMM for sm_103a (GB300), shared by the MatMul, Gemm,
// QLinearMatMul and GroupedMatMul fast paths.
//
// Structure (one persistent CTA per SM, 576 threads):
//   warp 0      TMA producer: one thread streams A and B tiles (BK = 64) into a
//               shared-memory ring, 128-byte swizzled, completing on per-stage
//               mbarriers (full[s]); it waits on empty[s] before reusing a stage.
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma
//               (K=16, fp32 accumulation) into one of two 256-column TMEM
//               accumulators and commits: empty[s] when a stage has been
//               consumed, acc_full[b] when an accumulation segment is complete.
//   warps 2-17  epilogue: wait acc_full[b], tcgen05.ld the accumulator (warp w
//               owns TMEM lanes 32*(w%4).. and a 64-column slice),
//               release the buffer (acc_empty[b]) and write the output through
//               a swizzled shared-memory stage so that every warp store covers
//               whole 32-byte sectors.
// Two TMEM accumulators let the epilogue of one segment overlap the MMAs of
// the next.  Every mbarrier wait is bounded; a wait that runs out sets the
// timeout bit of the device status word and the CTA winds down cleanly.
//
// Single CTAs compute 128 x 256 tiles with tcgen05.mma.cta_group::1 (4-stage
// ring of 48 KB).  For long-K dense products two CTAs of a cluster compute one
// 256 x 256 tile with tcgen05.mma.cta_group::2: each loads its 128 rows of A
// and half of the tile's B columns (6-stage ring of 32 KB), the even CTA
// issues the MMAs for both, and commits are multicast to the pair.  Each SM
// then takes in 64 bytes of operands per MMA cycle instead of 96.  A pair
// tile with at most 128 valid rows (a group's or a product's last row tile)
// runs as one M = 128 cta_group::2 MMA fed by 64 rows of A per CTA.
//
// Tiles are numbered in a grouped raster (bands of 8 row tiles, for L2 reuse)
// and decoded with 32-bit multiply-shift division by precomputed divisors.
//
// Modes (template parameter):
//   kDense    MatMul / Gemm: tiles over (batch, M, N); epilogue
//             y = alpha*acc + beta*C[bcast], rounded once to bf16/f16.
//   kGrouped  GroupedMatMul: A rows are the routed (group-ordered) copy of the
//             input rows, B is weights[g]; tiles come from the device-built
//             per-group tile table; epilogue adds bias[g] and scatters each
//             row to output[m, i, :].
//   kQLinear  QLinearMatMul: operands are int8/uint8 values moved into
//             [-128, 127] (uint8 minus 128) and held exactly in f16.  Products
//             are at most 2^14 in magnitude, so each 1024-deep segment sums
//             exactly in the fp32 accumulator; the epilogue converts each
//             segment to int32, adds with wrap-around, applies the zero points
//             from the operands' row and column sums, then requantises.
//   kGroupedQ GroupedMatMul with int8/uint8 weights: converter warps form
//             T((q - zp) * scale) in shared memory (CTA pairs).
//   kTF32     fp32 MatMul / Gemm as three tf32 products of split operands.
//   kSkinny   kDense for at most 64 rows of A': 256-column tiles whose
//             k-blocks are split over the CTAs of a cluster (non-persistent,
//             one tile per cluster), so that B' streams through every SM with
//             few, wide MMAs; each CTA leaves its partial sums in its shared
//             memory and each CTA adds the cluster's partials for its share
//             of the columns, in a fixed order, through distributed shared
//             memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "tc.h"
#include "tc_internal.h"
#include "tc_ptx.cuh"

namespace qg {

using namespace ptx;

namespace {

constexpr int BM = kTileM, BN = kTileN, BK = kTileK;
constexpr int kEpiWarp0 = 2;                     // warps 2.. run the epilogue

// Shared-memory ring geometry.  One CTA: A 128x64 + B 256x64 per stage (48 KB),
// 4 stages.  CTA pair (cta_group::2, a 256 x 256 tile per pair): each CTA holds
// its 128 rows of A and half (128) of the tile's B columns, 32 KB per stage,
// 6 stages.
template <int MODE, bool PAIR>
struct Geo {
  // kSkinny: 64-row A boxes; the M = 128 MMA's rows 64..127 read the
  // stage's B bytes and are never stored.
  static constexpr int kTileN = BN;
  static constexpr int kBRows = PAIR ? BN / 2 : kTileN;  // B columns (rows of B') held by one CTA
  static constexpr int kABytes = (MODE == kSkinny ? BM / 2 : BM) * BK * 2;   // rows x 128 bytes
  static constexpr int kBBytes = kBRows * BK * 2;
  // kTF32: each stage holds the loaded (then high) parts of A and B followed
  // by their low parts at kLoOff.
  static constexpr int kLoOff = MODE == kTF32 ? kABytes + kBBytes : 0;
  static constexpr int kStageBytes = (kABytes + kBBytes) * (MODE == kTF32 ? 2 : 1);
  // kGroupedQ gives one stage's worth of shared memory to its int8 staging ring.
  static constexpr int kStages =
      MODE == kTF32 ? (PAIR ? 3 : 2) : PAIR ? (MODE == kGroupedQ ? 5 : 6) : MODE == kSkinny ? 5 : 4;
  static constexpr int kTileRows = PAIR ? 2 * BM : BM;  // output rows per (pair) tile
  static constexpr int kRingBytes = kStages * kStageBytes;
};
// Raster band height (tiles, a power of two).  On the 8192^3 Gemm, bands of
// 8 pair tiles read 1.08 GB from DRAM per call against 1.28 GB for 16 (4:
// 1.41 GB, 32: 2.05 GB); under the power cap that traffic costs clock: 1620
// against 1608 TFLOP/s over 1000 calls.
constexpr int kGroupM = 8;
// kGroupedQ staging ring (per CTA and stage): the int8 weight tile (64 k x 128
// n), the k-block's scale row (128 x 16-bit) and zero-point row (128 bytes).
// Five slots fill the shared memory (0.4 % faster than four on the 64-expert
// workload).
constexpr int kQStages = 5;
constexpr int kQTileBytes = 64 * 128, kQScaleOff = kQTileBytes, kQZeroOff = kQScaleOff + 256;
constexpr int kQStageBytes = 9216;
constexpr int kConvWarps = 4;                    // kGroupedQ converter warps (one per SM sub-partition)
constexpr int kSignalBytes = 16;                 // per converter warp and k-block (see run_convert)
constexpr int kSignalOff = 240;                  // 16 spare bytes of the control block: signal source/target

__host__ __device__ constexpr bool is_grouped(int mode) { return mode == kGrouped || mode == kGroupedQ; }
constexpr int64_t kPairMinK = 1024;              // CTA pairs for K >= this
constexpr uint32_t kTmemCols = 512;
constexpr int kCtrlBytes = 256;                  // mbarriers, TMEM slot, abort flag
constexpr int kStageWords = 32 * 16;             // float per-warp output staging: 32 rows x 64 bytes

// Shape of the CTA: 16 epilogue warps of 64 columns each, enough warps to hide
// the epilogue's latency (short-K float products, the QLinear requantisation).
// With 18 warps ptxas caps a thread at 96 registers (five warps share one SM
// sub-partition's register file); QLinear keeps its 64 int32 running sums in
// registers and drains TMEM 16 columns at a time.  kGroupedQ runs 8 epilogue
// warps of 128 columns plus 4 converter warps (14 warps: 128 registers).
template <int MODE, bool PAIR>
struct Cfg {
  static constexpr int kEpiWarps = (MODE == kGroupedQ || MODE == kTF32) ? 8 : 16;
  static constexpr int kConv = (MODE == kGroupedQ || MODE == kTF32) ? kConvWarps : 0;
  static constexpr int kConvWarp0 = kEpiWarp0 + kEpiWarps;
  static constexpr int kThreads = (kEpiWarp0 + kEpiWarps + kConv) * 32;
  static constexpr int kCols = kTileN / (kEpiWarps / 4);      // columns per epilogue warp
  static constexpr int kWarpWords = MODE == kQLinear ? 3 * kCols : (MODE == kTF32 || MODE == kSkinny) ? 0 : kStageWords;
  static constexpr int kEpiBytes = kEpiWarps * kWarpWords * 4;
  // kGroupedQ staging ring, after the epilogue's slices (1024-byte aligned)
  static constexpr int kQOff = (Geo<MODE, PAIR>::kRingBytes + kCtrlBytes + kEpiBytes + 1023) / 1024 * 1024;
  static constexpr int kSmem = (MODE == kGroupedQ ? kQOff + kQStages * kQStageBytes
                                                  : Geo<MODE, PAIR>::kRingBytes + kCtrlBytes + kEpiBytes) +
                               1024;
  static_assert(kSmem <= 232448, "shared memory per block");
  static_assert(16 * Geo<MODE, PAIR>::kStages + 48 +
                        (MODE == kGroupedQ ? 16 * kQStages : MODE == kTF32 ? 8 * Geo<MODE, PAIR>::kStages : 0) <=
                    kSignalOff,
                "control block");
  static_assert(MODE != kGroupedQ || PAIR, "the fused dequantisation runs on CTA pairs");
};

struct Tile {
  uint32_t batch;    // dense: broadcast batch index
  int64_t m0, n0;    // first output row / column of the tile
  int32_t a_row;     // TMA coordinate of the first A row
  int32_t a_b, b_b;  // TMA batch coordinates
  int32_t rows;      // valid rows in the tile
  int32_t g;         // grouped: group
};

// Offset of broadcast batch index b for per-dimension strides `bstride`,
// decomposing b with the precomputed divisors.
__device__ __forceinline__ int64_t batch_off(const TcParams& p, const int64_t* bstride, uint32_t b) {
  int64_t off = 0;
  for (int d = p.bm.nb - 1; d >= 0; --d) {
    const uint32_t q = fast_div(b, p.fd_bshape[d]);
    off += (int64_t)(b - q * p.fd_bshape[d].d) * bstride[d];
    b = q;
  }
  return off;
}

// Tile t of the persistent schedule.  `g_hint` carries the group found for the
// previous tile of the same CTA (tiles only move forward), so the grouped
// lookup is a short forward scan.
template <int MODE, bool PAIR>
__device__ __forceinline__ bool get_tile(const TcParams& p, int64_t t, int64_t total, Tile& ti, int& g_hint) {
  if (t >= total) return false;
  if (is_grouped(MODE)) {
    constexpr int TR = Geo<MODE, PAIR>::kTileRows;
    int g = g_hint;
    while (g + 1 < p.G && __ldg(p.g_tile_start + g + 1) <= t) ++g;
    g_hint = g;
    const uint32_t local = (uint32_t)(t - __ldg(p.g_tile_start + g));
    const int cnt = __ldg(p.g_count + g);
    const uint32_t mtg = (uint32_t)((cnt + TR - 1) / TR);
    // Within a group, bands of up to kGroupM row tiles, each band's column
    // tiles in turn: the band's rows of A stay in L2 while its column tiles
    // stream the group's weights (8 groups: 2.32 -> 2.22 ms; 64: unchanged).
    const uint32_t ntot = (uint32_t)p.nt;
    const uint32_t band = local / (kGroupM * ntot), w = local - band * (kGroupM * ntot);
    const uint32_t h = min((uint32_t)kGroupM, mtg - band * kGroupM);
    const uint32_t ntile = w / h, mtile = band * kGroupM + (w - ntile * h);
    ti.batch = 0;
    ti.g = g;
    ti.m0 = (int64_t)mtile * TR;
    ti.n0 = (int64_t)ntile * BN;
    ti.a_row = __ldg(p.g_offset + g) + (int32_t)(mtile * TR);
    ti.a_b = 0;
    ti.b_b = g;
    ti.rows = min(TR, cnt - (int)(mtile * TR));
    return true;
  }
  const uint32_t tt = (uint32_t)t;
  const uint32_t b = fast_div(tt, p.fd_per_batch);
  const uint32_t r = tt - b * p.fd_per_batch.d;
  const uint32_t gband = fast_div(r, p.fd_band);
  const uint32_t w = r - gband * p.fd_band.d;
  uint32_t mtile, ntile;
  if (gband != p.last_band) {              // full bands are kGroupM (a power of two) tiles high
    mtile = gband * kGroupM + (w & (kGroupM - 1));
    ntile = w / kGroupM;
  } else {
    ntile = fast_div(w, p.fd_last_h);
    mtile = gband * kGroupM + (w - ntile * p.fd_last_h.d);
  }
  ti.batch = b;
  ti.g = 0;
  ti.m0 = (int64_t)mtile * Geo<MODE, PAIR>::kTileRows;
  ti.n0 = (int64_t)ntile * Geo<MODE, PAIR>::kTileN;
  ti.a_row = (int32_t)ti.m0;
  ti.a_b = (int32_t)batch_off(p, p.a_bc, b);
  ti.b_b = (int32_t)batch_off(p, p.b_bc, b);
  ti.rows = (int32_t)min((int64_t)Geo<MODE, PAIR>::kTileRows, p.M - ti.m0);
  return true;
}

template <int MODE>
__device__ __forceinline__ int64_t total_tiles(const TcParams& p) {
  return is_grouped(MODE) ? (int64_t)p.g_tile_start[p.G] : p.tiles;
}

// The persistent schedule: a CTA (or CTA pair) takes tiles first, first + step, ...
// kSkinny is not persistent: cluster c of p.split CTAs computes tile c.
template <int MODE, bool PAIR>
__device__ __forceinline__ int64_t first_tile(const TcParams& p) {
  return MODE == kSkinny ? (int64_t)(blockIdx.x / (unsigned)p.split) : PAIR ? (blockIdx.x >> 1) : blockIdx.x;
}
template <int MODE, bool PAIR>
__device__ __forceinline__ int64_t tile_step(const TcParams& p) {
  return MODE == kSkinny ? (int64_t)(gridDim.x / (unsigned)p.split) : PAIR ? (gridDim.x >> 1) : gridDim.x;
}
// The k-blocks this CTA multiplies: all of them, or (kSkinny) its share of
// the tile's, k-blocks [r*num_kb/split, (r+1)*num_kb/split) for cluster rank r.
template <int MODE>
__device__ __forceinline__ void kb_range(const TcParams& p, int& b, int& e) {
  if (MODE == kSkinny) {
    const int r = (int)(blockIdx.x % (unsigned)p.split);
    b = (int)((int64_t)r * p.num_kb / p.split);
    e = (int)((int64_t)(r + 1) * p.num_kb / p.split);
  } else {
    b = 0;
    e = p.num_kb;
  }
}

// ------------------------------------------------------------------ producer

template <int MODE, bool PAIR>
__device__ void run_producer(const CUtensorMap* tmA, const CUtensorMap* tmB, const CUtensorMap* tmS,
                             const CUtensorMap* tmZ, const TcParams& p, uint32_t sbase, uint32_t full0,
                             uint32_t empty0, uint32_t qbase, uint32_t qfull0, uint32_t qempty0,
                             volatile int* abort) {
  using G = Geo<MODE, PAIR>;
  prefetch_tmap(tmA);
  prefetch_tmap(tmB);
  if (MODE == kGroupedQ) {
    prefetch_tmap(tmS);
    if (p.wzp_present) prefetch_tmap(tmZ);
  }
  const int64_t total = total_tiles<MODE>(p);
  // In a pair each CTA loads its own 128 rows of A and 128 columns of B; every
  // copy completes on the leader CTA's full barrier, which expects both CTAs' bytes.
  const uint32_t rank = PAIR ? (cluster_ctarank() & 1) : 0;
  const int32_t arow_off = PAIR ? (int32_t)(rank * BM) : 0;
  const int32_t bcol_off = PAIR ? (int32_t)(rank * G::kBRows) : 0;
  uint32_t stage = 0, phase = 0;
  uint32_t pending = 0, pend_parity = 0;   // bit s: a load into stage s was issued (and its parity)
  uint32_t qstage = 0, qphase = 0, qpending = 0, qpend_parity = 0;   // the same for the staging ring
  // kGroupedQ: bytes one staging slot receives per k-block (weight tile,
  // scale row, zero-point row)
  const uint32_t qbytes = p.w4 ? kQTileBytes / 2 + 256 + (p.wzp_present ? 64 : 0)
                               : kQTileBytes + 256 + (p.wzp_present ? 128 : 0);
  Tile ti;
  int gh = 0;
  int kb_b, kb_e;
  kb_range<MODE>(p, kb_b, kb_e);
  for (int64_t t = first_tile<MODE, PAIR>(p); get_tile<MODE, PAIR>(p, t, total, ti, gh); t += tile_step<MODE, PAIR>(p)) {
    for (int kb = kb_b; kb < kb_e; ++kb) {
      if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort, p.status, p.timeout_ns)) goto done;
      const uint32_t full = full0 + 8 * stage;
      const uint32_t sa = sbase + stage * G::kStageBytes, sb = sa + G::kABytes;
      const int32_t k0 = kb * (MODE == kTF32 ? 32 : BK);
      const int32_t ar = ti.a_row + arow_off, bc = (int32_t)ti.n0 + bcol_off;
      if (MODE == kTF32) {
        // fp32 tiles land on this CTA's own "loaded" barrier; the converter
        // warps split them and then arm the stage (see run_split).
        const uint32_t ld = qfull0 + 8 * stage;
        if (PAIR && rank == 0) mbar_arrive_expect_tx(full, 2 * kConvWarps * kSignalBytes);
        mbar_arrive_expect_tx(ld, G::kABytes + G::kBBytes);
        // K-major tiles load straight into the high-part buffer; MN-major
        // tiles (32 x 32 boxes) into the low-part buffer, to be transposed.
        if (!p.a_mn) {
          tma_load_3d(sa, tmA, k0, ar, ti.a_b, ld);
        } else {
#pragma unroll
          for (int j = 0; j < BM / 32; ++j) tma_load_3d(sa + G::kLoOff + j * 4096, tmA, ar + 32 * j, k0, ti.a_b, ld);
        }
        if (!p.b_mn) {
          tma_load_3d(sb, tmB, k0, bc, ti.b_b, ld);
        } else {
#pragma unroll
          for (int j = 0; j < G::kBRows / 32; ++j)
            tma_load_3d(sb + G::kLoOff + j * 4096, tmB, bc + 32 * j, k0, ti.b_b, ld);
        }
        qpending |= 1u << stage;
        qpend_parity = (qpend_parity & ~(1u << stage)) | (phase << stage);
      } else if (MODE == kGroupedQ) {
        // A as usual; the B half arrives as int8 (plus its scale and zero-point
        // rows) in the staging ring, and the converter warps write it to sb.
        if (!mbar_wait(qempty0 + 8 * qstage, qphase ^ 1, abort, p.status, p.timeout_ns)) goto done;
        const uint32_t qfull = qfull0 + 8 * qstage, qs = qbase + qstage * kQStageBytes;
        if (rank == 0) mbar_arrive_expect_tx(full, 2 * G::kABytes + 2 * kConvWarps * kSignalBytes);
        tma_load_3d_pair(sa, tmA, k0, ar, ti.a_b, mapa_shared(full, 0));
        const int32_t kq = kb / p.kb_per_q;
        // 4-bit weights and zero points: maps over bytes (two columns each)
        const int32_t bq = p.w4 ? bc >> 1 : bc;
        mbar_arrive_expect_tx(qfull, qbytes);
        tma_load_3d(qs, tmB, bq, k0, ti.b_b, qfull);
        tma_load_3d(qs + kQScaleOff, tmS, bc, kq, ti.b_b, qfull);
        if (p.wzp_present) tma_load_3d(qs + kQZeroOff, tmZ, bq, kq, ti.b_b, qfull);
        qpending |= 1u << qstage;
        qpend_parity = (qpend_parity & ~(1u << qstage)) | (qphase << qstage);
        if (++qstage == kQStages) { qstage = 0; qphase ^= 1; }
      } else if (PAIR) {
        const uint32_t bar = mapa_shared(full, 0);
        // A tail tile (at most 128 rows) takes 64 rows of A per CTA.
        const bool tail = p.pair_tail && ti.rows <= BM;
        if (rank == 0) mbar_arrive_expect_tx(full, 2 * (tail ? G::kStageBytes - G::kABytes / 2 : G::kStageBytes));
        if (tail) {
          tma_load_3d_pair(sa, tmS, k0, ti.a_row + (int32_t)(rank * (BM / 2)), ti.a_b, bar);
        } else if (!p.a_mn) {
          tma_load_3d_pair(sa, tmA, k0, ar, ti.a_b, bar);
        } else {
          tma_load_3d_pair(sa, tmA, ar, k0, ti.a_b, bar);
          tma_load_3d_pair(sa + 8192, tmA, ar + 64, k0, ti.a_b, bar);
        }
        if (!p.b_mn) {
          tma_load_3d_pair(sb, tmB, k0, bc, ti.b_b, bar);
        } else {
#pragma unroll
          for (int j = 0; j < G::kBRows / 64; ++j) tma_load_3d_pair(sb + j * 8192, tmB, bc + 64 * j, k0, ti.b_b, bar);
        }
      } else {
        mbar_arrive_expect_tx(full, G::kStageBytes);
        if (!p.a_mn) {
          tma_load_3d(sa, tmA, k0, ar, ti.a_b, full);
        } else {
          tma_load_3d(sa, tmA, ar, k0, ti.a_b, full);
          tma_load_3d(sa + 8192, tmA, ar + 64, k0, ti.a_b, full);
        }
        if (!p.b_mn) {
          tma_load_3d(sb, tmB, k0, bc, ti.b_b, full);
        } else {
#pragma unroll
          for (int j = 0; j < G::kBRows / 64; ++j) tma_load_3d(sb + j * 8192, tmB, bc + 64 * j, k0, ti.b_b, full);
        }
      }
      pending |= 1u << stage;
      pend_parity = (pend_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == G::kStages) { stage = 0; phase ^= 1; }
    }
  }
done:
  // Let every issued copy land before the CTA can exit.  In a pair the leader's
  // full barriers count both CTAs' bytes, so the leader waits for both.  The
  // waits share one deadline (after an abort, a kGroupedQ full barrier may
  // also lack the converters' arrivals and only the deadline ends its wait).
  const uint64_t t_end = globaltimer() + p.teardown_ns;
  auto left = [&]() -> uint64_t {
    const uint64_t now = globaltimer();
    return now < t_end ? t_end - now : 0;
  };
  if (!PAIR || rank == 0)
    for (int s = 0; s < G::kStages; ++s)
      if (pending & (1u << s)) {
        if (PAIR) mbar_wait_teardown_cluster(full0 + 8 * s, (pend_parity >> s) & 1u, left());
        else mbar_wait_teardown(full0 + 8 * s, (pend_parity >> s) & 1u, left());
      }
  if (MODE == kGroupedQ || MODE == kTF32)
    for (int s = 0; s < (MODE == kTF32 ? G::kStages : kQStages); ++s)
      if (qpending & (1u << s)) mbar_wait_teardown(qfull0 + 8 * s, (qpend_parity >> s) & 1u, left());
}

// ------------------------------------------------------------------ MMA issuer

// In a pair only the leader CTA runs this: one M=256 MMA covers both CTAs' rows
// (A and B halves read from both CTAs' shared memory at the same offsets), and
// every commit signals the barrier of that name in both CTAs.
template <int MODE, bool PAIR>
__device__ void run_mma(const TcParams& p, uint32_t sbase, uint32_t tmem, uint32_t full0, uint32_t empty0,
                        uint32_t accf0, uint32_t acce0, uint32_t drain, volatile int* abort) {
  using G = Geo<MODE, PAIR>;
  const int64_t total = total_tiles<MODE>(p);
  uint32_t stage = 0, phase = 0, seg = 0;
  Tile ti;
  int gh = 0;
  int kb_b, kb_e;
  kb_range<MODE>(p, kb_b, kb_e);
  for (int64_t t = first_tile<MODE, PAIR>(p); get_tile<MODE, PAIR>(p, t, total, ti, gh); t += tile_step<MODE, PAIR>(p)) {
    for (int kb0 = kb_b; kb0 < kb_e; kb0 += p.kb_per_seg) {
      const uint32_t buf = seg & 1, aph = (seg >> 1) & 1;
      const bool ok = PAIR ? mbar_wait_cluster(acce0 + 8 * buf, aph ^ 1, abort, p.status, p.timeout_ns)
                           : mbar_wait(acce0 + 8 * buf, aph ^ 1, abort, p.status, p.timeout_ns);
      if (!ok) goto done;
      tc_fence_after();
      const uint32_t d = tmem + buf * BN;
      const int kb1 = min(kb0 + p.kb_per_seg, kb_e);
      const uint32_t idesc = (PAIR && p.pair_tail && ti.rows <= BM) ? p.idesc_tail : p.idesc;
      for (int kb = kb0; kb < kb1; ++kb) {
        const bool got = PAIR ? mbar_wait_cluster(full0 + 8 * stage, phase, abort, p.status, p.timeout_ns)
                              : mbar_wait(full0 + 8 * stage, phase, abort, p.status, p.timeout_ns);
        if (!got) goto done;
        tc_fence_after();
        const uint32_t sa = sbase + stage * G::kStageBytes, sb = sa + G::kABytes;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          // K-major: advance 32 bytes inside the 128-byte swizzle row.
          // MN-major: advance two 8-row (1024-byte) swizzle atoms.
          // (kTF32 operands are K-major in shared memory whatever their layout in memory.)
          const bool amn = MODE != kTF32 && p.a_mn, bmn = MODE != kTF32 && p.b_mn;
          const uint64_t ad = amn ? smem_desc_sw128(sa + k * 2048, 8192, 1024) : smem_desc_sw128(sa + k * 32, 16, 1024);
          const uint64_t bd = bmn ? smem_desc_sw128(sb + k * 2048, 8192, 1024) : smem_desc_sw128(sb + k * 32, 16, 1024);
          const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
          if (MODE == kTF32) {
            // 8 fp32 of k per instruction: lo*hi and hi*lo (the small terms
            // first), then hi*hi.
            const uint64_t adl = smem_desc_sw128(sa + G::kLoOff + k * 32, 16, 1024);
            const uint64_t bdl = smem_desc_sw128(sb + G::kLoOff + k * 32, 16, 1024);
            if (PAIR) {
              tc_mma_tf32_pair(d, adl, bd, p.idesc, acc);
              tc_mma_tf32_pair(d, ad, bdl, p.idesc, 1u);
              tc_mma_tf32_pair(d, ad, bd, p.idesc, 1u);
            } else {
              tc_mma_tf32(d, adl, bd, p.idesc, acc);
              tc_mma_tf32(d, ad, bdl, p.idesc, 1u);
              tc_mma_tf32(d, ad, bd, p.idesc, 1u);
            }
          } else if (PAIR) {
            tc_mma_f16_pair(d, ad, bd, idesc, acc);
          } else {
            tc_mma_f16(d, ad, bd, p.idesc, acc);
          }
        }
        if (PAIR) tc_commit_pair(empty0 + 8 * stage, 0x3);
        else tc_commit(empty0 + 8 * stage);
        if (++stage == G::kStages) { stage = 0; phase ^= 1; }
      }
      if (PAIR) tc_commit_pair(accf0 + 8 * buf, 0x3);
      else tc_commit(accf0 + 8 * buf);
      ++seg;
    }
  }
done:
  if (PAIR) tc_commit_pair(drain, 0x3);
  else tc_commit(drain);
  mbar_wait_teardown(drain, 0, p.teardown_ns);
}

// ------------------------------------------------------------------ epilogue helpers

__device__ __forceinline__ uint32_t pack2(float a, float b, int f16) {
  if (f16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float unpack16(uint16_t x, int f16) {
  return f16 ? __half2float(__ushort_as_half(x)) : __bfloat162float(__ushort_as_bfloat16(x));
}

// v[j] += beta * C[n + j] for the 32 columns starting at n.
__device__ __forceinline__ void add_c32(const TcParams& p, const uint16_t* crow, int64_t n, float (&v)[32]) {
  if (p.c_vec && n + 32 <= p.N) {
    const uint4* src = reinterpret_cast<const uint4*>(crow + n);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = __ldg(src + q);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[q * 8 + 2 * e] = __fmaf_rn(p.beta, unpack16((uint16_t)(w[e] & 0xFFFF), p.out_f16), v[q * 8 + 2 * e]);
        v[q * 8 + 2 * e + 1] = __fmaf_rn(p.beta, unpack16((uint16_t)(w[e] >> 16), p.out_f16), v[q * 8 + 2 * e + 1]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n + j < p.N) v[j] = __fmaf_rn(p.beta, unpack16(crow[(n + j) * p.c_cs], p.out_f16), v[j]);
  }
}

__device__ __forceinline__ float load_scale(const void* base, int64_t off, int is_f16) {
  return is_f16 ? __half2float(static_cast<const __half*>(base)[off]) : static_cast<const float*>(base)[off];
}
__device__ __forceinline__ float load_q8(const void* base, int64_t off, int is_signed) {
  const uint8_t u = static_cast<const uint8_t*>(base)[off];
  return is_signed ? (float)(int8_t)u : (float)u;
}

// The requantisation of requant_f32 (common.cuh), returning the output byte,
// with two exact shortcuts.  rint: for |q| < 2^22, (q + 1.5*2^23) - 1.5*2^23
// rounds q to the nearest integer, ties to even, exactly as rintf; any larger
// |q| (or an infinity or NaN) saturates to the same end of [qmin, qmax] either
// way.  Byte: t is an integer in [-128, 255], so the low bits of t + 1.5*2^23
// are t in two's complement.
__device__ __forceinline__ uint32_t requant_byte(int32_t acc, float sa, float sb, float ys, float yzp, float qmin,
                                                 float qmax) {
  constexpr float kMagic = 12582912.0f;
  const float s = __fmul_rn(sa, sb);
  const float v = __fmul_rn(__int2float_rn(acc), s);
  const float q = __fdiv_rn(v, ys);
  const float r = __fsub_rn(__fadd_rn(q, kMagic), kMagic);
  const float t = fminf(fmaxf(__fadd_rn(r, yzp), qmin), qmax);
  return (uint32_t)(__float_as_int(__fadd_rn(t, kMagic)) - 0x4B400000) & 0xFFu;
}

// The same byte without a division in the common case.  With rys = RN(1/ys)
// (ys normal, |ys| < 2^126), qa = RN(v*rys) differs from the correctly rounded
// quotient qo = RN(v/ys) by less than 2^-21 |qa|: |qa - v/ys| <= ~1.5*2^-23 |qa|
// and |qo - v/ys| <= 2^-24 |qa|.  So when qa lies more than 2^-20 |qa| from
// the nearest half-integer, qa and qo lie strictly inside the same interval
// between half-integers, neither is a tie, and rint(qa) = rint(qo).  When
// |qa| >= 2^21 the result saturates whatever the rounding.  Otherwise
// (rarely) *slow is set and the caller recomputes with requant_byte.
__device__ __forceinline__ uint32_t requant_byte_fast(int32_t acc, float sa, float sb, float rys, bool fast,
                                                      float yzp, float qmin, float qmax, bool* slow) {
  constexpr float kMagic = 12582912.0f;
  const float s = __fmul_rn(sa, sb);
  const float v = __fmul_rn(__int2float_rn(acc), s);
  const float qa = __fmul_rn(v, rys);
  const float r = __fsub_rn(__fadd_rn(qa, kMagic), kMagic);
  const float half_gap = __fsub_rn(0.5f, fabsf(__fsub_rn(qa, r)));
  const float aq = fabsf(qa);
  *slow = !(fast && (aq >= 2097152.0f || half_gap > __fmul_rn(aq, 9.5367431640625e-07f)));
  const float t = fminf(fmaxf(__fadd_rn(r, yzp), qmin), qmax);
  return (uint32_t)(__float_as_int(__fadd_rn(t, kMagic)) - 0x4B400000) & 0xFFu;
}

// ------------------------------------------------------------------ dequantising converters (kGroupedQ)

// kConvWarps warps per CTA turn each k-block's int8/uint8 weight tile
// (64 k x this CTA's 128 columns, in the staging ring) into the MMA's B
// operand: W = T((q - zp) * scale), rounded once to bf16/f16, written in the
// MN-major 128-byte-swizzled layout a TMA load would give (two 64-column
// sub-tiles; the 16-byte chunk c of row k sits at chunk c ^ (k % 8)).  Thread t
// owns columns 8*(t%16) .. +7 and rows t/16 + R*i, R = 2*kConvWarps.  q - zp is
// formed exactly in fp32: the byte placed in the low mantissa of 2^23 (after
// adding 128 to int8 values) minus 2^23 + 128 + zp.  Its product with a bf16
// or f16 scale has at most 9 + 11 significant bits, so it is exact too and the
// final conversion is the only rounding.  Each warp then makes its writes
// visible to the tensor cores, frees the staging slot and arrives on the
// leader CTA's stage barrier, which the MMA waits on.
template <int MODE, bool PAIR, bool W4>
__device__ void run_convert(const TcParams& p, uint8_t* smem, uint32_t sbase, uint32_t full0, uint32_t qbase,
                            uint32_t qfull0, uint32_t qempty0, uint32_t ctrl_u32, volatile int* abort) {
  using G = Geo<MODE, PAIR>;
  const int ct = (int)threadIdx.x - Cfg<MODE, PAIR>::kConvWarp0 * 32;
  const int lane = threadIdx.x & 31;
  const int cc = ct & 15, k_first = ct >> 4;
  const int sub = cc >> 3, c = cc & 7;
  // Signed values are moved to [0, 2^bits) by flipping their top bit: + 128
  // for int8, + 8 for int4 (W4: 4-bit weights, two per byte, the even column
  // in the low nibble; a staged row is 64 bytes instead of 128).
  const float wshift = p.w_signed ? (W4 ? 8.f : 128.f) : 0.f;
  const uint32_t flip = p.w_signed ? (W4 ? 0x08080808u : 0x80808080u) : 0u;
  const float zbias = 8388608.f + wshift;
  const float hbias = 1024.f + wshift;
  const bool f16 = p.out_f16 != 0;
  // smem is the kernel's shared memory; sbase and qbase are shared addresses in it.
  const uint32_t sm0 = smem_u32(smem);
  const int64_t total = total_tiles<MODE>(p);
  uint32_t stage = 0, qstage = 0, qphase = 0;
  Tile ti;
  int gh = 0;
  for (int64_t t = first_tile<MODE, PAIR>(p); get_tile<MODE, PAIR>(p, t, total, ti, gh); t += tile_step<MODE, PAIR>(p)) {
    for (int kb = 0; kb < p.num_kb; ++kb) {
      if (!__all_sync(0xffffffffu, mbar_wait(qfull0 + 8 * qstage, qphase, abort, p.status, p.timeout_ns))) return;
      const uint8_t* qs = smem + (qbase - sm0) + qstage * kQStageBytes;
      // All of this thread's staged bytes first (kRows rows x 8 bytes), then the
      // arithmetic, then the stores: the loads overlap instead of each waiting
      // for the previous chunk's store.
      constexpr int kRowStep = 2 * kConvWarps, kRows = 64 / kRowStep;
      uint2 raw[kRows];
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        if constexpr (W4)
          raw[i] = make_uint2(*reinterpret_cast<const uint32_t*>(qs + (k_first + kRowStep * i) * 64 + cc * 4), 0u);
        else
          raw[i] = *reinterpret_cast<const uint2*>(qs + (k_first + kRowStep * i) * 128 + cc * 8);
      }
      const uint4 sraw = *reinterpret_cast<const uint4*>(qs + kQScaleOff + cc * 16);
      uint2 zraw = make_uint2(0u, 0u);
      if (p.wzp_present) {
        if constexpr (W4) zraw.x = *reinterpret_cast<const uint32_t*>(qs + kQZeroOff + cc * 4);
        else zraw = *reinterpret_cast<const uint2*>(qs + kQZeroOff + cc * 8);
      }
      // Per column pair e2: the scales as staged (a bf16/f16 pair) and the
      // zero-point bias cz = bias + zp, in fp32 (bf16) or as an f16 pair.
      const uint32_t sw[4] = {sraw.x, sraw.y, sraw.z, sraw.w};
      const uint32_t zw[2] = {zraw.x, zraw.y};
      int zp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if constexpr (W4) {
          const int nib = (int)((zraw.x >> (4 * e)) & 15u);
          zp[e] = p.w_signed ? nib - ((nib & 8) << 1) : nib;
        } else {
          const uint32_t zb = (zw[e >> 2] >> (8 * (e & 3))) & 0xFFu;
          zp[e] = p.w_signed ? (int)(int8_t)zb : (int)zb;
        }
      }
      // A row's 8 values as bytes in [0, 2^bits), in column order: 4-bit
      // values are spread over the bytes of two words (even columns from the
      // low nibbles, odd ones from the high) and interleaved back.
      auto row_bytes = [&](const uint2& r, uint32_t& qx, uint32_t& qy) {
        if constexpr (W4) {
          const uint32_t lo = (r.x & 0x0F0F0F0Fu) ^ flip, hi = ((r.x >> 4) & 0x0F0F0F0Fu) ^ flip;
          qx = __byte_perm(lo, hi, 0x5140u);
          qy = __byte_perm(lo, hi, 0x7362u);
        } else {
          qx = r.x ^ flip;
          qy = r.y ^ flip;
        }
      };
      uint8_t* bsm = smem + (sbase - sm0) + stage * G::kStageBytes + G::kABytes + sub * 8192;
      if (f16) {
        // 1024 + u as f16 (byte u in the low mantissa of 0x6400) minus
        // 1024 + shift + zp is q - zp exactly (all below 2048); the f16 pair
        // product is rounded once.
        __half2 czh[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2)
          czh[e2] = __floats2half2_rn(hbias + (float)zp[2 * e2], hbias + (float)zp[2 * e2 + 1]);
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          const int k = k_first + kRowStep * i;
          uint32_t qx, qy;
          row_bytes(raw[i], qx, qy);
          uint32_t w[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const uint32_t src = e2 < 2 ? qx : qy;
            const uint32_t hv = __byte_perm(src, 0x64u, (e2 & 1) ? 0x4342u : 0x4140u);
            const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&hv), czh[e2]);
            const __half2 y = __hmul2(d, *reinterpret_cast<const __half2*>(&sw[e2]));
            w[e2] = *reinterpret_cast<const uint32_t*>(&y);
          }
          *reinterpret_cast<uint4*>(bsm + k * 128 + ((c ^ (k & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        // The byte u (q moved to [0, 2^bits)) in byte 1 of the pattern
        // 0x47000000 is the fp32 value 32768 + u.  With the column's bf16 scale
        // s (8 significant bits) and kc = -(32768 + c) * s, c = shift + zp
        // (a 16-bit integer times s: at most 24 significant bits, exact),
        // fma(32768 + u, s, kc) is (u - c) * s = (q - zp) * s before its one
        // rounding, and that value has at most 9 + 8 significant bits: the
        // fp32 result is exact and the pair conversion to bf16 is the only
        // rounding.  Two columns per packed fp32x2 FMA.  (kc overflows for
        // |s| near 2^112; a scale of 2^100 or more in any of the thread's
        // columns takes the subtract-then-multiply form below instead.)
        float sf[8], kc[8], smax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sf[e] = __uint_as_float((e & 1) ? (sw[e >> 1] & 0xFFFF0000u) : (sw[e >> 1] << 16));
          kc[e] = __fmul_rn(-(32768.f + wshift + (float)zp[e]), sf[e]);
          smax = fmaxf(smax, fabsf(sf[e]));
        }
        if (smax < 0x1p100f) {
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            const int k = k_first + kRowStep * i;
            uint32_t qx, qy;
            row_bytes(raw[i], qx, qy);
            uint32_t w[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const uint32_t src = e2 < 2 ? qx : qy;
              const uint32_t j = (e2 & 1) * 2;
              const float2 f = make_float2(__uint_as_float(__byte_perm(src, 0x47000000u, 0x7404u + (j << 4))),
                                           __uint_as_float(__byte_perm(src, 0x47000000u, 0x7404u + ((j + 1) << 4))));
              const float2 y = fma2_rn(f, make_float2(sf[2 * e2], sf[2 * e2 + 1]), make_float2(kc[2 * e2], kc[2 * e2 + 1]));
              const __nv_bfloat162 h = __floats2bfloat162_rn(y.x, y.y);
              w[e2] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(bsm + k * 128 + ((c ^ (k & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          // q - zp exactly in fp32 (the byte in the low mantissa of 2^23, minus
          // 2^23 + c); at most 8 significant bits, so its bf16 is the upper
          // half of the fp32 pattern; the bf16 pair product is rounded once.
          float cz[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) cz[e] = zbias + (float)zp[e];
#pragma unroll
          for (int i = 0; i < kRows; ++i) {
            const int k = k_first + kRowStep * i;
            uint32_t qx, qy;
            row_bytes(raw[i], qx, qy);
            uint32_t w[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const uint32_t src = e2 < 2 ? qx : qy;
              const int b0 = (e2 & 1) * 2;
              const float f0 = __fsub_rn(__uint_as_float(__byte_perm(src, 0x4Bu, 0x4550u + b0)), cz[2 * e2]);
              const float f1 = __fsub_rn(__uint_as_float(__byte_perm(src, 0x4Bu, 0x4550u + b0 + 1)), cz[2 * e2 + 1]);
              const uint32_t dv = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);
              const __nv_bfloat162 y = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&dv),
                                               *reinterpret_cast<const __nv_bfloat162*>(&sw[e2]));
              w[e2] = *reinterpret_cast<const uint32_t*>(&y);
            }
            *reinterpret_cast<uint4*>(bsm + k * 128 + ((c ^ (k & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      // Publish the stage: each lane orders its writes before the async
      // proxy; then one 16-byte bulk copy into the leader CTA completes its
      // bytes on the leader's stage barrier, which the MMA waits on.  (A
      // cluster-scope release arrive did the same but held the warp for
      // about 1100 cycles per k-block; the copy is issued without waiting.)
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(qempty0 + 8 * qstage);
        bulk_copy_to_cluster(mapa_shared(ctrl_u32 + kSignalOff, 0), ctrl_u32 + kSignalOff, kSignalBytes,
                             mapa_shared(full0 + 8 * stage, 0));
      }
      if (++stage == G::kStages) stage = 0;
      if (++qstage == kQStages) { qstage = 0; qphase ^= 1; }
    }
  }
}

// ------------------------------------------------------------------ fp32 splitting converters (kTF32)

// Four warps per CTA turn each loaded fp32 k-block (A and this CTA's part of
// B, 32 values of k per 128-byte row, 128-byte swizzled) into two tf32
// operands in place: hi = tf32(x) overwrites x and lo = tf32(x - hi) goes to
// the same offset of the low-part buffer, so both keep the loaded layout.
// x - hi is exact in fp32, and ab - (hi_a hi_b + hi_a lo_b + lo_a hi_b) is at
// most about 3 * 2^-22 |ab|.  The stage is then published to the MMA as in
// run_convert (bulk-copy signals for a pair; plain arrivals for one CTA).
// hi = tf32(x), lo = tf32(x - hi) for four values.
__device__ __forceinline__ void split4(const float4& x, uint4& hi, uint4& lo) {
  hi.x = cvt_tf32(x.x); lo.x = cvt_tf32(__fsub_rn(x.x, __uint_as_float(hi.x)));
  hi.y = cvt_tf32(x.y); lo.y = cvt_tf32(__fsub_rn(x.y, __uint_as_float(hi.y)));
  hi.z = cvt_tf32(x.z); lo.z = cvt_tf32(__fsub_rn(x.z, __uint_as_float(hi.z)));
  hi.w = cvt_tf32(x.w); lo.w = cvt_tf32(__fsub_rn(x.w, __uint_as_float(hi.w)));
}

template <int MODE, bool PAIR>
__device__ void run_split(const TcParams& p, uint8_t* smem, uint32_t sbase, uint32_t full0, uint32_t ld0,
                          uint32_t ctrl_u32, volatile int* abort) {
  using G = Geo<MODE, PAIR>;
  constexpr int kThr = kConvWarps * 32;
  constexpr int kBatchN = 8;
  const int ct = (int)threadIdx.x - Cfg<MODE, PAIR>::kConvWarp0 * 32;
  const int lane = threadIdx.x & 31;
  const uint32_t sm0 = smem_u32(smem);
  // K-major operand of `bytes` at `hi`: split each 16-byte piece in place,
  // the low parts at the same offset + kLoOff.
  auto split_k = [&](uint8_t* hi, int bytes) {
#pragma unroll 1
    for (int j0 = ct; j0 < bytes / 16; j0 += kThr * kBatchN) {
      float4 x[kBatchN];
#pragma unroll
      for (int u = 0; u < kBatchN; ++u) x[u] = *reinterpret_cast<const float4*>(hi + (j0 + u * kThr) * 16);
#pragma unroll
      for (int u = 0; u < kBatchN; ++u) {
        uint4 h, l;
        split4(x[u], h, l);
        uint8_t* q = hi + (j0 + u * kThr) * 16;
        *reinterpret_cast<uint4*>(q) = h;
        *reinterpret_cast<uint4*>(q + G::kLoOff) = l;
      }
    }
  };
  // MN-major operand of `boxes` 32 x 32 boxes loaded at hi + kLoOff (box j:
  // k-row r of 128 bytes holds mn 32j..32j+31, 16-byte chunk c at c ^ (r % 8)).
  // Written K-major: row mn of 128 bytes holds k 0..31, chunk c at c ^ (mn % 8).
  // Box j's K-major rows (mn 32j..) occupy exactly its own bytes, so boxes are
  // independent; within a pass of two boxes every thread reads its 4 x 4 block
  // before any thread writes.
  auto split_mn = [&](uint8_t* hi, int boxes) {
    uint8_t* lo = hi + G::kLoOff;
    const int kb4 = ct & 7, mb4 = (ct >> 3) & 7, half = ct >> 6;
#pragma unroll 1
    for (int pass = 0; pass < boxes / 2; ++pass) {
      const int box = 2 * pass + half;
      float4 x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 4 * kb4 + i;
        x[i] = *reinterpret_cast<const float4*>(lo + box * 4096 + r * 128 + ((mb4 ^ (r & 7)) << 4));
      }
      bar1_sync(kThr);
      const float t[4][4] = {{x[0].x, x[1].x, x[2].x, x[3].x}, {x[0].y, x[1].y, x[2].y, x[3].y},
                             {x[0].z, x[1].z, x[2].z, x[3].z}, {x[0].w, x[1].w, x[2].w, x[3].w}};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mn = 32 * box + 4 * mb4 + i;
        uint4 h, l;
        split4(make_float4(t[i][0], t[i][1], t[i][2], t[i][3]), h, l);
        const int off = mn * 128 + ((kb4 ^ (mn & 7)) << 4);
        *reinterpret_cast<uint4*>(hi + off) = h;
        *reinterpret_cast<uint4*>(lo + off) = l;
      }
    }
  };
  const int64_t total = total_tiles<MODE>(p);
  uint32_t stage = 0, phase = 0;
  Tile ti;
  int gh = 0;
  for (int64_t t = first_tile<MODE, PAIR>(p); get_tile<MODE, PAIR>(p, t, total, ti, gh); t += tile_step<MODE, PAIR>(p)) {
    for (int kb = 0; kb < p.num_kb; ++kb) {
      // One decision for all converter warps (they meet at named barriers).
      const bool ok = __all_sync(0xffffffffu, mbar_wait(ld0 + 8 * stage, phase, abort, p.status, p.timeout_ns));
      if (!bar1_and(ok, kThr)) return;
      uint8_t* st = smem + (sbase - sm0) + stage * G::kStageBytes;
      if (p.a_mn) split_mn(st, BM / 32);
      else split_k(st, G::kABytes);
      if (p.b_mn) split_mn(st + G::kABytes, G::kBRows / 32);
      else split_k(st + G::kABytes, G::kBBytes);
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          bulk_copy_to_cluster(mapa_shared(ctrl_u32 + kSignalOff, 0), ctrl_u32 + kSignalOff, kSignalBytes,
                               mapa_shared(full0 + 8 * stage, 0));
        else
          mbar_arrive(full0 + 8 * stage);
      }
      if (++stage == G::kStages) { stage = 0; phase ^= 1; }
    }
  }
}

// ------------------------------------------------------------------ epilogue

template <int MODE, bool PAIR>
__device__ void run_epilogue(const TcParams& p, const CUtensorMap* tmY, uint32_t tmem, uint32_t accf0, uint32_t acce0,
                             volatile int* abort, uint32_t* stage) {
  // Warp-private shared memory: QLinear column data (kQColWords) or the
  // output staging rows (kStageWords).
  int32_t* qcol = reinterpret_cast<int32_t*>(stage);
  uint32_t* stg = stage;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3, slice = (warp - kEpiWarp0) >> 2;
  constexpr int kCols = Cfg<MODE, PAIR>::kCols;
  // In a pair this CTA's TMEM lanes hold rows rank*128.. of the 256-row tile.
  const uint32_t rank = PAIR ? (cluster_ctarank() & 1) : 0;
  const int64_t row_off = (int64_t)rank * BM;
  // acc_empty lives in the leader CTA; every epilogue warp of the pair arrives there.
  auto release = [&](uint32_t buf) {
    if (lane == 0) {
      if (PAIR) mbar_arrive_cluster(mapa_shared(acce0 + 8 * buf, 0));
      else mbar_arrive(acce0 + 8 * buf);
    }
  };
  auto wait_full = [&](uint32_t buf, uint32_t aph) {
    return PAIR ? mbar_wait_cluster(accf0 + 8 * buf, aph, abort, p.status, p.timeout_ns)
                : mbar_wait(accf0 + 8 * buf, aph, abort, p.status, p.timeout_ns);
  };
  const int rloc = quad * 32 + lane;
  const uint32_t tlane = (uint32_t)(quad * 32) << 16;
  const int64_t total = total_tiles<MODE>(p);
  const int nseg = (p.num_kb + p.kb_per_seg - 1) / p.kb_per_seg;
  uint32_t seg = 0;
  Tile ti;
  float ys = 0.f, yz = 0.f, qmin = 0.f, qmax = 0.f, rys = 0.f;
  bool fast = false;
  if (MODE == kQLinear) {
    ys = load_scale(p.ys, 0, p.ys_f16);
    rys = __frcp_rn(ys);
    fast = fabsf(ys) >= 1.17549435e-38f && fabsf(ys) < 8.50705917e+37f;   // 2^-126 <= |ys| < 2^126
    yz = load_q8(p.yz, 0, p.y_signed);
    qmin = p.y_signed ? -128.f : 0.f;
    qmax = p.y_signed ? 127.f : 255.f;
  }
  int gh = 0;
  for (int64_t t = first_tile<MODE, PAIR>(p); get_tile<MODE, PAIR>(p, t, total, ti, gh); t += tile_step<MODE, PAIR>(p)) {
    const int rows_cta = PAIR ? max(0, min(BM, ti.rows - (int)row_off)) : ti.rows;
    const bool row_ok = rloc < rows_cta;
    const int64_t ncol0 = ti.n0 + slice * kCols;
    if (MODE == kQLinear) {
      // Column data of this warp's kCols columns (zero point, column sum,
      // scale), staged once per tile in a warp-private shared-memory slice.
      {
        const int64_t zboff = batch_off(p, p.zb.bstride, ti.batch);
        const int64_t sboff = batch_off(p, p.sb.bstride, ti.batch);
        const int32_t* cs = p.q_cs + (int64_t)ti.b_b * p.N;
        const int bshift = p.b_signed ? 0 : 128;
        for (int j = lane; j < kCols; j += 32) {
          const int64_t n = ncol0 + j;
          int32_t zbv = 0, csv = 0;
          float sbv = 0.f;
          if (n < p.N) {
            zbv = (int32_t)load_q8(p.zb.ptr, zboff + n * p.zb.vs, p.b_signed) - bshift;
            csv = cs[n];
            sbv = load_scale(p.sb.ptr, sboff + n * p.sb.vs, p.sb_f16);
          }
          qcol[j] = zbv;
          qcol[kCols + j] = csv;
          qcol[2 * kCols + j] = __float_as_int(sbv);
        }
        __syncwarp();
      }
      constexpr int kChunks = kCols / 32;
      int32_t acc[kChunks][32];
      for (int s = 0; s < nseg; ++s, ++seg) {
        const uint32_t buf = seg & 1, aph = (seg >> 1) & 1;
        if (!__all_sync(0xffffffffu, wait_full(buf, aph))) return;
        tc_fence_after();
        const uint32_t taddr = tmem + tlane + buf * BN + slice * kCols;
#pragma unroll
        for (int h = 0; h < 2 * kChunks; ++h) {     // 16 columns at a time: few live registers
          uint32_t r[16];
          tmem_ld16(taddr + h * 16, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int32_t v = __float2int_rn(__uint_as_float(r[j]));   // exact: |v| <= 2^24
            int32_t& a = acc[h >> 1][(h & 1) * 16 + j];
            a = s == 0 ? v : (int32_t)((uint32_t)a + (uint32_t)v);
          }
        }
        tc_fence_before();
        __syncwarp();
        release(buf);
      }
      if (row_ok) {
        const int64_t m = ti.m0 + row_off + rloc;
        const float sa = load_scale(p.sa.ptr, batch_off(p, p.sa.bstride, ti.batch) + m * p.sa.vs, p.sa_f16);
        const uint32_t za = (uint32_t)((int32_t)load_q8(p.za.ptr, batch_off(p, p.za.bstride, ti.batch) + m * p.za.vs,
                                                        p.a_signed) - (p.a_signed ? 0 : 128));
        const uint32_t rs = (uint32_t)p.q_rs[(int64_t)ti.a_b * p.M + m];
        // acc - zb'*rs - za'*cs + K*za'*zb' = acc - zb'*(rs - K*za') - za'*cs   (mod 2^32)
        const uint32_t rowterm = rs - (uint32_t)p.K * za;
        uint8_t* yrow = static_cast<uint8_t*>(p.y) + batch_off(p, p.y_bstride, ti.batch) + m * p.y_rs;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          const int64_t n = ncol0 + c * 32;
          if (n >= p.N) break;
          uint32_t packed[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int4 zb4 = *reinterpret_cast<const int4*>(qcol + c * 32 + 4 * q);
            const int4 cs4 = *reinterpret_cast<const int4*>(qcol + kCols + c * 32 + 4 * q);
            const int4 sb4 = *reinterpret_cast<const int4*>(qcol + 2 * kCols + c * 32 + 4 * q);
            const int32_t zbv[4] = {zb4.x, zb4.y, zb4.z, zb4.w};
            const int32_t csv[4] = {cs4.x, cs4.y, cs4.z, cs4.w};
            const int32_t sbv[4] = {sb4.x, sb4.y, sb4.z, sb4.w};
            uint32_t w = 0;
            bool any_slow = false;
            int32_t tot[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              tot[e] = (int32_t)((uint32_t)acc[c][4 * q + e] - (uint32_t)zbv[e] * rowterm - za * (uint32_t)csv[e]);
              bool sl;
              w |= requant_byte_fast(tot[e], sa, __int_as_float(sbv[e]), rys, fast, yz, qmin, qmax, &sl) << (8 * e);
              any_slow |= sl;
            }
            if (any_slow) {   // near a rounding boundary (or an unusual y_scale): divide
              w = 0;
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w |= requant_byte(tot[e], sa, __int_as_float(sbv[e]), ys, yz, qmin, qmax) << (8 * e);
            }
            packed[q] = w;
          }
          if (p.y_vec && n + 32 <= p.N) {
            uint4* dst = reinterpret_cast<uint4*>(yrow + n);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n + j < p.N) yrow[n + j] = (uint8_t)(packed[j >> 2] >> (8 * (j & 3)));
          }
        }
      }
      __syncwarp();   // every lane is done with qcol before the next tile restages it
    } else {
      const uint32_t buf = seg & 1, aph = (seg >> 1) & 1;
      ++seg;
      if (!__all_sync(0xffffffffu, wait_full(buf, aph))) return;
      tc_fence_after();
      // A pair's tail tile (one M = 128 MMA) leaves this CTA's 64 rows in
      // TMEM lanes 0-63 for the tile's columns 0-127 and again in lanes
      // 64-127 for columns 128-255, in TMEM columns 0-127: the warps of
      // column slices 0 and 1 hold it, the others only release the buffer.
      const bool tail = PAIR && p.pair_tail && ti.rows <= BM;
      if ((tail && slice * kCols >= BN / 2) || slice * kCols >= Geo<MODE, PAIR>::kTileN) {
        tc_fence_before();
        __syncwarp();
        release(buf);
        continue;
      }
      const int64_t roff = tail ? (int64_t)rank * (BM / 2) : row_off;
      const int rbase = tail ? (quad & 1) * 32 : quad * 32;
      const int rl = rbase + lane;
      const int rows_t = PAIR ? max(0, min(tail ? BM / 2 : BM, ti.rows - (int)roff)) : ti.rows;
      const bool rok = rl < rows_t;
      const int64_t ncol = ncol0 + (tail ? (int64_t)(quad >> 1) * (BN / 2) : 0);
      const uint32_t taddr0 = tmem + tlane + buf * BN + slice * kCols;
      // This thread's output row (kept even when the row is past the tile's
      // valid rows: it is then only shuffled around, never dereferenced).
      uint16_t* yrow;
      const uint16_t* crow = nullptr;
      if (is_grouped(MODE)) {
        const int64_t orow = rok ? p.g_rowlist[ti.a_row + roff + rl] : 0;
        yrow = static_cast<uint16_t*>(p.y) + orow * p.y_rs;
        if (p.c && rok) crow = static_cast<const uint16_t*>(p.c) + (int64_t)ti.g * p.c_gs;
      } else {
        const int64_t m = ti.m0 + roff + rl;
        yrow = static_cast<uint16_t*>(p.y) + batch_off(p, p.y_bstride, ti.batch) + m * p.y_rs;
        if (p.c && rok)
          crow = static_cast<const uint16_t*>(p.c) + batch_off(p, p.c_bstride, ti.batch) + m * p.c_rs;
      }
      if constexpr (MODE == kDense || MODE == kSkinny) {
        if (p.y_tma) {
          // The warp's 32 rows x 64 columns: into registers, release the
          // accumulator, then alpha/beta/C and the rounding to 16 bits.
          uint32_t r[2][32];
#pragma unroll
          for (int c = 0; c < 2; ++c) tmem_ld32(taddr0 + c * 32, r[c]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          release(buf);
          const int32_t yrow0 = (int32_t)(ti.m0 + roff + rbase), yb = (int32_t)batch_off(p, p.y_bc, ti.batch);
          // 32 columns at a time into the warp's 2 KB staging slice in the
          // 64-byte swizzled layout of the output's tensor map (row r's 16-byte
          // chunk c at c ^ ((r / 2) % 4): conflict-free row-wise writes), then
          // one tensor store of the 32 x 32 box; before the slice is written
          // again the previous store must have read it.  The store clips rows
          // and columns past M and N.
          const uint32_t sbox = smem_u32(stage);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[h][j]);
            if (crow) add_c32(p, crow, ncol + 32 * h, v);
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              sts128(sbox + (uint32_t)lane * 64 + (((uint32_t)q ^ ((uint32_t)(lane >> 1) & 3u)) << 4),
                     make_uint4(pack2(v[8 * q], v[8 * q + 1], p.out_f16), pack2(v[8 * q + 2], v[8 * q + 3], p.out_f16),
                                pack2(v[8 * q + 4], v[8 * q + 5], p.out_f16),
                                pack2(v[8 * q + 6], v[8 * q + 7], p.out_f16)));
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0 && rbase < rows_t) {
              tma_store_3d(tmY, sbox, (int32_t)(ncol + 32 * h), yrow0, yb);
              bulk_commit();
            }
          }
          continue;
        }
      }
      // The warp's columns, 64 at a time (two tcgen05.ld of 32); the
      // accumulator is released once its last columns are in registers.
#pragma unroll 1
      for (int q64 = 0; q64 < kCols / 64; ++q64) {
        const uint32_t taddr = taddr0 + q64 * 64;
        uint32_t r[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld32(taddr + c * 32, r[c]);
        tmem_ld_wait();
        if (q64 == kCols / 64 - 1) {
          tc_fence_before();
          __syncwarp();
          release(buf);
        }
        // Each 32-column chunk (64 bytes of each of the warp's 32 rows) is staged
        // through the warp's shared-memory slice (16-byte pieces XOR-swizzled by
        // row pair, so both the row-wise writes and the column-wise reads are
        // bank-conflict free) and written back so that each warp store covers 8
        // rows x 64 bytes of whole 32-byte sectors.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t n = ncol + q64 * 64 + 32 * h;
          if (n >= p.N) break;
          if constexpr (MODE == kTF32) {
            // fp32 output: each thread writes its row's 32 values (128 bytes).
            if (rok) {
              const int64_t m = ti.m0 + roff + rl;
              float* yf = static_cast<float*>(p.y) + batch_off(p, p.y_bstride, ti.batch) + m * p.y_rs;
              const float* cf = p.c ? static_cast<const float*>(p.c) + batch_off(p, p.c_bstride, ti.batch) +
                                          m * p.c_rs
                                    : nullptr;
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                v[j] = p.alpha * __uint_as_float(r[h][j]);
                if (cf && n + j < p.N) v[j] = __fmaf_rn(p.beta, cf[(n + j) * p.c_cs], v[j]);
              }
              if (p.y_vec && n + 32 <= p.N) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  *reinterpret_cast<float4*>(yf + n + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2],
                                                                           v[4 * q + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (n + j < p.N) yf[n + j] = v[j];
              }
            }
            continue;
          }
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = p.alpha * __uint_as_float(r[h][j]);
          if (crow) add_c32(p, crow, n, v);
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) w[j] = pack2(v[2 * j], v[2 * j + 1], p.out_f16);
          if (p.y_vec && n + 32 <= p.N) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(stg + lane * 16 + ((q ^ ((lane >> 1) & 3)) * 4)) =
                  make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i * 8 + (lane >> 2), pc = lane & 3;
              const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * 16 + ((pc ^ ((rr >> 1) & 3)) * 4));
              uint16_t* dst = reinterpret_cast<uint16_t*>(
                  __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(yrow), rr));
              if (rbase + rr < rows_t) *reinterpret_cast<uint4*>(dst + n + pc * 8) = val;
            }
            __syncwarp();
          } else if (rok) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n + j < p.N) yrow[n + j] = (uint16_t)((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ few-row epilogue (kSkinny)

// Each CTA of a cluster has accumulated its share of the tile's k-blocks in
// TMEM columns 0..255; rows 0..63 (lanes of quadrants 0 and 1) hold the A'
// rows.  The epilogue warps of those quadrants copy them, fp32, into the
// CTA's own shared memory (the drained ring) as [64 rows][kSkinnyPitch]
// (a padded pitch, so the row-wise 16-byte writes of a warp are conflict-free).
constexpr int kSkinnyPitch = BN + 4;   // floats per partial-sum row

template <int MODE, bool PAIR>
__device__ void run_skinny_partial(const TcParams& p, uint32_t tmem, uint32_t accf0, volatile int* abort,
                                   uint32_t part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3, slice = (warp - kEpiWarp0) >> 2;
  if (quad >= 2) return;
  if (!__all_sync(0xffffffffu, mbar_wait(accf0, 0, abort, p.status, p.timeout_ns))) return;
  tc_fence_after();
  const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(slice * 64);
  uint32_t r[2][32];
#pragma unroll
  for (int c = 0; c < 2; ++c) tmem_ld32(taddr + c * 32, r[c]);
  tmem_ld_wait();
  const uint32_t row = part + (uint32_t)((quad * 32 + lane) * kSkinnyPitch * 4) + (uint32_t)(slice * 64 * 4);
#pragma unroll
  for (int q = 0; q < 16; ++q)
    sts128(row + q * 16, make_uint4(r[q >> 3][4 * (q & 7)], r[q >> 3][4 * (q & 7) + 1], r[q >> 3][4 * (q & 7) + 2],
                                    r[q >> 3][4 * (q & 7) + 3]));
}

// Once every CTA's partial sums are in its shared memory, CTA r of the cluster
// finishes columns [r * 256 / split, (r + 1) * 256 / split) of the tile: each
// item is one row and 8 columns; its epilogue threads add the split partials
// in rank order (the other CTAs' through distributed shared memory), apply
// alpha, beta * C and the rounding to 16 bits, and store 16 bytes.
template <int MODE, bool PAIR>
__device__ void run_skinny_reduce(const TcParams& p, uint32_t part) {
  constexpr int kThr = Cfg<MODE, PAIR>::kEpiWarps * 32;
  const int et = (int)threadIdx.x - kEpiWarp0 * 32;
  const int64_t total = total_tiles<MODE>(p);
  Tile ti;
  int gh = 0;
  if (!get_tile<MODE, PAIR>(p, first_tile<MODE, PAIR>(p), total, ti, gh)) return;
  const int rank = (int)(cluster_ctarank());
  const int width = BN / p.split, groups = width / 8;
  const uint16_t* cbase =
      p.c ? static_cast<const uint16_t*>(p.c) + batch_off(p, p.c_bstride, ti.batch) : nullptr;
  uint16_t* ybase = static_cast<uint16_t*>(p.y) + batch_off(p, p.y_bstride, ti.batch);
  for (int item = et; item < ti.rows * groups; item += kThr) {
    const int row = item / groups;
    const int col = rank * width + (item - row * groups) * 8;   // within the tile
    const int64_t m = ti.m0 + row, n = ti.n0 + col;
    if (n >= p.N) continue;
    const uint32_t src = part + (uint32_t)(row * kSkinnyPitch * 4) + (uint32_t)(col * 4);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.f;
    for (int rk = 0; rk < p.split; ++rk) {
      const uint32_t a = mapa_shared(src, (uint32_t)rk);
      const float4 f0 = lds128_cluster(a), f1 = lds128_cluster(a + 16);
      v[0] += f0.x; v[1] += f0.y; v[2] += f0.z; v[3] += f0.w;
      v[4] += f1.x; v[5] += f1.y; v[6] += f1.z; v[7] += f1.w;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = p.alpha * v[j];
      if (cbase && n + j < p.N) v[j] = __fmaf_rn(p.beta, unpack16(cbase[m * p.c_rs + (n + j) * p.c_cs], p.out_f16), v[j]);
    }
    uint16_t* yrow = ybase + m * p.y_rs;
    const uint4 w = make_uint4(pack2(v[0], v[1], p.out_f16), pack2(v[2], v[3], p.out_f16),
                               pack2(v[4], v[5], p.out_f16), pack2(v[6], v[7], p.out_f16));
    if (p.y_vec && n + 8 <= p.N) {
      *reinterpret_cast<uint4*>(yrow + n) = w;
    } else {
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (n + j < p.N) yrow[n + j] = (uint16_t)((j & 1) ? (ws[j >> 1] >> 16) : (ws[j >> 1] & 0xFFFFu));
    }
  }
}

// ------------------------------------------------------------------ kernel

template <int MODE, bool PAIR>
__global__ void __launch_bounds__(Cfg<MODE, PAIR>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmZ,
                   const TcParams p) {
  using G = Geo<MODE, PAIR>;
  constexpr int S = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  // [ring][epilogue slices][control block][kGroupedQ staging ring]
  uint8_t* ctrl = smem_raw + (sbase - raw) + G::kRingBytes + Cfg<MODE, PAIR>::kEpiBytes;
  const uint32_t cbase = sbase + G::kRingBytes + Cfg<MODE, PAIR>::kEpiBytes;
  const uint32_t full0 = cbase, empty0 = cbase + 8 * S, accf0 = cbase + 16 * S;
  const uint32_t acce0 = accf0 + 16, drain = acce0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 16 * S + 40);
  volatile int* abort = reinterpret_cast<volatile int*>(ctrl + 16 * S + 44);
  const uint32_t qfull0 = cbase + 16 * S + 48, qempty0 = qfull0 + 8 * kQStages;   // kGroupedQ only
  const uint32_t qbase = sbase + Cfg<MODE, PAIR>::kQOff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // kGroupedQ: a stage is full once the leader's producer has armed it and
    // both CTAs' A bytes and converter signals (below) have landed.
    // kTF32 on one CTA: the converter warps' arrivals fill the stage.
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, (MODE == kTF32 && !PAIR) ? kConvWarps : 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    if (MODE == kTF32)
      for (int s = 0; s < S; ++s) mbar_init(qfull0 + 8 * s, 1);
    if (MODE == kGroupedQ)
      for (int s = 0; s < kQStages; ++s) {
        mbar_init(qfull0 + 8 * s, 1);
        mbar_init(qempty0 + 8 * s, kConvWarps);
      }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, (PAIR ? 2 : 1) * Cfg<MODE, PAIR>::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  // A pair's barriers must be initialised in both CTAs before either CTA
  // signals the other's.
  if (PAIR) cluster_sync();
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched with programmatic stream serialization, this grid may start while
  // the previous kernel on the stream is finishing: the set-up above overlaps
  // its tail, and nothing below touches global memory before it completes.
  pdl_wait();
  if constexpr (MODE == kDense || MODE == kTF32) pdl_trigger();
  const uint32_t rank = PAIR ? (cluster_ctarank() & 1) : 0;

  if (warp == 0) {
    if (lane == 0)
      run_producer<MODE, PAIR>(&tmA, &tmB, &tmS, &tmZ, p, sbase, full0, empty0, qbase, qfull0, qempty0, abort);
  } else if (warp == 1) {
    if (lane == 0) {
      if (rank == 0) run_mma<MODE, PAIR>(p, sbase, tmem, full0, empty0, accf0, acce0, drain, abort);
      else mbar_wait_teardown(drain, 0, p.teardown_ns);   // the leader's last commit reaches this CTA too
    }
  } else if (warp < Cfg<MODE, PAIR>::kConvWarp0) {
    uint32_t* stage = reinterpret_cast<uint32_t*>(smem_raw + (sbase - raw) + G::kRingBytes) +
                      (warp - kEpiWarp0) * Cfg<MODE, PAIR>::kWarpWords;
    if constexpr (MODE == kSkinny) run_skinny_partial<MODE, PAIR>(p, tmem, accf0, abort, sbase);
    else run_epilogue<MODE, PAIR>(p, &tmZ, tmem, accf0, acce0, abort, stage);
    // Every tensor store has read its box before the CTA can exit.
    if (p.y_tma && lane == 0) bulk_wait_all();
  } else if (MODE == kGroupedQ) {
    if (p.w4) run_convert<MODE, PAIR, true>(p, smem_raw, sbase, full0, qbase, qfull0, qempty0, cbase, abort);
    else run_convert<MODE, PAIR, false>(p, smem_raw, sbase, full0, qbase, qfull0, qempty0, cbase, abort);
  } else if (MODE == kTF32) {
    run_split<MODE, PAIR>(p, smem_raw, sbase, full0, qfull0, cbase, abort);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (MODE == kSkinny) {
    // Every CTA's partial sums are in its shared memory; each CTA adds the
    // cluster's partials for its share of the columns, and no CTA leaves
    // (taking its shared memory with it) until all have read them.
    cluster_sync();
    if (warp >= kEpiWarp0) run_skinny_reduce<MODE, PAIR>(p, sbase);
    cluster_sync();
  }
  // Neither CTA of a pair may leave (or free tensor memory) while the other
  // can still signal its barriers or its MMAs can still touch its memory.
  if (PAIR) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int64_t gcd64(int64_t a, int64_t b) {
  while (b) { const int64_t t = a % b; a = b; b = t; }
  return a;
}

// Per-device values cached on first use; host threads may race to fill an
// entry, which is harmless (they compute the same value), so atomics suffice.
int sm_count() {
  static std::atomic<int> counts[128];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) return 148;
  int c = counts[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    if (c <= 0) c = 148;
    counts[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

}  // namespace

// A 16-bit operand of rows `mn_len` (M of A, N of B) and depth `k_len`, with
// element strides `mn_stride` / `k_stride` and batch strides `bstride` over the
// broadcast batch `bm`, described as a 3-D tensor map (contiguous dimension,
// other matrix dimension, batch).  The batch coordinate of batch index b is
// sum_d i_d * bc[d]; false when the layout does not fit TMA.
bool plan_operand(const void* ptr, int dtype, int64_t mn_len, int64_t k_len, int64_t mn_stride, int64_t k_stride,
                  const BatchMap& bm, const int64_t* bstride, int box_mn, OperandPlan* out) {
  auto encode = encode_fn();
  if (!encode || !ptr || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
  if (mn_len < 1 || k_len < 1 || mn_len > 0x7fffffffLL || k_len > 0x7fffffffLL) return false;
  int64_t unit = 0;
  for (int d = 0; d < bm.nb; ++d)
    if (bm.shape[d] > 1 && bstride[d] != 0) unit = gcd64(unit, bstride[d]);
  int64_t nbat = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) out->bc[d] = 0;
  if (unit != 0) {
    if (unit % (dtype == MM_F32 ? 4 : 8)) return false;
    int64_t maxc = 0;
    for (int d = 0; d < bm.nb; ++d)
      if (bm.shape[d] > 1 && bstride[d] != 0) {
        out->bc[d] = bstride[d] / unit;
        maxc += (bm.shape[d] - 1) * out->bc[d];
      }
    nbat = maxc + 1;
    if (nbat > 0x7fffffffLL) return false;
  }
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  const cuuint32_t estr[3] = {1, 1, 1};
  if (dtype == MM_F32) {
    // fp32 (three-tf32 products): K-major tiles as 32-element (128-byte) k
    // boxes of box_mn rows; MN-major tiles as 32 x 32 boxes, transposed to
    // K-major by the splitting converters.
    if (unit % 4) return false;
    if (k_stride == 1 && mn_stride > 0 && mn_stride % 4 == 0) {
      out->mn_major = 0;
      dims[0] = (cuuint64_t)k_len; dims[1] = (cuuint64_t)mn_len;
      strides[0] = (cuuint64_t)mn_stride * 4;
      box[0] = 32; box[1] = (cuuint32_t)box_mn;
    } else if (mn_stride == 1 && k_stride > 0 && k_stride % 4 == 0) {
      out->mn_major = 1;
      dims[0] = (cuuint64_t)mn_len; dims[1] = (cuuint64_t)k_len;
      strides[0] = (cuuint64_t)k_stride * 4;
      box[0] = 32; box[1] = 32;
    } else {
      return false;
    }
    dims[2] = (cuuint64_t)nbat;
    box[2] = 1;
    strides[1] = unit != 0 ? (cuuint64_t)unit * 4 : (cuuint64_t)(((strides[0] * dims[1]) + 15) & ~15ull);
    if (strides[0] >= (1ull << 40) || strides[1] >= (1ull << 40)) return false;
    return encode(&out->map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const CUtensorMapDataType dt = dtype == MM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (k_stride == 1 && mn_stride > 0 && mn_stride % 8 == 0) {
    out->mn_major = 0;
    dims[0] = (cuuint64_t)k_len; dims[1] = (cuuint64_t)mn_len; dims[2] = (cuuint64_t)nbat;
    strides[0] = (cuuint64_t)mn_stride * 2;
    box[0] = 64; box[1] = (cuuint32_t)box_mn; box[2] = 1;
  } else if (mn_stride == 1 && k_stride > 0 && k_stride % 8 == 0) {
    out->mn_major = 1;
    dims[0] = (cuuint64_t)mn_len; dims[1] = (cuuint64_t)k_len; dims[2] = (cuuint64_t)nbat;
    strides[0] = (cuuint64_t)k_stride * 2;
    box[0] = 64; box[1] = 64; box[2] = 1;
  } else {
    return false;
  }
  strides[1] = unit != 0 ? (cuuint64_t)unit * 2 : (cuuint64_t)(((strides[0] * dims[1]) + 15) & ~15ull);
  if (strides[0] >= (1ull << 40) || strides[1] >= (1ull << 40)) return false;
  const CUresult r = encode(&out->map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool plan_plain_3d(const void* ptr, int elem_bytes, int64_t d0, int64_t d1, int64_t d2, int64_t s1, int64_t s2,
                   int box0, int box1, OperandPlan* out) {
  auto encode = encode_fn();
  if (!encode || !ptr || (reinterpret_cast<uintptr_t>(ptr) & 15)) return false;
  if (d0 < 1 || d1 < 1 || d2 < 1 || d0 > 0x7fffffffLL || d1 > 0x7fffffffLL || d2 > 0x7fffffffLL) return false;
  if (s1 <= 0 || s2 <= 0 || (s1 & 15) || (s2 & 15) || s1 >= (1ll << 40) || s2 >= (1ll << 40)) return false;
  if ((box0 * elem_bytes) % 16 || box0 > 256 || box1 > 256) return false;
  const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  if (elem_bytes != 1 && elem_bytes != 2) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  const cuuint64_t strides[2] = {(cuuint64_t)s1, (cuuint64_t)s2};
  const cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  out->mn_major = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) out->bc[d] = 0;
  return encode(&out->map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t make_idesc(int f16, int a_mn, int b_mn, bool pair) {
  return make_idesc_rows(f16, a_mn, b_mn, pair ? 2 * BM : BM);   // a pair's MMA covers both CTAs' rows
}

uint32_t make_idesc_rows(int f16, int a_mn, int b_mn, uint32_t m) { return make_idesc_mn(f16, a_mn, b_mn, m, BN); }

uint32_t make_idesc_mn(int f16, int a_mn, int b_mn, uint32_t m, uint32_t n) {
  return (1u << 4)                              // D: fp32
         | ((f16 ? 0u : 1u) << 7)               // A: f16 (0) / bf16 (1)
         | ((f16 ? 0u : 1u) << 10)              // B: f16 (0) / bf16 (1)
         | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16)
         | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// kind::tf32: A and B tf32 (format 2), D fp32, both K-major.
uint32_t make_idesc_tf32(bool pair) {
  const uint32_t m = pair ? 2 * BM : BM;
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) | ((m >> 4) << 24);
}

namespace {
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;   // 2 s
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitNs};
}  // namespace

void tc_set_wait_limit_ns(unsigned long long ns) { g_wait_limit_ns.store(ns ? ns : kDefaultWaitNs); }

void init_params(TcParams* p) {
  memset(p, 0, sizeof(*p));
  p->timeout_ns = g_wait_limit_ns.load();
  p->teardown_ns = kDefaultWaitNs;
  p->alpha = 1.f;
  p->kb_per_seg = 1 << 30;
}

namespace {

// Clusters of 2 CTAs (one CTA per SM) that can be resident at once for a
// kernel, queried once per device (0 if none).
template <int MODE>
int max_pair_clusters() {
  static std::atomic<int> cache[128];   // value + 1 once known (0: not yet queried)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128) return 0;
  const int known = cache[dev].load(std::memory_order_relaxed);
  if (known > 0) return known - 1;
  {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(sm_count() & ~1));
    cfg.blockDim = dim3(Cfg<MODE, true>::kThreads);
    cfg.dynamicSmemBytes = Cfg<MODE, true>::kSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(tc_gemm_kernel<MODE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<MODE, true>::kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<MODE, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[dev].store(n + 1, std::memory_order_relaxed);
    return n;
  }
}

template <int MODE, bool PAIR>
mm_status launch_kernel(const OperandPlan& a, const OperandPlan& b, const CUtensorMap& ms, const CUtensorMap& mz,
                        const TcParams& p_in, int64_t work, cudaStream_t stream) {
  constexpr int kSmem = Cfg<MODE, PAIR>::kSmem, kThreadsM = Cfg<MODE, PAIR>::kThreads;
  TcParams p = p_in;
  if (MODE != kDense) p.y_tma = 0;
  if (cudaFuncSetAttribute(tc_gemm_kernel<MODE, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
      cudaSuccess)
    return MM_ERR_CUDA;
  // Every launch allows programmatic stream serialization: the kernel's
  // set-up (barriers, tensor memory, descriptor prefetch) may overlap the
  // previous kernel's last blocks; it waits for that kernel before any
  // global-memory access.  Clustered launches add the cluster size.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreadsM);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  if constexpr (MODE == kSkinny) {
    // One cluster per 256-column tile; its CTAs split the tile's k-blocks:
    // the largest power of two up to 8 that keeps tiles x split within the
    // SMs and gives every CTA at least one k-block.
    const int sms = sm_count();
    int split = 8;
    while (split > 1 && (work * split > sms || split > p.num_kb)) split >>= 1;
    p.split = split;
    if (work * split > 0x7fffffffLL) return MM_ERR_UNSUPPORTED;
    attr[1].val.clusterDim.x = (unsigned)split;
    cfg.gridDim = dim3((unsigned)(work * split));
    cfg.numAttrs = 2;
  } else if constexpr (!PAIR) {
    const int sms = sm_count();
    cfg.gridDim = dim3((unsigned)(work < sms ? (work > 0 ? work : 1) : sms));
    cfg.numAttrs = 1;
  } else {
    // One persistent pair per resident cluster slot: a pair that could not be
    // resident would only start after the others finish.
    const int slots = max_pair_clusters<MODE>();
    if (slots <= 0) return MM_ERR_UNSUPPORTED;
    const int clusters = (int)(work < slots ? (work > 0 ? work : 1) : slots);
    attr[1].val.clusterDim.x = 2;
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE, PAIR>, a.map, b.map, ms, mz, p) == cudaSuccess ? MM_OK
                                                                                                      : MM_ERR_CUDA;
}

}  // namespace

mm_status launch_tc(int mode, bool pair, const OperandPlan& a, const OperandPlan& b, TcParams& p,
                    cudaStream_t stream, const OperandPlan* s, const OperandPlan* z) {
  p.a_mn = a.mn_major;
  p.b_mn = b.mn_major;
  for (int d = 0; d < kMaxBatchDims; ++d) { p.a_bc[d] = a.bc[d]; p.b_bc[d] = b.bc[d]; }
  const int kb_elems = mode == kTF32 ? 32 : BK;   // k-block: one 128-byte row of the operand type
  p.num_kb = (int)((p.K + kb_elems - 1) / kb_elems);
  int64_t work = 0;
  if (!is_grouped(mode)) {
    const int64_t rows = pair ? 2 * BM : BM;
    const int64_t cols = BN;
    p.mt = (p.M + rows - 1) / rows;
    p.nt = (p.N + cols - 1) / cols;
    p.tiles = p.mt * p.nt * p.bm.count;
    if (p.tiles >= (1ll << 31) || p.mt * p.nt >= (1ll << 31)) return MM_ERR_UNSUPPORTED;
    const uint32_t per_batch = (uint32_t)(p.mt * p.nt);
    const uint32_t bands = (uint32_t)((p.mt + kGroupM - 1) / kGroupM);
    p.fd_per_batch = make_fastdiv(per_batch);
    p.fd_band = make_fastdiv((uint32_t)(kGroupM * p.nt));
    p.last_band = bands - 1;
    p.fd_last_h = make_fastdiv((uint32_t)(p.mt - (int64_t)(bands - 1) * kGroupM));
    work = p.tiles;
  } else {
    work = sm_count();          // the tile count is known only on the device
  }
  for (int d = 0; d < kMaxBatchDims; ++d) {
    if (p.bm.shape[d] >= (1ll << 31)) return MM_ERR_UNSUPPORTED;
    p.fd_bshape[d] = make_fastdiv((uint32_t)(p.bm.shape[d] > 0 ? p.bm.shape[d] : 1));
  }
  if (p.kb_per_seg > p.num_kb) p.kb_per_seg = p.num_kb > 0 ? p.num_kb : 1;
  if (p.kb_per_q < 1) p.kb_per_q = 1 << 30;
  // Only kGroupedQ reads the scale and zero-point maps; other modes get A's map
  // in those (unused) parameters.
  const CUtensorMap& ms = s ? s->map : a.map;
  const CUtensorMap& mz = z ? z->map : (s ? s->map : a.map);
  switch (mode) {
    case kDense:
      return pair ? launch_kernel<kDense, true>(a, b, ms, mz, p, work, stream)
                  : launch_kernel<kDense, false>(a, b, ms, mz, p, work, stream);
    case kSkinny:   // single CTAs only
      return pair ? MM_ERR_UNSUPPORTED : launch_kernel<kSkinny, false>(a, b, ms, mz, p, work, stream);
    case kGrouped:
      return pair ? launch_kernel<kGrouped, true>(a, b, ms, mz, p, work, stream)
                  : launch_kernel<kGrouped, false>(a, b, ms, mz, p, work, stream);
    case kQLinear:   // single CTAs only: the product is bound by its epilogue
      return pair ? MM_ERR_UNSUPPORTED : launch_kernel<kQLinear, false>(a, b, ms, mz, p, work, stream);
    case kTF32:
      return pair ? launch_kernel<kTF32, true>(a, b, ms, mz, p, work, stream)
                  : launch_kernel<kTF32, false>(a, b, ms, mz, p, work, stream);
    case kGroupedQ:  // CTA pairs only
      if (!pair || !s) return MM_ERR_UNSUPPORTED;
      return launch_kernel<kGroupedQ, true>(a, b, ms, mz, p, work, stream);
    default:
      return MM_ERR_UNSUPPORTED;
  }
}

// CTA pairs halve the operand bytes each SM must take in per MMA cycle, which
// is what bounds long-K products; short-K (output-bound) products run better
// on single CTAs, whose smaller tiles keep more epilogues in flight.
bool use_pair(int64_t M, int64_t K) { return M > BM && K >= kPairMinK; }

// Grouped pairs: a group's last row tile with at most 128 rows runs as an
// M = 128 MMA, so pairs pad each group no more than single CTAs do; they need
// groups of 256 rows on average to have full pair tiles to gain on.
bool grouped_q_pairs_available() { return max_pair_clusters<kGroupedQ>() > 0; }

bool use_grouped_pair(int64_t rows, int64_t G, int64_t K) {
  return K >= kPairMinK && rows >= 2 * BM * G && max_pair_clusters<kGrouped>() > 0;
}

int sm_count_public() { return sm_count(); }

// ------------------------------------------------------------------ MatMul / Gemm

namespace {

// The 16-bit output Y [batch.., M, N] (row stride y.rs, unit column stride) as
// a tensor map of 32 x 32 boxes, 64-byte swizzled, for the TMA-store
// epilogue: sets p->y_tma and p->y_bc when Y's layout fits TMA.
void plan_output(const GemmArgs& g, TcParams* p, OperandPlan* y) {
  p->y_tma = 0;
  if (g.dtype != MM_BF16 && g.dtype != MM_F16) return;
  if (g.y.cs != 1 || g.y.rs < g.N || g.M < 1 || g.N < 1) return;
  auto encode = encode_fn();
  if (!encode || (reinterpret_cast<uintptr_t>(g.y.ptr) & 15)) return;
  const int64_t pitch = g.M == 1 ? (g.N + 7) / 8 * 8 : g.y.rs;   // one row: any valid pitch
  if (pitch % 8 || g.M > 0x7fffffffLL || g.N > 0x7fffffffLL) return;
  int64_t unit = 0;
  for (int d = 0; d < g.bm.nb; ++d)
    if (g.bm.shape[d] > 1 && g.y.bstride[d] != 0) unit = gcd64(unit, g.y.bstride[d]);
  int64_t nbat = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) y->bc[d] = 0;
  if (unit != 0) {
    if (unit % 8) return;
    int64_t maxc = 0;
    for (int d = 0; d < g.bm.nb; ++d)
      if (g.bm.shape[d] > 1 && g.y.bstride[d] != 0) {
        y->bc[d] = g.y.bstride[d] / unit;
        maxc += (g.bm.shape[d] - 1) * y->bc[d];
      }
    nbat = maxc + 1;
    if (nbat > 0x7fffffffLL) return;
  }
  const cuuint64_t dims[3] = {(cuuint64_t)g.N, (cuuint64_t)g.M, (cuuint64_t)nbat};
  const cuuint64_t strides[2] = {(cuuint64_t)pitch * 2,
                                 unit != 0 ? (cuuint64_t)unit * 2 : (cuuint64_t)((pitch * 2 * g.M + 15) & ~15ll)};
  if (strides[0] >= (1ull << 40) || strides[1] >= (1ull << 40)) return;
  const cuuint32_t box[3] = {32u, 32u, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = g.dtype == MM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (encode(&y->map, dt, 3, const_cast<void*>(g.y.ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return;
  y->mn_major = 0;
  p->y_tma = 1;
  for (int d = 0; d < kMaxBatchDims; ++d) p->y_bc[d] = y->bc[d];
}

bool plan_dense(const GemmArgs& g, bool pair, OperandPlan* a, OperandPlan* b) {
  if (g.dtype != MM_BF16 && g.dtype != MM_F16 && g.dtype != MM_F32) return false;
  if (g.M < 1 || g.N < 2 || g.K < 1) return false;
  if (g.y.cs != 1) return false;
  // A single row of A' (a vector-matrix product: M = 1, MatMul's promoted 1-D
  // A) with unit stride along k is a K-major tile whatever its row stride
  // (0 for a promoted vector, 1 for A stored [K, 1]), which only row 0 uses:
  // give the tensor map a row pitch TMA accepts.  The other 127 rows of the
  // tile read the fill value and are never stored.
  const int64_t vec = g.dtype == MM_F32 ? 4 : 8;
  const int64_t a_rs = (g.M == 1 && g.a.cs == 1) ? (g.K + vec - 1) / vec * vec : g.a.rs;
  if (!plan_operand(g.a.ptr, g.dtype, g.M, g.K, a_rs, g.a.cs, g.bm, g.a.bstride, BM, a)) return false;
  if (!plan_operand(g.b.ptr, g.dtype, g.N, g.K, g.b.cs, g.b.rs, g.bm, g.b.bstride, pair ? BN / 2 : BN, b)) return false;
  return true;
}

}  // namespace

bool tc_gemm_supported(const GemmArgs& g) {
  OperandPlan a, b;
  return plan_dense(g, false, &a, &b);
}

mm_status launch_tc_gemm(const GemmArgs& g, unsigned* status, cudaStream_t stream) {
  if (!status) return MM_ERR_UNSUPPORTED;
  TcParams p;
  init_params(&p);
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.bm = g.bm;
  p.out_f16 = g.dtype == MM_F16;
  p.out_f32 = g.dtype == MM_F32;
  const int64_t vec = p.out_f32 ? 4 : 8;      // elements per 16 bytes
  p.y = const_cast<void*>(g.y.ptr);
  for (int d = 0; d < kMaxBatchDims; ++d) { p.y_bstride[d] = g.y.bstride[d]; p.c_bstride[d] = g.c.bstride[d]; }
  p.y_rs = g.y.rs;
  p.y_vec = (reinterpret_cast<uintptr_t>(g.y.ptr) % 16 == 0) && (g.y.rs % vec == 0);
  for (int d = 0; d < g.bm.nb; ++d) p.y_vec = p.y_vec && (g.y.bstride[d] % vec == 0);
  p.alpha = g.alpha;
  p.beta = g.beta;
  if (g.c.ptr) {
    p.c = g.c.ptr;
    p.c_rs = g.c.rs;
    p.c_cs = g.c.cs;
    p.c_vec = g.c.cs == 1 && (reinterpret_cast<uintptr_t>(g.c.ptr) % 16 == 0) && (g.c.rs % vec == 0);
    for (int d = 0; d < g.bm.nb; ++d) p.c_vec = p.c_vec && (g.c.bstride[d] % vec == 0);
  }
  p.status = status;
  // A few rows (at most 64, K-major A) against fewer 256-column tiles than
  // SMs: the few-row configuration splits each tile's k-blocks over a cluster
  // so that every SM streams B'.
  if (!p.out_f32 && g.M <= BM / 2 && ((g.N + BN - 1) / BN) * g.bm.count < sm_count()) {
    OperandPlan a, b;
    const int64_t vec = 8;
    const int64_t a_rs = (g.M == 1 && g.a.cs == 1) ? (g.K + vec - 1) / vec * vec : g.a.rs;
    if (g.N >= 2 && g.y.cs == 1 &&
        plan_operand(g.a.ptr, g.dtype, g.M, g.K, a_rs, g.a.cs, g.bm, g.a.bstride, BM / 2, &a) && !a.mn_major &&
        plan_operand(g.b.ptr, g.dtype, g.N, g.K, g.b.cs, g.b.rs, g.bm, g.b.bstride, BN, &b)) {
      p.idesc = make_idesc_mn(p.out_f16, 0, b.mn_major, BM, BN);
      return launch_tc(kSkinny, false, a, b, p, stream);
    }
  }
  // CTA pairs (256-row tiles) for long-K products with more than one row tile;
  // one CTA per tile otherwise, or if no pair can be placed.
  for (int attempt = use_pair(g.M, g.K) ? 0 : 1; attempt < 2; ++attempt) {
    const bool pair = attempt == 0;
    OperandPlan a, b, a_tail;
    if (!plan_dense(g, pair, &a, &b)) return MM_ERR_UNSUPPORTED;
    p.idesc = p.out_f32 ? make_idesc_tf32(pair) : make_idesc(p.out_f16, a.mn_major, b.mn_major, pair);
    // 16-bit pairs with K-major A run a last row tile of at most 128 rows as
    // one M = 128 MMA fed by 64 rows of A per CTA.
    p.pair_tail = pair && !p.out_f32 && !a.mn_major &&
                  plan_operand(g.a.ptr, g.dtype, g.M, g.K, g.a.rs, g.a.cs, g.bm, g.a.bstride, BM / 2, &a_tail);
    if (p.pair_tail) p.idesc_tail = make_idesc_rows(p.out_f16, 0, b.mn_major, BM);
    OperandPlan ymap;
    plan_output(g, &p, &ymap);
    const mm_status st = launch_tc(p.out_f32 ? kTF32 : kDense, pair, a, b, p, stream,
                                   p.pair_tail ? &a_tail : nullptr, p.y_tma ? &ymap : nullptr);
    if (st != MM_ERR_UNSUPPORTED || !pair) return st;
  }
  return MM_ERR_UNSUPPORTED;
}

}  // namespace qg
