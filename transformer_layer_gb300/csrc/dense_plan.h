// Geometry and work plan of the tensor-core tile GEMMs, shared by the kernels
// (dense_impl.cuh), the host planner (dense.cu) and the CPU replay of the
// planner's invariants (tests/dense_plan_check.cpp): host and device code,
// no CUDA runtime calls (the one device query the planner needs, how many
// clusters of a size fit on the GPU at once, is passed in).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "internal.h"
#include "work_split.h"

// (the qualifiers the kernels were built and measured with)
#if defined(__CUDACC__)
#define DS_PLAN_HD __host__ __device__ inline
#else
#define DS_PLAN_HD inline
#endif

namespace ds {

constexpr int kDenseWTiles = 4;      // int8 weights: fp16 W tiles (in TMEM) the converters fill ahead of the MMAs
constexpr int kDenseWTileCols = 64;  // TMEM columns of one fp16 W tile: 128 rows x 128 codes of K
constexpr int kDenseMaxIssuers = 2;  // MMA-issuing warps: warp 1 and (two issuers) the last warp
constexpr int kDenseMaxStagesDev = 8;  // ring depth limit (the host plan uses at most this)
constexpr int kDenseMaxStages = kDenseMaxStagesDev;
constexpr size_t kDenseMinSmem = 120 * 1024;  // two tile CTAs never share an SM (nor its TMEM)

// One ring stage: W [KC/64 atoms][128 rows][128 B], then X [KC/64][NTOK][128 B]
// (and, for bf16, X lo the same), each part on a 1024-byte boundary.  With
// int8 weights a stage holds the TMA copy of the codes, [128 rows][KC bytes]
// (KC = 128, 128-byte swizzle), then X, then the scales of the stage's rows:
// the aligned block of 8 groups along K that holds the stage's groups,
// [128 rows][8 fp16] (a TMA box is at least 16 bytes wide).  The codes' fp16
// dequantisation goes to one of kDenseWTiles W tiles in tensor memory, the
// MMAs' A operand, so it costs neither ring depth nor shared-memory traffic.
constexpr int kDenseScaleGroups = 8;  // int8: scale groups per row in a stage's scale box
DS_PLAN_HD size_t dense_w_bytes(int kc) { return (size_t)128 * kc * 2; }
DS_PLAN_HD size_t dense_x_bytes(int ntok, int kc) { return (size_t)ntok * kc * 2; }
DS_PLAN_HD size_t dense_scale_bytes(bool i8) { return i8 ? (size_t)128 * kDenseScaleGroups * 2 : 0; }
DS_PLAN_HD size_t dense_stage_bytes(int ntok, int kc, bool split, bool i8 = false) {
  return (i8 ? (size_t)128 * kc : dense_w_bytes(kc)) + (split ? 2 : 1) * dense_x_bytes(ntok, kc) + dense_scale_bytes(i8);
}
// MMA issuers of a tile GEMM.  One thread issues a tcgen05.mma about every
// 50-120 cycles whatever NTOK, so at small NTOK a chunk's MMAs (8, bf16 16)
// take longer to issue than its bytes take to stream; two issuers split the
// chunks.  Each issuer must see every phase of the barriers it waits on:
// fp16 / bf16 issuers wait on the ring's stages, so the ring needs an even
// depth (issuer i then owns the stages st % 2 == i); int8 issuers wait on
// their own W tiles.  Up to 64 token rows (decode: at 128, a prompt chunk's
// tile, the MMAs run long enough for one issuer).  (Four int8 issuers were slower: a 21st warp
// caps every thread at 80 registers, since each SM sub-partition's register
// file serves its quarter of the warps.)
DS_PLAN_HD int dense_issuers(int ntok, int stages, bool i8) {
  if (i8) return kDenseMaxIssuers;
  return (ntok <= 64 && stages % 2 == 0) ? kDenseMaxIssuers : 1;
}
// Tensor memory columns: two accumulators of NTOK columns per MMA issuer,
// then (int8) the fp16 W tiles; an allocation is a power of two of at least 32.
DS_PLAN_HD uint32_t dense_tmem_cols(int ntok, int nis, bool i8) {
  const uint32_t need = (uint32_t)(2 * nis * ntok) + (i8 ? (uint32_t)(kDenseWTiles * kDenseWTileCols) : 0u);
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c;
}

// The work plan of one tile GEMM (y[M][N] = X[M][K] W[N][K]^T) on num_sms SMs
// with max_smem bytes of shared memory per CTA; false if the shape has none.
// dense_cluster_capacity(size): clusters of `size` tile CTAs the GPU holds at
// once.
template <typename ClusterCapacity>
inline bool dense_make_plan_t(ActKind ak, int N, int K, int M, int num_sms, int max_smem, DensePlan* plan, bool i8,
                              ClusterCapacity&& dense_cluster_capacity) {
  if (N <= 0 || K <= 0 || M < 1 || (N % 128) != 0 || (K % 128) != 0 || num_sms < 1) return false;
  const bool split = (ak == ActKind::BF16);
  if (i8 && split) return false;  // int8 tiles take fp16 activations
  DensePlan p;
  p.i8 = i8 ? 1 : 0;
  p.row_tiles = N / 128;
  int ntok = (M + 15) / 16 * 16;
  // Token tiles of up to 128 rows; prompt chunks of 256 rows and more take
  // 256 with fp16 (MMA N = 256: half the weight re-reads per FLOP) and 192
  // with bf16 (its hi/lo operand: a 64 KB stage, three in the ring).  int8: up
  // to 64 rows, so that the four accumulators (two per MMA issuer) and the
  // four fp16 W tiles fit the 512 tensor-memory columns.
  const int ntok_max = i8 ? 64 : (M >= 256 ? (split ? 192 : 256) : 128);
  if (ntok > ntok_max) ntok = ntok_max;
  p.ntok = ntok;
  p.tok_tiles = (M + ntok - 1) / ntok;
  p.kc = i8 ? 128 : ((ntok > 64 || K % 128 != 0) ? 64 : 128);
  GemvPlan& w = p.ws;
  w.tiles = p.row_tiles * p.tok_tiles;
  w.chunk_k = p.kc;
  w.nt = 1;
  w.nblk = 1;
  p.kchunks = K / p.kc;
  const size_t SB = (dense_stage_bytes(ntok, p.kc, split, i8) + 1023) & ~(size_t)1023;
  const size_t fixed = 1024 + 8 * (3 * kDenseMaxStages + 6 + 2 * kDenseWTiles) + 16;
  if ((size_t)max_smem < fixed + 2 * SB) return false;
  // The plan for KS slices per tile along K (uneven: a cluster's slices share
  // the K chunks as evenly as they go); false if it does not fit.
  auto make = [&](int KS, bool uneven, DensePlan* out) -> bool {
    DensePlan q = p;
    GemvPlan& w = q.ws;
    w.KS = KS;
    w.C = uneven ? (q.kchunks + KS - 1) / KS : q.kchunks / KS;  // (uneven: the longest slice)
    w.K_S = w.C * q.kc;
    w.units = w.tiles * KS;
    // More tiles than SMs with several token tiles (prompt chunks): whole
    // tiles only (no split-K fix-ups of large tiles), handed out round-robin,
    // so that the CTAs running at the same time take the token tiles of the
    // same weight rows and read those weights from DRAM once between them.
    // (With one token tile, e.g. N = 20480 at decode, the few leftover tiles
    // are split.)
    const bool many = w.tiles > num_sms && q.tok_tiles > 1;
    ws_distribute(w, num_sms, /*one_unit_each=*/true, /*force_whole=*/many);
    w.interleave = many ? 1 : 0;
    size_t s = ((size_t)max_smem - fixed) / SB;
    if (s > (size_t)kDenseMaxStages) s = kDenseMaxStages;
    if (s > (size_t)w.C * 2 && w.C >= 2) s = (size_t)w.C * 2;  // no deeper than the work
    if (s < 2) s = 2;
    // fp16 / bf16 at up to 64 token rows run two MMA issuers, each owning
    // the ring stages of one parity: an even depth (int8 issuers own W tiles)
    if (!i8 && ntok <= 64 && s >= 3 && (s & 1)) s -= 1;
    q.stages = (int)s;
    size_t smem = fixed + s * SB;
    if (smem < kDenseMinSmem) smem = kDenseMinSmem;
    if (smem > (size_t)max_smem) return false;
    q.smem = smem;
    w.stages = q.stages;
    w.smem = smem;
    // K-sliced tiles with one slice per CTA: the slices of a tile run as one
    // cluster and are summed on chip (no partial sums through global
    // memory); each CTA's partial tile is staged in its idle ring.
    q.cluster = (KS > 1 && w.grid == w.units && w.q == 1 && w.R == 0 &&
                 (size_t)q.stages * SB >= (size_t)ntok * 128 * 4) ? KS : 1;
    if (uneven && q.cluster != KS) return false;  // uneven slices only run as clusters
    *out = q;
    return true;
  };
  // With at least ~60 % as many tiles as SMs every CTA takes one whole tile
  // (no split-K: a fix-up costs more than the idle SMs).  With fewer, each
  // tile is cut into KS slices along K (a power of two, at most 8, dividing
  // the chunks), one whole unit per CTA, as many as the SMs hold; when those
  // run as clusters, as many slices as the SMs hold (at most 8, the portable
  // cluster size) if all the clusters fit at once, of unequal length if need
  // be -- 40 tiles (N = 5120) take 120 SMs rather than 80.  With more tiles
  // than SMs, the even split over CTAs (whole units first, leftover chunks
  // spread).
  int KS = 1;
  if (p.ws.tiles * 5 < num_sms * 3)
    while (KS < 8 && p.ws.tiles * KS * 2 <= num_sms && p.kchunks % (KS * 2) == 0) KS *= 2;
  if (!make(KS, false, &p)) return false;
  if (p.cluster > 1) {
    // (only a size whose clusters all fit on the device at once: a second
    // wave would cost far more than the idle SMs)
    int KSu = num_sms / p.ws.tiles;
    if (KSu > 8) KSu = 8;
    if (KSu > p.kchunks) KSu = p.kchunks;
    DensePlan q;
    if (KSu > KS && dense_cluster_capacity(KSu) >= p.ws.tiles && make(KSu, p.kchunks % KSu != 0, &q)) p = q;
  }
  *plan = p;
  return true;
}

}  // namespace ds
