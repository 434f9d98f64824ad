// Skinny-GEMM region kernels: y[M][N] = x[M][K] W[N][K]^T for M = 1..64 batch
// rows, with the region's prologue fused in front of the GEMM and its
// epilogue fused at the GEMM reduction boundary.
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持".
//   §3 intro: a vector-matrix / skinny matrix-matrix GEMM built so that more
//     operations fuse at its reduction boundary.
//   §3.1: keep each CTA's access pattern fixed along the fused chain; CTAs
//     only meet through global memory, at the reduction boundary.
//   §3.2: region 1 (LayerNorm + QKV + bias), region 3 (FF + LayerNorm + bias +
//     residual + GeLU), region 4 (bias + residual).
//   §3.3: shared memory stages data between reductions and element-wise work;
//     warp-level instructions reduce partial results.
//   §5.2: int8 weights are dequantised inside the GEMM, without int8 hardware.
//
// GB300 design (not the pages'):
//  * Weights stream from HBM exactly once: a copy warp issues one TMA tensor
//    copy per chunk (16 weight rows x up to 2 KB, 128-byte swizzle) into a
//    shared-memory ring of up to 8 stages, from two lanes so the issue rate
//    never limits the stream.  It never waits for the previous kernel
//    (griddepcontrol): the ring fills during the previous kernel's tail, and
//    once its own copies are issued it asks L2 to prefetch the next GEMV's
//    first chunks.  One CTA per SM.
//  * 8 MMA warps run the 16 x 8 x 16 tensor-core MMA (weights are the 16-row A
//    side, batch rows the 8-column B side): at M <= 8 it needs ~5x fewer
//    instructions per weight byte than CUDA-core FMAs.  Each warp takes one
//    step of every chunk (up to 4 blocks x 16 bytes per lane and row); the
//    fragment loads are conflict-free (ring_layout.h).
//  * Work: a unit is 16 weight rows x one K slice, a chunk is 8 warp steps of
//    it.  Each CTA owns q whole units; the leftover units' chunks are spread
//    evenly over all CTAs (balanced to within one chunk), and the last CTA to
//    contribute to a row tile (acquire-release arrival counter, no waiting)
//    sums the partials in fixed order.  Leftover chunks are processed first
//    so that these fix-ups happen early, not at the kernel's tail.
//  * Two epilogue warps take alternate segments' per-warp partial tiles
//    through shared memory (four buffers at small batch, named barriers),
//    reduce them and run the region epilogue or the split-K fix-up, whose
//    global-memory round trips then overlap each other and the stream.
//
// K permutation: a lane of the MMA fragment owns k pairs {2c, 2c+1} and
// {2c+8, 2c+9} of a 16-wide k block.  Each lane instead reads 8 contiguous
// weights (16 bytes) of a ring row and the B operand is read with the same
// permutation, so the dot product is unchanged while every shared-memory
// read is a 128-bit access.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ring_layout.h"
#include "work_split.h"

namespace ds {

constexpr int kProducers = 8;             // MMA warps (each "produces" a partial tile per segment)
constexpr int kEpiWarp = kProducers;      // warps 8, 9: reduction, epilogue, split-K fix-up
constexpr int kEpiWarps = 2;              // (alternate segments: fix-up latencies overlap)
constexpr int kTmaWarp0 = kProducers + kEpiWarps; // warp 10: TMA tensor copies of the weights
constexpr int kTmaWarps = 1;
constexpr int kIssueLanes = 2;            // lanes of the TMA warp that issue copies
constexpr int kL2Lookahead = 16;          // chunks of the next GEMV prefetched into L2 per CTA
constexpr int kGemvThreads = (kProducers + kEpiWarps + kTmaWarps) * 32;
constexpr int kMaxStages = 8;             // weight ring depth (chunks in flight per CTA)

// Named barriers (0 is __syncthreads, unused here).
constexpr int kBarStage = 1;  // the 8 streaming warps
constexpr int kBarFull = 2;   // 2 .. 5: segment partials written (streaming -> epilogue)
constexpr int kBarEmpty = 6;  // 6 .. 9: segment partials consumed (epilogue -> streaming)

// Segment buffers between the MMA warps and the epilogue warp: four at small
// NT, so the MMA warps run up to four segments ahead of a slow split-K fix-up.
template <int NT> struct SegBufs {
  static constexpr int n = NT <= 2 ? 4 : 2;
};

__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

template <WKind WK> struct Geom {
  static constexpr int BLK_K = (WK == WKind::I8) ? 64 : 32;  // k per 16-byte lane load
  static constexpr int PAD = (WK == WKind::I8) ? 8 : 32;     // x row pad, elements (bank spread)
};

template <int NT> struct SmemLayout {
  // Weight ring: `stages` chunks, each 16 rows of chunk_k weights in the
  // swizzled [segment][row][128 bytes] layout of ring_layout.h, plus, for
  // int8, their [16][chunk_k/64] fp16 scales; stages start on 1024-byte
  // boundaries (the swizzle pattern repeats every 1024 bytes).
  // Then the x slice [M][K_S + pad] (hi, and lo for bf16), the segment
  // buffers [2][8 warps][NT][16][8] fp32, tile values [16][8 NT], LN mean /
  // rstd [64] and the full / empty mbarriers of the ring.
  static __host__ __device__ size_t chunk_bytes(int chunk_k, int esize) { return (size_t)16 * chunk_k * esize; }
  static __host__ __device__ size_t scale_bytes(int chunk_k, bool i8) {
    return i8 ? (size_t)16 * (chunk_k / 32) * 2 : 0;  // room for the finest grouping (32)
  }
  static __host__ __device__ size_t stage_bytes(int chunk_k, int esize, bool i8) {
    return (chunk_bytes(chunk_k, esize) + scale_bytes(chunk_k, i8) + 1023) & ~(size_t)1023;
  }
  static __host__ __device__ size_t xs_bytes(int M, int K_S, int pad, bool split) {
    const size_t b = (size_t)(split ? 2 : 1) * M * (K_S + pad) * 2;
    return (b + 15) & ~(size_t)15;
  }
  static __host__ __device__ size_t red_floats() { return (size_t)SegBufs<NT>::n * kProducers * NT * 128; }
  // Everything except the weight ring and its barriers.
  static __host__ __device__ size_t fixed(int M, int K_S, int pad, bool split) {
    return xs_bytes(M, K_S, pad, split) + 4 * (red_floats() + kEpiWarps * 16 * 8 * NT + 2 * 64);
  }
  static __host__ __device__ size_t total(int M, int K_S, int pad, bool split, int stages, int chunk_k,
                                          int esize, bool i8) {
    return (size_t)stages * stage_bytes(chunk_k, esize, i8) + fixed(M, K_S, pad, split) +
           (size_t)16 * stages;
  }
};

template <typename MT> struct Mma;
template <> struct Mma<__half> {
  static __device__ __forceinline__ void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    mma_f16(d, a0, a1, a2, a3, b0, b1);
  }
};
template <> struct Mma<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    mma_bf16(d, a0, a1, a2, a3, b0, b1);
  }
};

constexpr int kMaxBlk = 4;  // k-blocks per warp step, at most

struct Slot {
  uint4 a[2 * kMaxBlk];            // [row r (g, g+8)][block]
  unsigned short sc[2 * kMaxBlk];  // int8 only: fp16 scale bits, [row r][block]
};

// Shared-memory carve-up of a GEMV CTA: the weight ring (S stages of SB
// bytes), the staged x slice (xs_cap bytes), the segment buffers, tile
// values, LayerNorm mean / rstd and the ring's full / empty mbarriers.
struct GemvSmem {
  unsigned char* ring;
  size_t SB;
  int S;
  unsigned char* xs;
  float* red;
  float* tileval;
  float* s_mean;
  float* s_rstd;
  uint64_t* mbar;
  __device__ __forceinline__ uint32_t full_bar(int i) const { return smem_u32(mbar + i); }
  __device__ __forceinline__ uint32_t empty_bar(int i) const { return smem_u32(mbar + S + i); }
};

template <int NT>
__device__ __forceinline__ GemvSmem gemv_carve(unsigned char* base, int S, size_t SB, size_t xs_cap) {
  GemvSmem m;
  base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(base) + 1023) & ~(uintptr_t)1023);
  m.ring = base;
  m.SB = SB;
  m.S = S;
  m.xs = base + (size_t)S * SB;
  m.red = reinterpret_cast<float*>(m.xs + xs_cap);
  m.tileval = m.red + SmemLayout<NT>::red_floats();
  m.s_mean = m.tileval + kEpiWarps * 16 * 8 * NT;
  m.s_rstd = m.s_mean + 64;
  m.mbar = reinterpret_cast<uint64_t*>(m.s_rstd + 64);
  return m;
}

// A role's position in the weight ring: stage, parity, chunks passed, and
// whether one of its waits has timed out (then it waits no more).
struct RingPos {
  int st = 0;
  uint32_t ph = 0;
  int n = 0;
  bool dead = false;
  __device__ __forceinline__ void advance(int S) {
    ++n;
    if (++st == S) {
      st = 0;
      ph ^= 1;
    }
  }
};

__device__ __forceinline__ void gemv_init_ring(const GemvSmem& sm) {
  for (int i = 0; i < sm.S; ++i) {
    mbar_init(sm.full_bar(i), kTmaWarps);
    mbar_init(sm.empty_bar(i), kProducers);
  }
  mbar_init_fence();
}

// TMA warp `tw`: copies this CTA's chunks of one GEMV phase into the ring.
template <Region R, WKind WK, typename ACT, int NT>
__device__ void gemv_tma_phase(const RegionArgs& a, const GemvPlan& P, const GemvSmem& sm, RingPos& rp, int tw,
                               uint64_t pol) {
  using G_ = Geom<WK>;
  using L = SmemLayout<NT>;
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;  // hi + lo bf16 operand
  constexpr int ROWS = 8 * NT;
  constexpr bool kStats = (R == Region::OprojRes || R == Region::FfnDown);
  constexpr int ESZ = (WK == WKind::I8) ? 1 : 2;  // weight bytes
  constexpr bool kI8 = (WK == WKind::I8);
  (void)kSplit; (void)ROWS; (void)kStats; (void)kI8;
  const int M = a.M, N = a.N, K = a.K;
  const int K_S = P.K_S;
  const int XS = K_S + G_::PAD;  // x row stride, elements
  const int S = sm.S;
  const size_t SB = sm.SB;
  const size_t RB = L::chunk_bytes(P.chunk_k, ESZ);  // offset of a stage's int8 scales
  unsigned char* ring = sm.ring;
  ACT* xs_hi = reinterpret_cast<ACT*>(sm.xs);
  ACT* xs_lo = xs_hi + M * XS;
  float* red = sm.red;
  float* tileval = sm.tileval;
  float* s_mean = sm.s_mean;
  float* s_rstd = sm.s_rstd;
  (void)xs_lo; (void)red; (void)tileval; (void)s_mean; (void)s_rstd; (void)RB; (void)XS; (void)N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  (void)g; (void)c; (void)tid; (void)warp;
  const int tiles = P.tiles, C = P.C;
  const int cta = blockIdx.x, G = gridDim.x;
  (void)tiles; (void)C;
  long long ra, rb;
  ws_left_range(P, cta, G, &ra, &rb);
  const int dp_b = cta * P.q;
  const int nchunks = (int)(rb - ra) + P.q * C;
  (void)nchunks; (void)K; (void)S; (void)SB; (void)ring; (void)M; (void)K_S;
  const uint32_t tx = (uint32_t)(RB + (kI8 ? 16 * (P.chunk_k / a.qgroup) * 2 : 0));
  const int qshift = 31 - __clz(a.qgroup);  // group lengths are powers of two (64, 128)
  (void)tw;
  // Lanes 0 .. kIssueLanes-1 each issue every kIssueLanes-th chunk: one
  // issuing thread cannot keep a CTA's copies in flight at HBM rate (it spends
  // most of its time between an empty-slot wait and the next issue).
  Cursor q;
  ws_cursor_init(q, P, ra, rb, dp_b);
  for (int i = 0; i < lane && i < kIssueLanes && i < nchunks; ++i) ws_cursor_next(q, P, dp_b);
  bool dead = rp.dead;
  for (int j = 0; j < nchunks; j += kIssueLanes) {
    if (lane < kIssueLanes && j + lane < nchunks) {
      // ring slot of chunk rp.n + lane (kIssueLanes < S, so at most one wrap)
      int st = rp.st + lane;
      uint32_t ph = rp.ph;
      if (st >= S) {
        st -= S;
        ph ^= 1;
      }
      if (rp.n + lane >= S && !dead) dead = !mbar_wait(sm.empty_bar(st), ph ^ 1, a.status);
      const int kg = q.s * K_S + q.kc * P.chunk_k;  // first k of the chunk
      const int row0 = q.t * 16;
      const uint32_t stage = smem_u32(ring + (size_t)st * SB);
      mbar_arrive_expect_tx(sm.full_bar(st), tx);
      tma_load_3d(stage, a.tmap_w, 0, row0, kg * ESZ / kSwizzleBytes, sm.full_bar(st), pol);
      if constexpr (kI8) tma_load_2d(stage + (uint32_t)RB, a.tmap_s, kg >> qshift, row0, sm.full_bar(st), pol);
      for (int i = 0; i < kIssueLanes; ++i) ws_cursor_next(q, P, dp_b);
    }
    __syncwarp();
    const int adv = nchunks - j < kIssueLanes ? nchunks - j : kIssueLanes;
    for (int i = 0; i < adv; ++i) rp.advance(S);
  }
  rp.dead = __any_sync(0xffffffffu, dead);
}

// Copy warp: asks L2 to prefetch the first `max_chunks` chunks (and int8
// scales) that CTA blockIdx.x streams in the GEMV of plan P.
template <WKind WK>
__device__ void gemv_l2_prefetch_phase(const void* tmap_w, const void* tmap_s, const GemvPlan& P,
                                       int max_chunks, int qgroup) {
  constexpr int ESZ = (WK == WKind::I8) ? 1 : 2;
  const int cta = blockIdx.x, G = P.grid;
  if ((threadIdx.x & 31) != 0 || cta >= G) return;
  long long ra, rb;
  ws_left_range(P, cta, G, &ra, &rb);
  const int dp_b = cta * P.q;
  int nchunks = (int)(rb - ra) + P.q * P.C;
  if (nchunks > max_chunks) nchunks = max_chunks;
  const int qshift = 31 - __clz(qgroup);  // group lengths are powers of two
  Cursor q;
  ws_cursor_init(q, P, ra, rb, dp_b);
  for (int j = 0; j < nchunks; ++j) {
    const int kg = q.s * P.K_S + q.kc * P.chunk_k;
    tma_prefetch_3d(tmap_w, 0, q.t * 16, kg * ESZ / kSwizzleBytes);
    if (WK == WKind::I8) tma_prefetch_2d(tmap_s, kg >> qshift, q.t * 16);
    ws_cursor_next(q, P, dp_b);
  }
}

// MMA warps: LayerNorm prologue, x staging and the chunk loop of one GEMV
// phase; each finished segment's per-warp tiles go to the epilogue warp.
// `seg` counts segments across phases (it picks the segment buffer).
// XB: input groups a thread loads together while staging x.
template <Region R, WKind WK, typename ACT, int NT, int XB = 2>
__device__ void gemv_mma_phase(const RegionArgs& a, const GemvPlan& P, const GemvSmem& sm, RingPos& rp,
                               int& seg) {
  using G_ = Geom<WK>;
  using L = SmemLayout<NT>;
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;  // hi + lo bf16 operand
  constexpr int ROWS = 8 * NT;
  constexpr bool kStats = (R == Region::OprojRes || R == Region::FfnDown);
  constexpr int ESZ = (WK == WKind::I8) ? 1 : 2;  // weight bytes
  constexpr bool kI8 = (WK == WKind::I8);
  (void)kSplit; (void)ROWS; (void)kStats; (void)kI8;
  const int M = a.M, N = a.N, K = a.K;
  const int K_S = P.K_S;
  const int XS = K_S + G_::PAD;  // x row stride, elements
  const int S = sm.S;
  const size_t SB = sm.SB;
  const size_t RB = L::chunk_bytes(P.chunk_k, ESZ);  // offset of a stage's int8 scales
  unsigned char* ring = sm.ring;
  ACT* xs_hi = reinterpret_cast<ACT*>(sm.xs);
  ACT* xs_lo = xs_hi + M * XS;
  float* red = sm.red;
  float* tileval = sm.tileval;
  float* s_mean = sm.s_mean;
  float* s_rstd = sm.s_rstd;
  (void)xs_lo; (void)red; (void)tileval; (void)s_mean; (void)s_rstd; (void)RB; (void)XS; (void)N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  (void)g; (void)c; (void)tid; (void)warp;
  const int tiles = P.tiles, C = P.C;
  const int cta = blockIdx.x, G = gridDim.x;
  (void)tiles; (void)C;
  long long ra, rb;
  ws_left_range(P, cta, G, &ra, &rb);
  const int dp_b = cta * P.q;
  const int nchunks = (int)(rb - ra) + P.q * C;
  (void)nchunks; (void)K; (void)S; (void)SB; (void)ring; (void)M; (void)K_S;
  const int step_k = P.nblk * G_::BLK_K;
  // A fragments of this warp's step of the chunk in ring stage `st`.
  // Fragment row g reads weight rows wr and wr + 8 of the tile; block blk of
  // this warp's step is byte o_step + 64 blk of each row (ring_layout.h).
  const int wr = rl_row(g);
  const int o_step = warp * step_k * ESZ + 16 * c;
  unsigned lofs[kMaxBlk];
#pragma unroll
  for (int blk = 0; blk < kMaxBlk; ++blk) lofs[blk] = rl_offset(wr, o_step + 64 * blk);
  // int8: scale groups per chunk row, and the group of block blk (groups of
  // 64 or 128 codes: uniform over the block, whose codes one MMA sums)
  const int gpc = P.chunk_k / a.qgroup;
  const int qshift = 31 - __clz(a.qgroup);  // group lengths are powers of two (64, 128)
  const int sofs = wr * gpc;
  const int sg0 = warp * step_k + 16 * c;
  auto load = [&](int st, Slot& sl) {
    const unsigned char* stage = ring + (size_t)st * SB;
#pragma unroll
    for (int blk = 0; blk < kMaxBlk; ++blk) {
      if (blk < P.nblk) {
        // row wr + 8 is 8 rows (1024 bytes) further in the same segment, same swizzle
        sl.a[blk] = *reinterpret_cast<const uint4*>(stage + lofs[blk]);
        sl.a[kMaxBlk + blk] = *reinterpret_cast<const uint4*>(stage + lofs[blk] + 8 * kSwizzleBytes);
      }
    }
    if constexpr (kI8) {
      const unsigned short* sc = reinterpret_cast<const unsigned short*>(stage + RB) + sofs;
#pragma unroll
      for (int blk = 0; blk < kMaxBlk; ++blk) {
        if (blk < P.nblk) {
          const int gi = (sg0 + 64 * blk) >> qshift;
          sl.sc[blk] = sc[gi];
          sl.sc[kMaxBlk + blk] = sc[8 * gpc + gi];
        }
      }
    }
  };
  // B operand of n-tile nt.  Columns n >= M of the product are never used,
  // so those lanes read row M - 1 instead of branching around the load.
  auto load_x = [&](const ACT* base, int nt, int off) -> uint4 {
    const int n = min(nt * 8 + g, M - 1);
    return *reinterpret_cast<const uint4*>(base + n * XS + off);
  };
  // Independent accumulator sets (NA) break the MMA dependency chain of a
  // warp step at small NT; set (blk, half) -> (2 blk + half) % NA.
  constexpr int NA = NT == 1 ? 4 : (NT == 2 ? 2 : 1);
  auto compute = [&](const Slot& sl, int kl, float (&acc)[NA][NT][4]) {
#pragma unroll
    for (int blk = 0; blk < kMaxBlk; ++blk) {
      if (blk >= P.nblk) break;
      float(&a0)[NT][4] = acc[blk % NA];
      float(&a1)[NT][4] = acc[blk % NA];
      if constexpr (WK == WKind::I8) {
        uint32_t lo0[4], hi0[4], lo1[4], hi1[4];
        const uint4 B0 = sl.a[blk], B1 = sl.a[kMaxBlk + blk];
        const uint32_t w0[4] = {B0.x, B0.y, B0.z, B0.w};
        const uint32_t w1[4] = {B1.x, B1.y, B1.z, B1.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if constexpr (kSplit) {
            i8x4_to_bf162x2(w0[m], lo0[m], hi0[m]);
            i8x4_to_bf162x2(w1[m], lo1[m], hi1[m]);
          } else {
            i8x4_to_half2x2(w0[m], lo0[m], hi0[m]);
            i8x4_to_half2x2(w1[m], lo1[m], hi1[m]);
          }
        }
        const float s0 = __half2float(__ushort_as_half(sl.sc[blk]));
        const float s1 = __half2float(__ushort_as_half(sl.sc[kMaxBlk + blk]));
        const int off = kl + blk * 64 + 16 * c;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (nt * 8 >= M) break;
          // two chains of MMAs over the 64 codes of the block, then one scale
          float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
          const uint4 X0 = load_x(xs_hi, nt, off), X1 = load_x(xs_hi, nt, off + 8);
          const uint32_t xw[8] = {X0.x, X0.y, X0.z, X0.w, X1.x, X1.y, X1.z, X1.w};
#pragma unroll
          for (int m = 0; m < 4; ++m)
            Mma<ACT>::run((m & 1) ? t1 : t0, lo0[m], lo1[m], hi0[m], hi1[m], xw[2 * m], xw[2 * m + 1]);
          if constexpr (kSplit) {
            const uint4 Y0 = load_x(xs_lo, nt, off), Y1 = load_x(xs_lo, nt, off + 8);
            const uint32_t yw[8] = {Y0.x, Y0.y, Y0.z, Y0.w, Y1.x, Y1.y, Y1.z, Y1.w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
              Mma<ACT>::run((m & 1) ? t1 : t0, lo0[m], lo1[m], hi0[m], hi1[m], yw[2 * m], yw[2 * m + 1]);
          }
          a0[nt][0] += (t0[0] + t1[0]) * s0;
          a0[nt][1] += (t0[1] + t1[1]) * s0;
          a0[nt][2] += (t0[2] + t1[2]) * s1;
          a0[nt][3] += (t0[3] + t1[3]) * s1;
        }
      } else {
        const uint4 A0 = sl.a[blk], A1 = sl.a[kMaxBlk + blk];
        const int off = kl + blk * 32 + 8 * c;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (nt * 8 >= M) break;
          const uint4 X = load_x(xs_hi, nt, off);
          Mma<ACT>::run(a0[nt], A0.x, A1.x, A0.y, A1.y, X.x, X.y);
          Mma<ACT>::run(a1[nt], A0.z, A1.z, A0.w, A1.w, X.z, X.w);
          if constexpr (kSplit) {
            const uint4 Y = load_x(xs_lo, nt, off);
            Mma<ACT>::run(a0[nt], A0.x, A1.x, A0.y, A1.y, Y.x, Y.y);
            Mma<ACT>::run(a1[nt], A0.z, A1.z, A0.w, A1.w, Y.z, Y.w);
          }
        }
      }
    }
  };
  // Stage x[:, slice s] (rows < M) into shared memory, the region prologue
  // fused in.  Each thread first loads kXB groups of 8 inputs, then converts
  // and stores them, so the loads of a batch are in flight together.
  auto stage = [&](int s) {
    constexpr int kXB = XB;
    constexpr bool kLn = (R == Region::LnQkv || R == Region::FfnUp);
    const int k0 = s * K_S;
    const int cpr = K_S / 8;
    const int total = M * cpr;
    for (int base = tid; base < total; base += kXB * kProducers * 32) {
      uint4 raw[kXB][2], gam[kXB], bet[kXB];
#pragma unroll
      for (int b = 0; b < kXB; ++b) {
        const int idx = base + b * kProducers * 32;
        if (idx >= total) continue;  // (continue, not break: keeps the arrays in registers)
        const int n = idx / cpr;
        const int kc = (idx - n * cpr) * 8;
        if constexpr (R == Region::LnQkv) {
          raw[b][0] = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.x_act) + (size_t)n * K + k0 + kc);
        } else {
          const float* src = a.x_f32 + (size_t)n * K + k0 + kc;
          raw[b][0] = *reinterpret_cast<const uint4*>(src);
          raw[b][1] = *reinterpret_cast<const uint4*>(src + 4);
        }
        if constexpr (kLn) {
          gam[b] = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_g) + k0 + kc);
          bet[b] = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_b) + k0 + kc);
        }
      }
#pragma unroll
      for (int b = 0; b < kXB; ++b) {
        const int idx = base + b * kProducers * 32;
        if (idx >= total) continue;
        const int n = idx / cpr;
        const int kc = (idx - n * cpr) * 8;
        float v[8];
        if constexpr (R == Region::LnQkv) {
          const uint32_t uw[4] = {raw[b][0].x, raw[b][0].y, raw[b][0].z, raw[b][0].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 xv = Act<ACT>::unpack2(uw[i]);
            v[2 * i] = xv.x;
            v[2 * i + 1] = xv.y;
          }
        } else {
          const float4 p0 = *reinterpret_cast<const float4*>(&raw[b][0]);
          const float4 p1 = *reinterpret_cast<const float4*>(&raw[b][1]);
          v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
          v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
        }
        if constexpr (kLn) {
          const uint32_t gw[4] = {gam[b].x, gam[b].y, gam[b].z, gam[b].w},
                         bw[4] = {bet[b].x, bet[b].y, bet[b].z, bet[b].w};
          const float mu = s_mean[n], rs = s_rstd[n];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 gv = Act<ACT>::unpack2(gw[i]), bv = Act<ACT>::unpack2(bw[i]);
            v[2 * i] = (v[2 * i] - mu) * rs * gv.x + bv.x;
            v[2 * i + 1] = (v[2 * i + 1] - mu) * rs * gv.y + bv.y;
          }
        }
        uint4 hi;
        hi.x = Act<ACT>::pack2(v[0], v[1]);
        hi.y = Act<ACT>::pack2(v[2], v[3]);
        hi.z = Act<ACT>::pack2(v[4], v[5]);
        hi.w = Act<ACT>::pack2(v[6], v[7]);
        *reinterpret_cast<uint4*>(xs_hi + n * XS + kc) = hi;
        if constexpr (kSplit) {
          const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
          uint32_t lw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 h2 = Act<ACT>::unpack2(hw[i]);
            lw[i] = Act<ACT>::pack2(v[2 * i] - h2.x, v[2 * i + 1] - h2.y);
          }
          *reinterpret_cast<uint4*>(xs_lo + n * XS + kc) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
  };

  // LayerNorm statistics of the GEMM input (regions 1 and 4a): one warp per
  // batch row, combined from the producer's per-tile partials or, when there
  // are none, computed directly in two passes.
  if constexpr (R == Region::LnQkv || R == Region::FfnUp) {
    for (int n = warp; n < M; n += kProducers) {
      float mean, m2;
      if (a.stats_in != nullptr && K / 16 <= 32 * 16) {
        // All of this lane's tile partials in flight at once, then two passes
        // over registers (mean, then the pooled second moment).
        const int tin = K / 16;
        const float2* st2 = reinterpret_cast<const float2*>(a.stats_in);
        float2 pr[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int i = lane + 32 * j;
          pr[j] = i < tin ? st2[(size_t)i * M + n] : make_float2(0.f, 0.f);
        }
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) s += pr[j].x;
        mean = warp_sum(s) / (float)K;
        float q = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (lane + 32 * j < tin) {
            const float d = pr[j].x * (1.0f / 16.0f) - mean;
            q += pr[j].y + 16.0f * d * d;
          }
        }
        m2 = warp_sum(q);
      } else if (a.stats_in != nullptr) {
        const int tin = K / 16;
        float s = 0.f;
        for (int i = lane; i < tin; i += 32) s += a.stats_in[((size_t)i * M + n) * 2];
        mean = warp_sum(s) / (float)K;
        float q = 0.f;
        for (int i = lane; i < tin; i += 32) {
          const float ts = a.stats_in[((size_t)i * M + n) * 2];
          const float tm2 = a.stats_in[((size_t)i * M + n) * 2 + 1];
          const float d = ts * (1.0f / 16.0f) - mean;
          q += tm2 + 16.0f * d * d;
        }
        m2 = warp_sum(q);
      } else {
        const ACT* xr = static_cast<const ACT*>(a.x_act) + (size_t)n * K;
        float s = 0.f;
        for (int k = lane * 8; k < K; k += 256) {
          const uint4 u = *reinterpret_cast<const uint4*>(xr + k);
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = Act<ACT>::unpack2(uw[i]);
            s += f.x + f.y;
          }
        }
        mean = warp_sum(s) / (float)K;
        float q = 0.f;
        for (int k = lane * 8; k < K; k += 256) {
          const uint4 u = *reinterpret_cast<const uint4*>(xr + k);
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = Act<ACT>::unpack2(uw[i]);
            q += (f.x - mean) * (f.x - mean) + (f.y - mean) * (f.y - mean);
          }
        }
        m2 = warp_sum(q);
      }
      if (lane == 0) {
        s_mean[n] = mean;
        s_rstd[n] = 1.0f / sqrtf(m2 / (float)K + a.eps);
      }
    }
  }

  float acc[NA][NT][4];
#pragma unroll
  for (int ia = 0; ia < NA; ++ia)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[ia][nt][0] = acc[ia][nt][1] = acc[ia][nt][2] = acc[ia][nt][3] = 0.f;
  int cur_s = -1;
  const int wk = warp * step_k;
  // One segment: chunks kc0 .. kc1-1 of unit u, then its partial tile to the
  // epilogue warp.  Segments come in the copy warp's order (work_split.h).
  auto run_segment = [&](int u, int kc0, int kc1) {
    const int s_ = u / P.tiles;
    if (s_ != cur_s) {  // first chunk of a K slice: stage its x (CTA-uniform)
      bar_sync(kBarStage, kProducers * 32);
      stage(s_);
      bar_sync(kBarStage, kProducers * 32);
      cur_s = s_;
    }
    for (int kc = kc0; kc < kc1; ++kc) {
      if (!rp.dead) rp.dead = !mbar_wait(sm.full_bar(rp.st), rp.ph, a.status);
      Slot cur;
      load(rp.st, cur);
      compute(cur, kc * P.chunk_k + wk, acc);
      // the warp-collective MMAs above have consumed every lane's loads
      if (lane == 0) mbar_arrive(sm.empty_bar(rp.st));
      rp.advance(S);
    }
    constexpr int NB = SegBufs<NT>::n;
    const int buf = seg % NB;
    if (seg >= NB) bar_sync(kBarEmpty + buf, kProducers * 32 + 32);
    float* p = red + ((size_t)buf * kProducers + warp) * NT * 128;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[e] = acc[0][nt][e];
#pragma unroll
        for (int ia = 1; ia < NA; ++ia) v[e] += acc[ia][nt][e];
#pragma unroll
        for (int ia = 0; ia < NA; ++ia) acc[ia][nt][e] = 0.f;
      }
      *reinterpret_cast<float2*>(p + nt * 128 + wr * 8 + 2 * c) = make_float2(v[0], v[1]);
      *reinterpret_cast<float2*>(p + nt * 128 + (wr + 8) * 8 + 2 * c) = make_float2(v[2], v[3]);
    }
    bar_arrive(kBarFull + buf, kProducers * 32 + 32);
    ++seg;
  };
  for (long long i = ra; i < rb;) {
    int u, j_slot;
    long long end;
    ws_leftover_segment(P, i, rb, cta, G, &u, &end, &j_slot);
    const int kc0 = (int)(i - (long long)(u - P.U_dp) * P.C);
    run_segment(u, kc0, kc0 + (int)(end - i));
    i = end;
  }
  for (int u = dp_b; u < dp_b + P.q; ++u) run_segment(u, 0, P.C);
}

// MMA warps, after their last phase: wait until the epilogue warp has
// released the last segment buffers (keeps every named-barrier phase matched).
template <int NT>
__device__ __forceinline__ void gemv_mma_drain(int seg) {
  constexpr int NB = SegBufs<NT>::n;
  for (int i = seg >= NB ? seg - NB : 0; i < seg; ++i) bar_sync(kBarEmpty + i % NB, kProducers * 32 + 32);
}

// Epilogue warp: reduces each segment of one GEMV phase and runs the region
// epilogue or the split-K fix-up.  `seg` counts segments across phases.
template <Region R, WKind WK, typename ACT, int NT>
__device__ void gemv_epi_phase(const RegionArgs& a, const GemvPlan& P, const GemvSmem& sm, int& seg, int e = 0,
                               int nepi = 1) {
  using G_ = Geom<WK>;
  using L = SmemLayout<NT>;
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;  // hi + lo bf16 operand
  constexpr int ROWS = 8 * NT;
  constexpr bool kStats = (R == Region::OprojRes || R == Region::FfnDown);
  constexpr int ESZ = (WK == WKind::I8) ? 1 : 2;  // weight bytes
  constexpr bool kI8 = (WK == WKind::I8);
  (void)kSplit; (void)ROWS; (void)kStats; (void)kI8;
  const int M = a.M, N = a.N, K = a.K;
  const int K_S = P.K_S;
  const int XS = K_S + G_::PAD;  // x row stride, elements
  const int S = sm.S;
  const size_t SB = sm.SB;
  const size_t RB = L::chunk_bytes(P.chunk_k, ESZ);  // offset of a stage's int8 scales
  unsigned char* ring = sm.ring;
  ACT* xs_hi = reinterpret_cast<ACT*>(sm.xs);
  ACT* xs_lo = xs_hi + M * XS;
  float* red = sm.red;
  float* tileval = sm.tileval + e * 16 * 8 * NT;  // this epilogue warp's tile scratch
  float* s_mean = sm.s_mean;
  float* s_rstd = sm.s_rstd;
  (void)xs_lo; (void)red; (void)tileval; (void)s_mean; (void)s_rstd; (void)RB; (void)XS; (void)N;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  (void)g; (void)c; (void)tid; (void)warp;
  const int tiles = P.tiles, C = P.C;
  const int cta = blockIdx.x, G = gridDim.x;
  (void)tiles; (void)C;
  long long ra, rb;
  ws_left_range(P, cta, G, &ra, &rb);
  const int dp_b = cta * P.q;
  const int nchunks = (int)(rb - ra) + P.q * C;
  (void)nchunks; (void)K; (void)S; (void)SB; (void)ring; (void)M; (void)K_S;
  constexpr int VPL = 4 * NT;  // reduced values per lane (16 x ROWS / 32)
  const int KS = P.KS;
  const int slots = KS * P.maxc;

  // Global operands of one output element, loaded before the segment's
  // partial tiles arrive so that their latency overlaps the MMA warps' work.
  struct EpiOp {
    float bias = 0.f;
    float res = 0.f;  // residual; region 1: the KV-cache position, as int bits
  };
  auto epi_load = [&](int n, int m) -> EpiOp {
    EpiOp o;
    o.bias = Act<ACT>::to_f(static_cast<const ACT*>(a.bias)[n]);
    if constexpr (R == Region::LnQkv) {
      const int b = m / a.T;
      o.res = __int_as_float(a.past_len[b] + (m - b * a.T));
    } else if constexpr (R == Region::OprojRes) {
      o.res = Act<ACT>::to_f(static_cast<const ACT*>(a.resid_act)[(size_t)m * N + n]);
    } else if constexpr (R == Region::FfnDown) {
      o.res = a.resid_f32[(size_t)m * N + n];
    }
    return o;
  };

  auto epilogue = [&](int n, int m, float acc, const EpiOp& op) -> float {
    float v = acc + op.bias;
    if (!ds_in_bounds(m < a.M && n < N, a.status)) return v;
    if constexpr (R == Region::LnQkv) {
      const int H = a.H;
      const int part = n / H;
      const int within = n - part * H;
      if (part == 0) {
        a.out_f32[(size_t)m * H + within] = v;
      } else {
        const int b = m / a.T;
        const int pos = __float_as_int(op.res);
        if (pos >= 0 && pos < a.max_len) {
          const int head = within / a.head_dim, dim = within - head * a.head_dim;
          ACT* cache = static_cast<ACT*>(part == 1 ? a.k_cache : a.v_cache);
          if (ds_in_bounds(b < a.B && head < a.heads, a.status))
            cache[(((size_t)b * a.heads + head) * a.max_len + pos) * a.head_dim + dim] = Act<ACT>::from_f(v);
        } else {
          atomicOr(a.status, 1u);
        }
      }
      return v;
    } else if constexpr (R == Region::OprojRes) {
      v += op.res;
      a.out_f32[(size_t)m * N + n] = v;
      return v;
    } else if constexpr (R == Region::FfnUp) {
      v = gelu_tanh(v);
      a.out_f32[(size_t)m * N + n] = v;
      return v;
    } else {
      v += op.res;
      const ACT y = Act<ACT>::from_f(v);
      static_cast<ACT*>(a.out_act)[(size_t)m * N + n] = y;
      return Act<ACT>::to_f(y);
    }
  };

  auto finish_tile = [&](int t, const float (&val)[VPL], const EpiOp (&op)[VPL]) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = lane + 32 * i;
      const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
      if (col < M) {
        const float y = epilogue(t * 16 + row, col, val[i], op[i]);
        if constexpr (kStats) tileval[row * ROWS + col] = y;
      }
    }
    if constexpr (kStats) {
      if (a.stats_out != nullptr) {
        __syncwarp();
        for (int m = lane; m < M; m += 32) {
          float sum = 0.f;
#pragma unroll
          for (int r = 0; r < 16; ++r) sum += tileval[r * ROWS + m];
          const float mean = sum * (1.0f / 16.0f);
          float m2 = 0.f;
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const float d = tileval[r * ROWS + m] - mean;
            m2 += d * d;
          }
          a.stats_out[((size_t)t * M + m) * 2] = sum;
          a.stats_out[((size_t)t * M + m) * 2 + 1] = m2;
        }
        __syncwarp();
      }
    }
  };

  // Epilogue warp e of nepi takes segments e, e + nepi, ... (its own buffers).
  auto process = [&](int u, int j_slot) {
    if (seg % nepi != e) {
      ++seg;
      return;
    }
    const int s = u / tiles, t = u - (u / tiles) * tiles;
    const int buf = seg % SegBufs<NT>::n;
    EpiOp op[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = lane + 32 * i;
      const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
      if (col < M) op[i] = epi_load(t * 16 + row, col);
    }
    bar_sync(kBarFull + buf, kProducers * 32 + 32);
    const float* rbuf = red + (size_t)buf * kProducers * NT * 128;
    float val[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = lane + 32 * i;
      const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
      const int nt = col >> 3, cc = col & 7;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kProducers; ++w) sum += rbuf[(w * NT + nt) * 128 + row * 8 + cc];
      val[i] = sum;
    }
    bar_arrive(kBarEmpty + buf, kProducers * 32 + 32);
    ++seg;
    const int contrib = ws_unit_contrib(u, P, G);
    if (KS == 1 && contrib == 1) {
      finish_tile(t, val, op);
      return;
    }
    // Partial of a tile shared with other CTAs / K slices: publish, count,
    // and let the last contributor combine (fixed order: slice, then CTA).
    const int slot = s * P.maxc + j_slot;
    float* pbase = a.partials + (size_t)t * slots * 16 * M;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = lane + 32 * i;
      const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
      if (col < M) pbase[((size_t)slot * 16 + row) * M + col] = val[i];
    }
    // The warp barrier orders every lane's partial stores before lane 0's
    // release-acquire arrival; the last arriver's acquire (then the warp
    // barrier) orders its reads of the other partials after all arrivals.
    __syncwarp();
    const int target = ws_tile_target(t, P, G);
    int last = 0;
    if (lane == 0) last = (atomic_add_acq_rel_gpu(&a.counters[t], 1) == target - 1);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < VPL; ++i) val[i] = 0.f;
    for (int s2 = 0; s2 < KS; ++s2) {
      const int n2 = ws_unit_contrib(s2 * tiles + t, P, G);
#pragma unroll 4
      for (int j2 = 0; j2 < n2; ++j2) {
        const int sl2 = s2 * P.maxc + j2;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const int v = lane + 32 * i;
          const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
          if (col < M) val[i] += ld_cg(pbase + ((size_t)sl2 * 16 + row) * M + col);
        }
      }
    }
    if (lane == 0) a.counters[t] = 0;
    finish_tile(t, val, op);
  };

  // Segments in the streaming warps' order: leftover chunks, then whole units.
  for (long long i = ra; i < rb;) {
    int u, j_slot;
    long long end;
    ws_leftover_segment(P, i, rb, cta, G, &u, &end, &j_slot);
    process(u, j_slot);
    i = end;
  }
  for (int u = dp_b; u < dp_b + P.q; ++u) process(u, 0);

}

template <Region R, WKind WK, typename ACT, int NT>
__global__ void __launch_bounds__(kGemvThreads, 1) region_gemv_kernel(const RegionArgs a) {
  constexpr int ESZ = (WK == WKind::I8) ? 1 : 2;
  constexpr int PAD = Geom<WK>::PAD;
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const GemvPlan& P = a.plan;
  const GemvSmem sm = gemv_carve<NT>(smem_raw, P.stages, SmemLayout<NT>::stage_bytes(P.chunk_k, ESZ, WK == WKind::I8),
                                     SmemLayout<NT>::xs_bytes(a.M, P.K_S, PAD, kSplit));
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) gemv_init_ring(sm);
  __syncthreads();

  if (warp < kProducers) {
    pdl_wait();
    pdl_launch_dependents();
    RingPos rp;
    int seg = 0;
    gemv_mma_phase<R, WK, ACT, NT, (NT <= 2 ? 4 : 2)>(a, a.plan, sm, rp, seg);
    gemv_mma_drain<NT>(seg);
  } else if (warp >= kTmaWarp0) {
    // Weights do not depend on the previous kernel, so the copy warps never
    // wait for it: the ring fills while the previous kernel is still finishing.
    RingPos rp;
    gemv_tma_phase<R, WK, ACT, NT>(a, a.plan, sm, rp, warp - kTmaWarp0, l2_evict_first_policy());
    if (a.next_tmap_w != nullptr)
      gemv_l2_prefetch_phase<WK>(a.next_tmap_w, a.next_tmap_s, a.next_plan, kL2Lookahead, a.next_qgroup);
    pdl_launch_dependents();
  } else {
    pdl_wait();
    pdl_launch_dependents();
    int seg = 0;
    const int e = warp - kEpiWarp;
    gemv_epi_phase<R, WK, ACT, NT>(a, a.plan, sm, seg, e, kEpiWarps);
    if constexpr (R == Region::FfnDown) {
      if (a.seq_len_inc != nullptr && blockIdx.x == 0 && e == 0)
        for (int b = threadIdx.x & 31; b < a.B; b += 32) a.seq_len_inc[b] += 1;
    }
  }
}

// Launches region kernel R for the NT chosen by the plan.
template <WKind WK, typename ACT>
cudaError_t launch_region_t(Region r, const RegionArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan.grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = a.plan.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;

#define DS_LAUNCH_NT(REG, NTV) return cudaLaunchKernelEx(&cfg, region_gemv_kernel<REG, WK, ACT, NTV>, a)
#define DS_LAUNCH_REG(REG)                 \
  switch (a.plan.nt) {                     \
    case 1: DS_LAUNCH_NT(REG, 1);          \
    case 2: DS_LAUNCH_NT(REG, 2);          \
    case 4: DS_LAUNCH_NT(REG, 4);          \
    case 8: DS_LAUNCH_NT(REG, 8);          \
    default: return cudaErrorInvalidValue; \
  }
  switch (r) {
    case Region::LnQkv: DS_LAUNCH_REG(Region::LnQkv);
    case Region::OprojRes: DS_LAUNCH_REG(Region::OprojRes);
    case Region::FfnUp: DS_LAUNCH_REG(Region::FfnUp);
    case Region::FfnDown: DS_LAUNCH_REG(Region::FfnDown);
  }
#undef DS_LAUNCH_REG
#undef DS_LAUNCH_NT
  return cudaErrorInvalidValue;
}

// Raises the dynamic shared-memory limit of every instantiation for this
// weight/activation pair.  Called once per device at layer creation, before
// any launch (and so before any stream capture).
template <WKind WK, typename ACT>
cudaError_t prepare_region_t(int max_smem) {
  cudaError_t e = cudaSuccess;
#define DS_PREP(REG, NTV)                                                                    \
  if (e == cudaSuccess)                                                                      \
    e = cudaFuncSetAttribute(region_gemv_kernel<REG, WK, ACT, NTV>,                          \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)
#define DS_PREP_REG(REG) DS_PREP(REG, 1); DS_PREP(REG, 2); DS_PREP(REG, 4); DS_PREP(REG, 8)
  DS_PREP_REG(Region::LnQkv);
  DS_PREP_REG(Region::OprojRes);
  DS_PREP_REG(Region::FfnUp);
  DS_PREP_REG(Region::FfnDown);
#undef DS_PREP_REG
#undef DS_PREP
  return e;
}

}  // namespace ds
