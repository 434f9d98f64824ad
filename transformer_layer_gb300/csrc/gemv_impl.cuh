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
//  * Weights stream from HBM exactly once, with 128-bit no-L1-allocate loads
//    held in a 6-deep register ring per warp (one CTA per SM).  The first loads are issued
//    before griddepcontrol.wait, so they overlap the previous kernel's tail.
//  * The 16 x 8 x 16 tensor-core MMA multiplies (weights are the 16-row A
//    side, batch rows the 8-column B side): at M <= 8 it needs ~5x fewer
//    instructions per weight byte than CUDA-core FMAs.
//  * Work: a unit is 16 weight rows x one K slice, a chunk is 8 warp steps of
//    it (one per streaming warp, so all 8 warps of a CTA always finish
//    together).  Each CTA owns q whole units; the leftover units' chunks are
//    spread evenly over all CTAs (balanced to within one chunk), and the last
//    CTA to contribute to a row tile (atomic arrival counter, no waiting) sums
//    the partials in fixed order.  Leftover chunks are processed first so
//    that these fix-ups happen early, not at the kernel's tail.
//  * Warp specialisation: four copy warps (TMA), 8 MMA warps that never touch
//    global memory in their loop, and one epilogue warp that takes each
//    finished segment's per-warp partial tiles through shared memory
//    (double-buffered, named barriers), reduces them, and runs the region
//    epilogue / split-K fix-up.
//
// K permutation: a lane of the MMA fragment owns k pairs {2c, 2c+1} and
// {2c+8, 2c+9} of a 16-wide k block.  Each lane instead reads 8 contiguous
// weights (16 bytes) of a ring row and the B operand is read with the same
// permutation, so the dot product is unchanged while every shared-memory read
// is a conflict-free 128-bit access (row pitch = chunk bytes + 64).
#pragma once

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "work_split.h"

namespace ds {

constexpr int kProducers = 8;             // MMA warps (each "produces" a partial tile per segment)
constexpr int kEpiWarp = kProducers;      // warp 8: reduction, epilogue, split-K fix-up
constexpr int kTmaWarp0 = kProducers + 1; // warps 9..12: TMA bulk copies of the weights
constexpr int kTmaWarps = 4;              // each copies 4 of a chunk's 16 rows (one warp's
                                          // bulk-copy issue rate alone caps near 3.5 TB/s)
constexpr int kGemvThreads = (kProducers + 1 + kTmaWarps) * 32;
constexpr int kMaxStages = 8;             // weight ring depth (chunks in flight per CTA)

// Named barriers (0 is __syncthreads, unused here).
constexpr int kBarStage = 1;  // the 8 streaming warps
constexpr int kBarFull = 2;   // 2, 3: segment partials written (streaming -> epilogue)
constexpr int kBarEmpty = 4;  // 4, 5: segment partials consumed (epilogue -> streaming)

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
  // Weight ring: `stages` chunks, each 16 rows of chunk_k weights (row pitch
  // padded by 64 bytes to spread banks) plus, for int8, their 16 x chunk_k/64
  // fp16 scales.  Then the x slice [M][K_S + pad] (hi, and lo for bf16), the
  // segment buffers [2][8 warps][NT][16][8] fp32, tile values [16][8 NT], LN
  // mean / rstd [64] and the full / empty mbarriers of the ring.
  static __host__ __device__ size_t row_bytes(int chunk_k, int esize) {
    return (size_t)chunk_k * esize + 64;
  }
  static __host__ __device__ size_t scale_bytes(int chunk_k, bool i8) {
    return i8 ? (size_t)16 * (chunk_k / 64) * 2 : 0;
  }
  static __host__ __device__ size_t stage_bytes(int chunk_k, int esize, bool i8) {
    return 16 * row_bytes(chunk_k, esize) + scale_bytes(chunk_k, i8);
  }
  static __host__ __device__ size_t xs_bytes(int M, int K_S, int pad, bool split) {
    const size_t b = (size_t)(split ? 2 : 1) * M * (K_S + pad) * 2;
    return (b + 15) & ~(size_t)15;
  }
  static __host__ __device__ size_t red_floats() { return (size_t)2 * kProducers * NT * 128; }
  // Everything except the weight ring and its barriers.
  static __host__ __device__ size_t fixed(int M, int K_S, int pad, bool split) {
    return xs_bytes(M, K_S, pad, split) + 4 * (red_floats() + 16 * 8 * NT + 2 * 64);
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

struct Slot {
  uint4 a[4];            // [row r (g, g+8)][block]
  unsigned short sc[4];  // int8 only: fp16 scale bits, [row r][block]
};

template <Region R, WKind WK, typename ACT, int NT>
__global__ void __launch_bounds__(kGemvThreads, 1) region_gemv_kernel(const RegionArgs a) {
  using G_ = Geom<WK>;
  using L = SmemLayout<NT>;
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;  // hi + lo bf16 operand
  constexpr int ROWS = 8 * NT;
  constexpr bool kStats = (R == Region::OprojRes || R == Region::FfnDown);
  extern __shared__ __align__(16) unsigned char smem_raw[];

  constexpr int ESZ = (WK == WKind::I8) ? 1 : 2;  // weight bytes
  constexpr bool kI8 = (WK == WKind::I8);
  const GemvPlan& P = a.plan;
  const int M = a.M, N = a.N, K = a.K;
  const int K_S = P.K_S;
  const int XS = K_S + G_::PAD;  // x row stride, elements
  const int S = P.stages;
  const size_t RB = L::row_bytes(P.chunk_k, ESZ);
  const size_t SB = L::stage_bytes(P.chunk_k, ESZ, kI8);
  unsigned char* ring = smem_raw;
  ACT* xs_hi = reinterpret_cast<ACT*>(smem_raw + (size_t)S * SB);
  ACT* xs_lo = xs_hi + M * XS;
  float* red = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(xs_hi) +
                                        L::xs_bytes(M, K_S, G_::PAD, kSplit));
  float* tileval = red + L::red_floats();  // [16][ROWS]
  float* s_mean = tileval + 16 * ROWS;     // [64]
  float* s_rstd = s_mean + 64;             // [64]
  uint64_t* mbar = reinterpret_cast<uint64_t*>(s_rstd + 64);  // full[S], empty[S]
  auto full_bar = [&](int i) { return smem_u32(mbar + i); };
  auto empty_bar = [&](int i) { return smem_u32(mbar + S + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int tiles = P.tiles, C = P.C;
  const int cta = blockIdx.x, G = gridDim.x;
  const long long ra = (long long)cta * P.R / G, rb = (long long)(cta + 1) * P.R / G;
  const int dp_b = cta * P.q;
  const int nchunks = (int)(rb - ra) + P.q * C;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full_bar(i), kTmaWarps);
      mbar_init(empty_bar(i), kProducers);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp < kProducers) {
    // =================== streaming warps ===================
    const int step_k = P.nblk * G_::BLK_K;
    auto cur_init = [&](Cursor& q) { ws_cursor_init(q, P, ra, rb, dp_b); };
    auto cur_next = [&](Cursor& q) { ws_cursor_next(q, P, dp_b); };
    // A fragments of this warp's step of the chunk in ring stage `st`.
    auto load = [&](int st, Slot& sl) {
      const unsigned char* base = ring + (size_t)st * SB + (size_t)g * RB + warp * step_k * ESZ + 16 * c;
      sl.a[0] = *reinterpret_cast<const uint4*>(base);
      sl.a[2] = *reinterpret_cast<const uint4*>(base + 8 * RB);
      if (P.nblk == 2) {
        sl.a[1] = *reinterpret_cast<const uint4*>(base + 64);
        sl.a[3] = *reinterpret_cast<const uint4*>(base + 8 * RB + 64);
      }
      if constexpr (kI8) {
        const int gpc = P.chunk_k / 64;  // scale groups per chunk row
        const unsigned short* sc =
            reinterpret_cast<const unsigned short*>(ring + (size_t)st * SB + 16 * RB);
        const int g0 = warp * step_k / 64;
        sl.sc[0] = sc[g * gpc + g0];
        sl.sc[2] = sc[(g + 8) * gpc + g0];
        if (P.nblk == 2) {
          sl.sc[1] = sc[g * gpc + g0 + 1];
          sl.sc[3] = sc[(g + 8) * gpc + g0 + 1];
        }
      }
    };
    // B operand of n-tile nt: rows >= M are zero and not read.
    auto load_x = [&](const ACT* base, int nt, int off) -> uint4 {
      const int n = nt * 8 + g;
      if (n < M) return *reinterpret_cast<const uint4*>(base + n * XS + off);
      return make_uint4(0u, 0u, 0u, 0u);
    };
    auto compute = [&](const Slot& sl, int kl, float (&acc)[NT][4]) {
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        if (blk == 1 && P.nblk == 1) break;
        if constexpr (WK == WKind::I8) {
          uint32_t lo0[4], hi0[4], lo1[4], hi1[4];
          const uint32_t w0[4] = {sl.a[blk].x, sl.a[blk].y, sl.a[blk].z, sl.a[blk].w};
          const uint32_t w1[4] = {sl.a[2 + blk].x, sl.a[2 + blk].y, sl.a[2 + blk].z, sl.a[2 + blk].w};
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
          const float s1 = __half2float(__ushort_as_half(sl.sc[2 + blk]));
          const int off = kl + blk * 64 + 16 * c;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt * 8 >= M) break;
            float tmp[4] = {0.f, 0.f, 0.f, 0.f};
            const uint4 X0 = load_x(xs_hi, nt, off), X1 = load_x(xs_hi, nt, off + 8);
            const uint32_t xw[8] = {X0.x, X0.y, X0.z, X0.w, X1.x, X1.y, X1.z, X1.w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
              Mma<ACT>::run(tmp, lo0[m], lo1[m], hi0[m], hi1[m], xw[2 * m], xw[2 * m + 1]);
            if constexpr (kSplit) {
              const uint4 Y0 = load_x(xs_lo, nt, off), Y1 = load_x(xs_lo, nt, off + 8);
              const uint32_t yw[8] = {Y0.x, Y0.y, Y0.z, Y0.w, Y1.x, Y1.y, Y1.z, Y1.w};
#pragma unroll
              for (int m = 0; m < 4; ++m)
                Mma<ACT>::run(tmp, lo0[m], lo1[m], hi0[m], hi1[m], yw[2 * m], yw[2 * m + 1]);
            }
            acc[nt][0] += tmp[0] * s0;
            acc[nt][1] += tmp[1] * s0;
            acc[nt][2] += tmp[2] * s1;
            acc[nt][3] += tmp[3] * s1;
          }
        } else {
          const uint4 A0 = sl.a[blk], A1 = sl.a[2 + blk];
          const int off = kl + blk * 32 + 8 * c;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (nt * 8 >= M) break;
            const uint4 X = load_x(xs_hi, nt, off);
            Mma<ACT>::run(acc[nt], A0.x, A1.x, A0.y, A1.y, X.x, X.y);
            Mma<ACT>::run(acc[nt], A0.z, A1.z, A0.w, A1.w, X.z, X.w);
            if constexpr (kSplit) {
              const uint4 Y = load_x(xs_lo, nt, off);
              Mma<ACT>::run(acc[nt], A0.x, A1.x, A0.y, A1.y, Y.x, Y.y);
              Mma<ACT>::run(acc[nt], A0.z, A1.z, A0.w, A1.w, Y.z, Y.w);
            }
          }
        }
      }
    };
    // Stage x[:, slice s] (rows < M) into shared memory, the region prologue fused in.
    auto stage = [&](int s) {
      const int k0 = s * K_S;
      const int cpr = K_S / 8;
      for (int idx = tid; idx < M * cpr; idx += kProducers * 32) {
        const int n = idx / cpr;
        const int kc = (idx - n * cpr) * 8;
        float v[8];
        if constexpr (R == Region::LnQkv) {
          const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.x_act) +
                                                          (size_t)n * K + k0 + kc);
          const uint4 gu = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_g) + k0 + kc);
          const uint4 bu = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_b) + k0 + kc);
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w}, gw[4] = {gu.x, gu.y, gu.z, gu.w},
                         bw[4] = {bu.x, bu.y, bu.z, bu.w};
          const float mu = s_mean[n], rs = s_rstd[n];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 xv = Act<ACT>::unpack2(uw[i]), gv = Act<ACT>::unpack2(gw[i]),
                         bv = Act<ACT>::unpack2(bw[i]);
            v[2 * i] = (xv.x - mu) * rs * gv.x + bv.x;
            v[2 * i + 1] = (xv.y - mu) * rs * gv.y + bv.y;
          }
        } else {
          const float* src = a.x_f32 + (size_t)n * K + k0 + kc;
          const float4 p0 = *reinterpret_cast<const float4*>(src);
          const float4 p1 = *reinterpret_cast<const float4*>(src + 4);
          v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
          v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
          if constexpr (R == Region::FfnUp) {
            const uint4 gu = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_g) + k0 + kc);
            const uint4 bu = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_b) + k0 + kc);
            const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
            const float mu = s_mean[n], rs = s_rstd[n];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 gv = Act<ACT>::unpack2(gw[i]), bv = Act<ACT>::unpack2(bw[i]);
              v[2 * i] = (v[2 * i] - mu) * rs * gv.x + bv.x;
              v[2 * i + 1] = (v[2 * i + 1] - mu) * rs * gv.y + bv.y;
            }
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
    };

    Cursor Cn;
    cur_init(Cn);

    pdl_wait();
    pdl_launch_dependents();

    // LayerNorm statistics of the GEMM input (regions 1 and 4a): one warp per
    // batch row, combined from the producer's per-tile partials or, when there
    // are none, computed directly in two passes.
    if constexpr (R == Region::LnQkv || R == Region::FfnUp) {
      for (int n = warp; n < M; n += kProducers) {
        float mean, m2;
        if (a.stats_in != nullptr) {
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

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    int cur_s = -1;
    int seg = 0;
    const int wk = warp * step_k;
    int st = 0;
    uint32_t phase = 0;
    bool timed_out = false;  // after a timed-out wait, no further waits (results are flagged invalid)
    for (int j = 0; j < nchunks; ++j) {
      if (Cn.s != cur_s) {  // first chunk of a K slice: stage its x (CTA-uniform)
        bar_sync(kBarStage, kProducers * 32);
        stage(Cn.s);
        bar_sync(kBarStage, kProducers * 32);
        cur_s = Cn.s;
      }
      if (!timed_out) timed_out = !mbar_wait(full_bar(st), phase, a.status);
      Slot sl;
      load(st, sl);
      compute(sl, Cn.kc * P.chunk_k + wk, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
      if (ws_segment_ends(Cn, P, j, nchunks)) {
        const int buf = seg & 1;
        if (seg >= 2) bar_sync(kBarEmpty + buf, kProducers * 32 + 32);
        float* p = red + ((size_t)buf * kProducers + warp) * NT * 128;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          *reinterpret_cast<float2*>(p + nt * 128 + g * 8 + 2 * c) = make_float2(acc[nt][0], acc[nt][1]);
          *reinterpret_cast<float2*>(p + nt * 128 + (g + 8) * 8 + 2 * c) =
              make_float2(acc[nt][2], acc[nt][3]);
          acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        }
        bar_arrive(kBarFull + buf, kProducers * 32 + 32);
        ++seg;
      }
      cur_next(Cn);
      if (++st == S) {
        st = 0;
        phase ^= 1;
      }
    }
    // Wait until the epilogue warp has released the last buffers (keeps every
    // named-barrier phase matched).
    for (int i = seg >= 2 ? seg - 2 : 0; i < seg; ++i) bar_sync(kBarEmpty + (i & 1), kProducers * 32 + 32);
  } else if (warp >= kTmaWarp0) {
    // =================== TMA warps: stream the weights ===================
    // Weights do not depend on the previous kernel, so these warps never wait
    // for it: the ring fills while the previous kernel is still finishing.
    // TMA warp i copies rows 4i..4i+3 of every chunk (and their int8 scales).
    const int tw = warp - kTmaWarp0;
    const uint64_t pol = l2_evict_first_policy();
    const uint32_t row_bytes = (uint32_t)(P.chunk_k * ESZ);
    const uint32_t sc_bytes = (uint32_t)(P.chunk_k / 64 * 2);
    const uint32_t tx = 4 * row_bytes + (kI8 ? 4 * sc_bytes : 0);
    Cursor q;
    ws_cursor_init(q, P, ra, rb, dp_b);
    int st = 0;
    uint32_t phase = 0;
    bool timed_out = false;
    for (int j = 0; j < nchunks; ++j) {
      if (j >= S && !timed_out) timed_out = !mbar_wait(empty_bar(st), phase ^ 1, a.status);
      if (lane == 0) mbar_arrive_expect_tx(full_bar(st), tx);
      __syncwarp();
      const size_t kg = (size_t)q.s * K_S + (size_t)q.kc * P.chunk_k;
      const size_t row0 = (size_t)q.t * 16;
      if (lane < 4) {
        const int r = 4 * tw + lane;
        const unsigned char* src = static_cast<const unsigned char*>(a.W) + ((row0 + r) * K + kg) * ESZ;
        bulk_g2s(smem_u32(ring + (size_t)st * SB + r * RB), src, row_bytes, full_bar(st), pol);
      } else if (kI8 && lane < 8) {
        const int r = 4 * tw + lane - 4;
        const unsigned char* src = reinterpret_cast<const unsigned char*>(a.Wscale) +
                                   ((row0 + r) * (K / 64) + kg / 64) * 2;
        bulk_g2s(smem_u32(ring + (size_t)st * SB + 16 * RB + r * sc_bytes), src, sc_bytes, full_bar(st),
                 pol);
      }
      ws_cursor_next(q, P, dp_b);
      if (++st == S) {
        st = 0;
        phase ^= 1;
      }
    }
    pdl_launch_dependents();
  } else {
    // =================== epilogue warp ===================
    pdl_wait();
    pdl_launch_dependents();
    constexpr int VPL = 4 * NT;  // reduced values per lane (16 x ROWS / 32)
    const int KS = P.KS;
    const int slots = KS * P.maxc;

    auto epilogue = [&](int n, int m, float acc) -> float {
      const float bias = Act<ACT>::to_f(static_cast<const ACT*>(a.bias)[n]);
      float v = acc + bias;
      if constexpr (R == Region::LnQkv) {
        const int H = a.H;
        const int part = n / H;
        const int within = n - part * H;
        if (part == 0) {
          a.out_f32[(size_t)m * H + within] = v;
        } else {
          const int b = m / a.T, tt = m - (m / a.T) * a.T;
          const int pos = a.past_len[b] + tt;
          if (pos >= 0 && pos < a.max_len) {
            const int head = within / a.head_dim, dim = within - head * a.head_dim;
            ACT* cache = static_cast<ACT*>(part == 1 ? a.k_cache : a.v_cache);
            cache[(((size_t)b * a.heads + head) * a.max_len + pos) * a.head_dim + dim] = Act<ACT>::from_f(v);
          } else {
            atomicOr(a.status, 1u);
          }
        }
        return v;
      } else if constexpr (R == Region::OprojRes) {
        v += Act<ACT>::to_f(static_cast<const ACT*>(a.resid_act)[(size_t)m * N + n]);
        a.out_f32[(size_t)m * N + n] = v;
        return v;
      } else if constexpr (R == Region::FfnUp) {
        v = gelu_tanh(v);
        a.out_f32[(size_t)m * N + n] = v;
        return v;
      } else {
        v += a.resid_f32[(size_t)m * N + n];
        const ACT y = Act<ACT>::from_f(v);
        static_cast<ACT*>(a.out_act)[(size_t)m * N + n] = y;
        return Act<ACT>::to_f(y);
      }
    };

    auto finish_tile = [&](int t, const float (&val)[VPL]) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int v = lane + 32 * i;
        const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
        if (col < M) {
          const float y = epilogue(t * 16 + row, col, val[i]);
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

    int seg = 0;
    auto process = [&](int u, int j_slot) {
      const int s = u / tiles, t = u - (u / tiles) * tiles;
      const int buf = seg & 1;
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
        finish_tile(t, val);
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
      __threadfence();
      __syncwarp();
      const int target = ws_tile_target(t, P, G);
      int last = 0;
      if (lane == 0) last = (atomicAdd(&a.counters[t], 1) == target - 1);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) return;
      __threadfence();
#pragma unroll
      for (int i = 0; i < VPL; ++i) val[i] = 0.f;
      for (int s2 = 0; s2 < KS; ++s2) {
        const int n2 = ws_unit_contrib(s2 * tiles + t, P, G);
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
      finish_tile(t, val);
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

    if constexpr (R == Region::FfnDown) {
      if (a.seq_len_inc != nullptr && cta == 0)
        for (int b = lane; b < a.B; b += 32) a.seq_len_inc[b] += 1;
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
