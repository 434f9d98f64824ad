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
// GB300 design (not the pages'): the weights stream from HBM exactly once with
// 128-bit no-L1-allocate loads held in a 4-deep register ring per warp (issued
// before griddepcontrol.wait, so they overlap the previous kernel's tail); the
// 16 x 8 x 16 tensor-core MMA (weights as the 16-row A side, batch rows as the
// 8-column B side) does the multiply, because at M <= 8 it needs ~5x fewer
// instructions per weight byte than CUDA-core FMAs.  Work is split into items
// (16 rows x one K slice); each CTA takes a contiguous run of items (balanced
// to within one item over all SMs) and its 8 warps split every item's K range,
// so all warps of a CTA finish together.  When K is split into several slices,
// the last CTA to finish a row tile (an atomic arrival counter, no waiting)
// sums the slice partials in fixed order and runs the epilogue.
//
// K permutation: a lane of the MMA fragment owns k pairs {2c, 2c+1} and
// {2c+8, 2c+9} of a 16-wide k block.  Each lane instead loads 8 contiguous
// weights (16 bytes) and the B operand is read with the same permutation, so
// the dot product is unchanged while every load is a full 128-bit access.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace ds {

template <WKind WK> struct Geom {
  static constexpr int BLK_K = (WK == WKind::I8) ? 64 : 32;  // k per load block (16 B per lane)
  static constexpr int PAD = (WK == WKind::I8) ? 8 : 32;     // x row pad, elements (bank spread)
};

constexpr int kDepth = 4;  // warp steps of weights in flight (register ring)

template <int NT> struct SmemLayout {
  // x slice (hi, and lo for bf16), then reduction buffers, tile values, stats, flag
  static __host__ __device__ size_t xs_bytes(int K_S, int pad, bool split) {
    return (size_t)(split ? 2 : 1) * 8 * NT * (K_S + pad) * 2;
  }
  static __host__ __device__ size_t red_floats() { return (size_t)2 * kWarps * NT * 128; }
  static __host__ __device__ size_t total(int K_S, int pad, bool split) {
    return xs_bytes(K_S, pad, split) + 4 * (red_floats() + 16 * 8 * NT + 2 * 8 * NT) + 16;
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
  uint4 a[4];             // [row r (g, g+8)][block]
  unsigned short sc[4];   // int8 only: fp16 scale bits, [row r][block]
};

template <Region R, WKind WK, typename ACT, int NT>
__global__ void __launch_bounds__(kThreads, 2) region_gemv_kernel(const RegionArgs a) {
  using G = Geom<WK>;
  using L = SmemLayout<NT>;
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;  // hi + lo bf16 operand
  constexpr int ROWS = 8 * NT;
  extern __shared__ __align__(16) unsigned char smem_raw[];

  const int K_S = a.plan.K_S;
  const int XS = K_S + G::PAD;  // x row stride, elements
  ACT* xs_hi = reinterpret_cast<ACT*>(smem_raw);
  ACT* xs_lo = xs_hi + ROWS * XS;
  float* red = reinterpret_cast<float*>(smem_raw + L::xs_bytes(K_S, G::PAD, kSplit));
  float* tileval = red + L::red_floats();  // [16][ROWS]
  float* s_mean = tileval + 16 * ROWS;     // [ROWS]
  float* s_rstd = s_mean + ROWS;           // [ROWS]
  int* s_flag = reinterpret_cast<int*>(s_rstd + ROWS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int N = a.N, K = a.K, M = a.M;
  const int tiles = a.plan.tiles, items = a.plan.items, KS = a.plan.KS;
  const int nblk = a.plan.nblk;
  const int step_k = nblk * G::BLK_K;
  const int ib = (int)(((long long)blockIdx.x * items) / gridDim.x);
  const int ie = (int)(((long long)(blockIdx.x + 1) * items) / gridDim.x);
  const int kw = K_S / kWarps;  // k per warp per item
  const int spi = kw / step_k;  // warp steps per item
  const int nsteps = (ie - ib) * spi;

  // ---- weight loads for warp step j (item ib + j / spi, sub-step j % spi)
  auto load = [&](int j, Slot& sl) {
    const int q = j / spi;
    const int sub = j - q * spi;
    const int it = ib + q;
    const int s = it / tiles;
    const int t = it - s * tiles;
    const int kg = s * K_S + warp * kw + sub * step_k;
    const size_t row = (size_t)t * 16 + g;
    if constexpr (WK == WKind::I8) {
      const int8_t* W = static_cast<const int8_t*>(a.W);
      const unsigned short* S = reinterpret_cast<const unsigned short*>(a.Wscale);
      const int gpr = K / 64;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        sl.a[r * 2] = ld_stream(W + (row + 8 * r) * K + kg + 16 * c);
        sl.sc[r * 2] = ld_stream_u16(S + (row + 8 * r) * gpr + kg / 64);
        if (nblk == 2) {
          sl.a[r * 2 + 1] = ld_stream(W + (row + 8 * r) * K + kg + 64 + 16 * c);
          sl.sc[r * 2 + 1] = ld_stream_u16(S + (row + 8 * r) * gpr + kg / 64 + 1);
        }
      }
    } else {
      const uint16_t* W = static_cast<const uint16_t*>(a.W);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        sl.a[r * 2] = ld_stream(W + (row + 8 * r) * K + kg + 8 * c);
        if (nblk == 2) sl.a[r * 2 + 1] = ld_stream(W + (row + 8 * r) * K + kg + 32 + 8 * c);
      }
    }
  };

  // ---- MMAs of one warp step against the staged x slice
  auto compute = [&](const Slot& sl, int sub, float (&acc)[NT][4]) {
    const int kl = warp * kw + sub * step_k;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      if (blk == 1 && nblk == 1) break;
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
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float tmp[4] = {0.f, 0.f, 0.f, 0.f};
          const ACT* xr = xs_hi + (nt * 8 + g) * XS + kl + blk * 64 + 16 * c;
          const uint4 X0 = *reinterpret_cast<const uint4*>(xr);
          const uint4 X1 = *reinterpret_cast<const uint4*>(xr + 8);
          const uint32_t xw[8] = {X0.x, X0.y, X0.z, X0.w, X1.x, X1.y, X1.z, X1.w};
#pragma unroll
          for (int m = 0; m < 4; ++m)
            Mma<ACT>::run(tmp, lo0[m], lo1[m], hi0[m], hi1[m], xw[2 * m], xw[2 * m + 1]);
          if constexpr (kSplit) {
            const ACT* xl = xs_lo + (nt * 8 + g) * XS + kl + blk * 64 + 16 * c;
            const uint4 Y0 = *reinterpret_cast<const uint4*>(xl);
            const uint4 Y1 = *reinterpret_cast<const uint4*>(xl + 8);
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
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const ACT* xr = xs_hi + (nt * 8 + g) * XS + kl + blk * 32 + 8 * c;
          const uint4 X = *reinterpret_cast<const uint4*>(xr);
          Mma<ACT>::run(acc[nt], A0.x, A1.x, A0.y, A1.y, X.x, X.y);
          Mma<ACT>::run(acc[nt], A0.z, A1.z, A0.w, A1.w, X.z, X.w);
          if constexpr (kSplit) {
            const uint4 Y = *reinterpret_cast<const uint4*>(xs_lo + (nt * 8 + g) * XS + kl +
                                                            blk * 32 + 8 * c);
            Mma<ACT>::run(acc[nt], A0.x, A1.x, A0.y, A1.y, Y.x, Y.y);
            Mma<ACT>::run(acc[nt], A0.z, A1.z, A0.w, A1.w, Y.z, Y.w);
          }
        }
      }
    }
  };

  // ---- stage x[:, slice s] into shared memory (region prologue fused here)
  auto stage = [&](int s) {
    const int k0 = s * K_S;
    const int cpr = K_S / 8;
    for (int idx = tid; idx < ROWS * cpr; idx += kThreads) {
      const int n = idx / cpr;
      const int kc = (idx - n * cpr) * 8;
      float v[8];
      if (n < M) {
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
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
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

  // ---- region epilogue for one output (global row n, batch row m)
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
          cache[(((size_t)b * a.heads + head) * a.max_len + pos) * a.head_dim + dim] =
              Act<ACT>::from_f(v);
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

  constexpr int VPT = (16 * ROWS + kThreads - 1) / kThreads;  // reduced values per thread
  constexpr bool kStats = (R == Region::OprojRes || R == Region::FfnDown);

  // ---- item complete: reduce the 8 warps' partial tiles, then split-K
  //      fix-up or direct epilogue (the GEMM reduction boundary).
  auto finish = [&](int t, int s, float (&acc)[NT][4], int buf) {
    float* rb = red + buf * (kWarps * NT * 128);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float* p = rb + (warp * NT + nt) * 128;
      *reinterpret_cast<float2*>(p + g * 8 + 2 * c) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(p + (g + 8) * 8 + 2 * c) = make_float2(acc[nt][2], acc[nt][3]);
      acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    }
    __syncthreads();
    float val[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = tid + i * kThreads;
      val[i] = 0.f;
      if (v < 16 * ROWS) {
        const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
        const int nt = col >> 3, cc = col & 7;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) sum += rb[(w * NT + nt) * 128 + row * 8 + cc];
        val[i] = sum;
      }
    }
    bool last = true;
    if (KS > 1) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * kThreads;
        const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
        if (v < 16 * ROWS && col < M)
          a.partials[((size_t)s * N + t * 16 + row) * M + col] = val[i];
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int prev = atomicAdd(&a.counters[t], 1);
        *s_flag = (prev == KS - 1);
      }
      __syncthreads();
      last = (*s_flag != 0);
      if (last) {
        __threadfence();
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = tid + i * kThreads;
          const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
          if (v < 16 * ROWS && col < M) {
            float sum = 0.f;
            for (int s2 = 0; s2 < KS; ++s2)
              sum += ld_cg(a.partials + ((size_t)s2 * N + t * 16 + row) * M + col);
            val[i] = sum;
          }
        }
        if (tid == 0) a.counters[t] = 0;
      }
    }
    if (last) {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * kThreads;
        const int row = v / ROWS, col = v - (v / ROWS) * ROWS;
        if (v < 16 * ROWS && col < M) {
          const float y = epilogue(t * 16 + row, col, val[i]);
          if constexpr (kStats) tileval[row * ROWS + col] = y;
        }
      }
    }
    if constexpr (kStats) {
      if (a.stats_out != nullptr) {
        __syncthreads();
        if (last && tid < M) {
          float sum = 0.f;
#pragma unroll
          for (int r = 0; r < 16; ++r) sum += tileval[r * ROWS + tid];
          const float mean = sum * (1.0f / 16.0f);
          float m2 = 0.f;
#pragma unroll
          for (int r = 0; r < 16; ++r) {
            const float d = tileval[r * ROWS + tid] - mean;
            m2 += d * d;
          }
          a.stats_out[((size_t)t * M + tid) * 2] = sum;
          a.stats_out[((size_t)t * M + tid) * 2 + 1] = m2;
        }
      }
    }
  };

  // =========================== kernel body ===========================
  Slot ring[kDepth];
#pragma unroll
  for (int d = 0; d < kDepth; ++d)
    if (d < nsteps) load(d, ring[d]);

  pdl_wait();
  pdl_launch_dependents();

  // LayerNorm statistics of the GEMM input (regions 1 and 3/4 prologue): one
  // warp per batch row, either combined from the producer's per-tile partials
  // or, when there are none, computed directly (two passes).
  if constexpr (R == Region::LnQkv || R == Region::FfnUp) {
    for (int n = warp; n < M; n += kWarps) {
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
  int buf = 0;
  for (int j0 = 0; j0 < nsteps; j0 += kDepth) {
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
      const int j = j0 + d;
      if (j < nsteps) {
        const int q = j / spi;
        const int sub = j - q * spi;
        const int it = ib + q;
        const int s = it / tiles;
        const int t = it - s * tiles;
        if (s != cur_s) {
          __syncthreads();
          stage(s);
          __syncthreads();
          cur_s = s;
        }
        compute(ring[d], sub, acc);
        if (j + kDepth < nsteps) load(j + kDepth, ring[d]);
        if (sub == spi - 1) {
          finish(t, s, acc, buf);
          buf ^= 1;
        }
      }
    }
  }

  if constexpr (R == Region::FfnDown) {
    if (a.seq_len_inc != nullptr && blockIdx.x == 0 && tid < a.B) a.seq_len_inc[tid] += 1;
  }
}

// Launches region kernel R for NT chosen by the plan.
template <WKind WK, typename ACT>
cudaError_t launch_region_t(Region r, const RegionArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.plan.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;

#define DS_LAUNCH_NT(REG, NTV) \
  return cudaLaunchKernelEx(&cfg, region_gemv_kernel<REG, WK, ACT, NTV>, a)
#define DS_LAUNCH_REG(REG)              \
  switch (a.plan.nt) {                  \
    case 1: DS_LAUNCH_NT(REG, 1);       \
    case 2: DS_LAUNCH_NT(REG, 2);       \
    case 4: DS_LAUNCH_NT(REG, 4);       \
    case 8: DS_LAUNCH_NT(REG, 8);       \
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
