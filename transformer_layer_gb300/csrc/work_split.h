// Work split of the skinny-GEMM region kernels, shared by the host planner,
// the device kernels and the CPU replay test (tests/work_split_check.cpp).
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持", §3 intro (a skinny GEMM scheduled so that ops
// fuse at its reduction boundary) and §3.1 (CTAs meet only through global
// memory at the reduction boundary).
//
// y[M][N] = x[M][K] W[N][K]^T is cut into units of 16 weight rows x one K
// slice (slice-major: u = s * tiles + t) and every unit into C chunks of
// chunk_k = 8 warps x one warp step along K.  With G CTAs:
//   * CTA c owns the q whole units [c q, (c+1) q) ("data-parallel" units);
//   * the R = (units - q G) C chunks of the leftover units are split into G
//     contiguous ranges [c R / G, (c+1) R / G), processed first.
// A row tile whose result is spread over several CTAs or K slices is summed
// by its last contributor, in fixed order (slice, then CTA), so results are
// deterministic.
#pragma once

#include <stddef.h>

#include "internal.h"

#if defined(__CUDACC__)
#define DS_HD __host__ __device__ __forceinline__
#else
#define DS_HD inline
#endif

namespace ds {

// a / b for a >= 0, b > 0: the 32-bit divide whenever both fit (always, for
// the shapes this library takes), which is far shorter code on the GPU.
DS_HD long long ws_div(long long a, long long b) {
  if ((((unsigned long long)a | (unsigned long long)b) >> 32) == 0) return (long long)((unsigned)a / (unsigned)b);
  return a / b;
}

// The CTA whose leftover range holds leftover chunk i.
DS_HD int ws_cta_of(long long i, long long R, int G) { return (int)ws_div((i + 1) * (long long)G - 1, R); }

// CTA cta's range [ra, rb) of leftover chunks (whole units when P.whole).
DS_HD void ws_left_range(const GemvPlan& P, int cta, int G, long long* ra, long long* rb) {
  if (P.whole) {
    const long long lu = ws_div(P.R, P.C);  // leftover units
    *ra = ws_div((long long)cta * lu, G) * P.C;
    *rb = ws_div((long long)(cta + 1) * lu, G) * P.C;
    return;
  }
  *ra = ws_div((long long)cta * P.R, G);
  *rb = ws_div((long long)(cta + 1) * P.R, G);
}

// Number of CTAs contributing to unit u.  With at least as many leftover
// chunks as CTAs every CTA owns >= 1 of them and a unit's contributors are
// consecutive CTAs; with fewer (a fixed grid larger than the work) every CTA
// owns at most one, so each chunk of a unit has its own CTA.
DS_HD int ws_unit_contrib(int u, const GemvPlan& P, int G) {
  if (u < P.U_dp || P.whole) return 1;
  if (P.R < G) return P.C;
  const long long first = (long long)(u - P.U_dp) * P.C;
  return ws_cta_of(first + P.C - 1, P.R, G) - ws_cta_of(first, P.R, G) + 1;
}

// Partial-sum contributions that complete row tile t (all K slices).
DS_HD int ws_tile_target(int t, const GemvPlan& P, int G) {
  int n = 0;
  for (int s = 0; s < P.KS; ++s) n += ws_unit_contrib(s * P.tiles + t, P, G);
  return n;
}

// First whole unit of CTA cta (the cursors' dp_b), and its i-th.
DS_HD int ws_dp_first(const GemvPlan& P, int cta) { return P.interleave ? cta : cta * P.q; }
DS_HD int ws_dp_unit(const GemvPlan& P, int cta, int i) { return P.interleave ? cta + i * P.grid : cta * P.q + i; }

// Position in a CTA's chunk sequence: leftover chunks first, then whole units.
struct Cursor {
  int s, t, kc;  // slice, row tile, chunk within the unit
  int rem_left;  // leftover chunks still to come, including this one
};

DS_HD void ws_cursor_init(Cursor& q, const GemvPlan& P, long long ra, long long rb, int dp_b) {
  if (rb > ra) {
    const long long uq = ws_div(ra, P.C);
    const long long u = P.U_dp + uq;
    q.kc = (int)(ra - uq * P.C);
    q.s = (int)(u / P.tiles);
    q.t = (int)(u - (long long)q.s * P.tiles);
    q.rem_left = (int)(rb - ra);
  } else {
    q.rem_left = 0;
    q.s = dp_b / P.tiles;
    q.t = dp_b - q.s * P.tiles;
    q.kc = 0;
  }
}

DS_HD void ws_cursor_next(Cursor& q, const GemvPlan& P, int dp_b) {
  if (q.rem_left > 0) {
    if (--q.rem_left == 0) {
      q.s = dp_b / P.tiles;
      q.t = dp_b - q.s * P.tiles;
      q.kc = 0;
      return;
    }
  }
  if (++q.kc == P.C) {
    q.kc = 0;
    if (P.interleave) {  // next whole unit: grid units further on
      const int u = q.s * P.tiles + q.t + P.grid;
      q.s = u / P.tiles;
      q.t = u - q.s * P.tiles;
    } else if (++q.t == P.tiles) {
      q.t = 0;
      ++q.s;
    }
  }
}

// True when the chunk at cursor q is the last of its segment (a segment is a
// run of one CTA's chunks inside one unit); j is the chunk's index in the CTA.
DS_HD bool ws_segment_ends(const Cursor& q, const GemvPlan& P, int j, int nchunks) {
  return q.kc == P.C - 1 || q.rem_left == 1 || j == nchunks - 1;
}

// The epilogue side's view of the leftover segments: starting at leftover
// chunk i of CTA cta, the segment's unit, its end and the CTA's slot among
// the unit's contributors.
DS_HD void ws_leftover_segment(const GemvPlan& P, long long i, long long rb, int cta, int G, int* u,
                               long long* end, int* j_slot) {
  const long long uo = ws_div(i, P.C);
  *end = (uo + 1) * P.C < rb ? (uo + 1) * P.C : rb;
  *u = (int)(P.U_dp + uo);
  *j_slot = P.whole ? 0 : (P.R < G) ? (int)(i - uo * P.C) : cta - ws_cta_of(uo * P.C, P.R, G);
}

// Distributes p.units units of p.C chunks each over at most num_ctas CTAs:
// p.grid, q whole units per CTA, and either whole leftover units or their
// chunks spread evenly (p.whole, p.U_dp, p.R, p.maxc).  p.units and p.C must
// be set.  one_unit_each: when there are no more units than CTAs, give each
// CTA exactly one whole unit (grid = units, nothing split).  force_whole:
// leftover units always go whole to CTAs (no split-K fix-ups).
inline void ws_distribute(GemvPlan& p, int num_ctas, bool one_unit_each = false, bool force_whole = false) {
  if (one_unit_each && p.units <= num_ctas) {
    p.grid = p.units;
    p.q = 1;
    p.whole = 0;
    p.U_dp = p.units;
    p.R = 0;
    p.maxc = 1;
    return;
  }
  const long long total = (long long)p.units * p.C;
  long long G = num_ctas;
  if (G > total) G = total;
  p.grid = (int)G;
  p.q = p.units / p.grid;
  p.whole = 0;
  // Leftover units go whole to CTAs when that lengthens the busiest CTA by at
  // most 3 chunks: a split-K fix-up costs global round trips (several us under
  // the weight stream) that the short kernels cannot hide.
  {
    const long long lu = p.units - (long long)p.q * p.grid;
    const long long whole_max = ((long long)p.q + (lu > 0 ? 1 : 0)) * p.C;
    long long qs = p.q;
    if (qs > 0 && lu * p.C > 0 && lu * p.C < p.grid) qs -= 1;
    const long long rs = (p.units - qs * p.grid) * p.C;
    const long long split_max = qs * p.C + (rs + p.grid - 1) / p.grid;
    if (lu > 0 && (force_whole || whole_max - split_max <= 3)) p.whole = 1;
  }
  // Every CTA must own at least one leftover chunk when there are any (so the
  // CTAs sharing a leftover unit are consecutive, with no empty ranges in
  // between): with fewer leftover chunks than CTAs, hand one whole unit per
  // CTA back to the leftover pool.
  const long long left = (long long)(p.units - p.q * p.grid) * p.C;
  if (!p.whole && p.q > 0 && left > 0 && left < p.grid) p.q -= 1;
  p.U_dp = p.q * p.grid;
  p.R = (long long)(p.units - p.U_dp) * p.C;
  p.maxc = 1;
  for (int u = p.U_dp; u < p.units; ++u) {
    const int n = ws_unit_contrib(u, p, p.grid);
    if (n > p.maxc) p.maxc = n;
  }
}

// Host planner: the longest K slice whose staged x fits `x_budget` bytes, then
// q whole units per CTA and the leftover units' chunks spread evenly.
// xs_bytes(K_S) gives the staged-x bytes for a slice length.
template <typename XsBytes>
inline bool ws_make_plan(int N, int K, int M, int num_ctas, int blk_k, int warps, size_t x_budget,
                         XsBytes xs_bytes, GemvPlan* plan) {
  if (N <= 0 || K <= 0 || M < 1 || M > 64 || (N % 16) != 0 || num_ctas < 1) return false;
  GemvPlan p;
  p.nt = M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 32 ? 4 : 8));
  // k-blocks per warp step: as many as K allows, up to 4 (more bytes per
  // ring handshake), then the longest K slice whose staged x fits the budget.
  p.tiles = N / 16;
  p.K_S = 0;
  for (int nb = 4; nb >= 1 && p.K_S == 0; nb /= 2) {
    if (K % (warps * nb * blk_k) != 0) continue;
    p.nblk = nb;
    p.chunk_k = warps * nb * blk_k;
    const int nck = K / p.chunk_k;
    for (int d = 1; d <= nck; ++d) {
      if (nck % d != 0) continue;
      if (xs_bytes(K / d) <= x_budget) {
        p.K_S = K / d;
        break;
      }
    }
  }
  if (p.K_S == 0) return false;
  p.KS = K / p.K_S;
  p.C = p.K_S / p.chunk_k;
  p.units = p.KS * p.tiles;
  ws_distribute(p, num_ctas);
  *plan = p;
  return true;
}

}  // namespace ds
