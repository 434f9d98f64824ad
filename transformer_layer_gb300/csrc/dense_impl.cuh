// Tensor-core tile path of the region GEMMs (tcgen05 + TMEM), for the batch
// rows at which the skinny GEMM becomes a real dense contraction: decode at
// B*T = 8..64 rows and multi-token (prompt) steps of up to a few thousand rows.
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持".
//   §3 intro: the GEMM is built so that more operations fuse at its reduction
//     boundary -- here the region epilogues run straight out of the tensor
//     memory accumulator.
//   §3.2: regions 1 (LayerNorm + QKV + bias), 3 (FF + LayerNorm + bias +
//     residual + GeLU) and 4 (bias + residual).
//   §3.3: shared memory stages the operands between the reductions.
//
// What one launch computes: y[m][n] = sum_k X[m][k] W[n][k] for m < M (batch
// rows or tokens), n < N, followed by the region epilogue.  The region
// prologue (the LayerNorm) has already been applied to X by the row
// normalisation kernel (or X is the attention / GeLU output), and X is stored
// in the MMA operand format: the activation dtype, plus for bf16 the residual
// lo = bf16(x - bf16(x)) so that hi + lo carries ~16 significant bits.
//
// GB300 design:
//  * One output tile is 128 weight rows x NTOK (16..256) rows of X, held as an
//    fp32 accumulator in tensor memory (two buffers of NTOK columns, so the
//    MMAs of the next tile overlap the epilogue of the previous one).
//  * Warp 0 streams W (128 rows x KC) and X (NTOK rows x KC) chunks with TMA
//    tensor copies (128-byte swizzle, K-major) into a ring of up to 8 stages.
//    The weights of the first stages are requested before griddepcontrol.wait
//    (they do not depend on the previous kernel); X after it.
//  * Warp 1 allocates the tensor memory and one lane issues tcgen05.mma
//    (kind::f16, M = 128, N = NTOK, K = 16 per instruction; bf16 issues the lo
//    operand as a second MMA into the same accumulator) and tcgen05.commit to
//    release ring stages and to publish finished tiles.  At up to 64 token
//    rows (and for int8) a second issuing warp, the last, takes every other
//    chunk into its own accumulator pair: one thread issues an MMA only every
//    ~50-120 cycles, whatever N (see dense_issuers).
//  * Warps 2..9 read the accumulator with tcgen05.ld (warp w owns TMEM lanes
//    32 (w % 4) ..: one weight row per thread; the two warps of a lane
//    quarter take alternate groups of 8 token columns) and run the region
//    epilogue.  When the K slices of a tile run as one cluster (one slice
//    per CTA) their partial tiles are summed through distributed shared
//    memory; otherwise a shared tile's partials go through global memory and
//    its last contributor (acquire-release counter, nothing waits) stages them
//    in its idle ring with bulk copies and sums them in fixed order.  Results
//    are deterministic either way.
//  * int8 weights: warps 10..17 dequantise each stage's codes to fp16 straight
//    into tensor memory (tcgen05.st), where the MMAs read them as the A
//    operand: the fp16 weights never pass through shared memory (see the
//    converter role below).
//  * Work split (work_split.h): a unit is one output tile x one K slice,
//    chunks are KC-wide K ranges.  With at least ~60 % as many tiles as SMs
//    each CTA takes one whole tile (no split-K); with fewer (N = 4096 at
//    decode) each tile is cut into K slices, one per CTA, a cluster per tile
//    (slices of unequal length where that fills more SMs: 3 for N = 5120);
//    with more, CTAs own whole tiles (round-robin when several token tiles
//    share the weights) and, at decode, an even share of the leftover tiles'
//    chunks.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "work_split.h"
#include "dense_plan.h"

namespace ds {

constexpr int kDenseEpiWarps = 8;    // two per TMEM lane quarter, each taking half the columns
constexpr int kDenseConvWarps = 8;   // int8 weights: warps that dequantise the codes to fp16
constexpr int kDenseTmaWarp = 0;
constexpr int kDenseMmaWarp = 1;
constexpr int kDenseEpiWarp0 = 2;    // warps 2 .. 9
constexpr int kDenseConvWarp0 = 10;  // int8: warps 10 .. 10 + kDenseConvWarps - 1
// the second MMA issuer: after the epilogue warps (int8: after the converters)
__host__ __device__ constexpr int dense_mma2_warp(bool i8) {
  return i8 ? kDenseConvWarp0 + kDenseConvWarps : kDenseEpiWarp0 + kDenseEpiWarps;
}
// threads of a tile CTA with nis MMA issuers
__host__ __device__ constexpr int dense_threads(bool i8, int nis) {
  return (1 + nis + kDenseEpiWarps + (i8 ? kDenseConvWarps : 0)) * 32;
}
constexpr int kDenseEpiThreads = kDenseEpiWarps * 32;
constexpr int kDenseBarEpi = 1;      // named barrier of the eight epilogue warps
constexpr int kL2Ahead = 8;            // weight chunks requested into L2 ahead of the ring

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor of a K-major operand tile in the canonical
// 128-byte-swizzle layout: rows of 128 bytes (64 16-bit elements), groups of
// 8 rows 1024 bytes apart (stride byte offset), descriptor version 1,
// swizzle mode 2 (128 B).  Advancing K by 16 elements inside the 128-byte row
// adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, A and B fp16 (0) or
// bf16 (1), both K-major, N >> 3 at bit 17, M >> 4 (M = 128) at bit 24.
__device__ __forceinline__ uint32_t umma_idesc(bool bf16, int n) {
  return (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)(n >> 3) << 17) | (8u << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(acc));
}
// The same with A (M = 128 rows x K = 16, one row per TMEM lane, two 16-bit
// elements per 32-bit column, the lower K index in the low half) read from
// tensor memory at column address tmem_a.
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t db, uint32_t idesc,
                                                uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(db), "r"(idesc), "r"(acc));
}
// Arrives on `bar` once every tcgen05.mma issued so far by this thread is complete.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Stores 32 consecutive 32-bit columns of this thread's TMEM lane (the warp
// writes its lane quarter); tmem_wait_st waits until they have landed.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 8 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- geometry
// A role's position in the ring (same convention as the GEMV ring).
struct DRing {
  int st = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void advance(int S) {
    if (++st == S) {
      st = 0;
      ph ^= 1;
    }
  }
};

// Segment enumeration shared by the three roles: leftover segments of CTA
// `cta` (its place in the work split), then its whole units.
// f(u, kc0, kc1, j_slot) per segment.
template <typename F>
__device__ __forceinline__ void dense_for_segments(const GemvPlan& P, int cta, F&& f) {
  const int G = gridDim.x;
  long long ra, rb;
  ws_left_range(P, cta, G, &ra, &rb);
  for (long long i = ra; i < rb;) {
    int u, j_slot;
    long long end;
    ws_leftover_segment(P, i, rb, cta, G, &u, &end, &j_slot);
    const int kc0 = (int)(i - (long long)(u - P.U_dp) * P.C);
    f(u, kc0, kc0 + (int)(end - i), j_slot);
    i = end;
  }
  for (int i = 0; i < P.q; ++i) f(ws_dp_unit(P, cta, i), 0, P.C, 0);
}

// Distributed shared memory: a float of CTA `rank` of this cluster at the
// offset of `local_addr` in this CTA.
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes
// before it are visible to the cluster's reads after it.
__device__ __forceinline__ void dense_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// kI8: W is int8 codes with fp16 scales per group of qgroup along K (MoQ);
// the converter warps dequantise each stage's codes to fp16 (q * s rounded
// once to fp16, the MMA operand type) before its MMAs.
// NIS: MMA issuers (dense_issuers of the plan; the launch picks the instance).
template <Region R, typename ACT, bool kI8, int NIS>
__global__ void __launch_bounds__(dense_threads(kI8, NIS), 1)
    dense_region_kernel(const __grid_constant__ CUtensorMap xmap_hi, const __grid_constant__ CUtensorMap xmap_lo,
                        const DenseArgs a) {
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;
  static_assert(!kI8 || !kSplit, "int8 tiles take fp16 activations");
  constexpr bool kStats = (R == Region::OprojRes || R == Region::FfnDown);
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  const DensePlan& DP = a.plan;
  const GemvPlan& P = DP.ws;
  const int S = DP.stages, KC = DP.kc, NTOK = DP.ntok;
  const size_t WB = dense_w_bytes(KC), XB = dense_x_bytes(NTOK, KC);
  const size_t SB = (dense_stage_bytes(NTOK, KC, kSplit, kI8) + 1023) & ~(size_t)1023;
  const uint32_t XOFF = kI8 ? (uint32_t)(128 * KC) : (uint32_t)WB;  // X within a stage
  const uint32_t SOFF = XOFF + (uint32_t)XB;                         // int8: the scale box within a stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + (size_t)S * SB);
  // full[S], empty[S], acc_full[2], acc_empty[2], fix, done, (int8)
  // wfull[kDenseWTiles], wempty[kDenseWTiles], xfull[S]
  auto full_bar = [&](int i) { return smem_u32(bars + i); };
  auto empty_bar = [&](int i) { return smem_u32(bars + S + i); };
  auto accf_bar = [&](int i) { return smem_u32(bars + 2 * S + i); };
  auto acce_bar = [&](int i) { return smem_u32(bars + 2 * S + 2 + i); };
  const uint32_t fix_bar = smem_u32(bars + 2 * S + 4);   // staged partials of a fix-up
  const uint32_t done_bar = smem_u32(bars + 2 * S + 5);  // epilogue warps done with TMEM
  // int8: fp16 W tile i written (converter warps) / read by the MMAs (commit)
  auto wfull_bar = [&](int i) { return smem_u32(bars + 2 * S + 6 + i); };
  auto wempty_bar = [&](int i) { return smem_u32(bars + 2 * S + 6 + kDenseWTiles + i); };
  // int8, a stage's first use (the S chunks requested before the dependency
  // wait): its full barrier counts the codes and scales only, which do not
  // depend on the previous kernel, so the converters start on them before
  // the wait; its X (after the wait) completes xfull, which the MMAs wait
  // for.  Later uses count codes, scales and X on full.
  auto xfull_bar = [&](int i) { return smem_u32(bars + 2 * S + 6 + 2 * kDenseWTiles + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 6 + 2 * kDenseWTiles);
  int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);
  static_assert(NIS == 1 || NIS == kDenseMaxIssuers, "one or two MMA issuers");
  static_assert(!kI8 || NIS == kDenseMaxIssuers, "int8 issuers own W tiles: two of them");
  constexpr int nis = NIS;
  const uint32_t tcols = dense_tmem_cols(NTOK, nis, kI8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 32) {  // the descriptors' first use is the TMA warp's first copy
    if (a.sel_idx == nullptr) asm volatile("prefetch.tensormap [%0];" ::"l"(a.tmap_w) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap_hi) : "memory");
    if (kSplit) asm volatile("prefetch.tensormap [%0];" ::"l"(&xmap_lo) : "memory");
    if (kI8) asm volatile("prefetch.tensormap [%0];" ::"l"(a.tmap_s) : "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(accf_bar(i), nis);  // one commit per MMA issuer
      mbar_init(acce_bar(i), kDenseEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(fix_bar, 1);
    mbar_init(done_bar, kDenseEpiWarps);
    if (kI8) {
      for (int i = 0; i < kDenseWTiles; ++i) {
        mbar_init(wfull_bar(i), kDenseConvWarps);
        mbar_init(wempty_bar(i), 1);
      }
      for (int i = 0; i < S; ++i) mbar_init(xfull_bar(i), 1);
    }
    mbar_init_fence();
  }
  if (warp == kDenseMmaWarp) tmem_alloc(smem_u32(tmem_slot), tcols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Tile t covers weight rows [128 (t / tok_tiles), +128) and X rows
  // [NTOK (t % tok_tiles), +NTOK): the token tiles of one weight tile are
  // consecutive units, so CTAs that run at the same time share its weights
  // through L2.
  const int tok_tiles = DP.tok_tiles;
  // Place in the work split: with a cluster per tile, CTA rank s of cluster t
  // takes K slice s of tile t (unit s * tiles + t).
  const int KSC = DP.cluster;
  const int vcta = KSC > 1 ? (int)(blockIdx.x % KSC) * P.tiles + (int)(blockIdx.x / KSC) : (int)blockIdx.x;
  // K slice sl's first chunk along K: a cluster's slices share the K chunks
  // as evenly as they go (their lengths differ by one at most; a cluster CTA
  // only ever asks for its own slice, computed once here), otherwise every
  // slice holds P.C chunks.
  const int cl_c0 = KSC > 1 ? (vcta / P.tiles) * DP.kchunks / KSC : 0;
  const int cl_len = KSC > 1 ? (vcta / P.tiles + 1) * DP.kchunks / KSC - cl_c0 : 0;
  auto slice_c0 = [&](int sl) { return KSC > 1 ? cl_c0 : sl * P.C; };
  // This CTA's segments, f(unit, first chunk, end chunk, slot) -- with a
  // cluster, its one whole slice.
  auto for_segments = [&](auto&& f) {
    if (KSC > 1) f(vcta, 0, cl_len, 0);
    else dense_for_segments(P, vcta, f);
  };

  if (warp == kDenseTmaWarp) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      // the weights of an expert chosen by the previous kernels: wait first
      const void* tmap_w = a.tmap_w;
      if (a.sel_idx != nullptr) {
        pdl_wait();
        tmap_w = a.tmap_table + (size_t)128 * (size_t)(*a.sel_idx);
      }
      // weights read once: evict first; read again by other token tiles: keep
      const uint64_t pol_w = tok_tiles > 1 ? l2_evict_normal_policy() : l2_evict_first_policy();
      const uint64_t pol_x = l2_evict_normal_policy();
      // bytes a stage's full barrier counts (int8, first use: X goes to xfull)
      const uint32_t tx = (uint32_t)((kI8 ? (size_t)128 * KC : WB) + (kSplit ? 2 : 1) * XB + dense_scale_bytes(kI8));
      const uint32_t tx_first = kI8 ? tx - (uint32_t)XB : tx;
      const int qshift = kI8 ? 31 - __clz(a.qgroup) : 0;
      const uint32_t woff = 0u;                                    // where W's copy lands
      auto wk_of = [&](const Cursor& c) {                          // W's K coordinate (128-byte atoms)
        return (slice_c0(c.s) + c.kc) * (kI8 ? KC / 128 : KC / 64);
      };
      // int8: the stage's scale box, the aligned 8 groups holding its first
      // (K is a multiple of 8 groups, so the box never leaves the matrix)
      auto load_scales = [&](uint32_t stage, const Cursor& c, int trow, uint32_t bar) {
        if constexpr (kI8) {
          const int g0 = (((slice_c0(c.s) + c.kc) * KC) >> qshift) & ~(kDenseScaleGroups - 1);
          tma_load_2d(stage + SOFF, a.tmap_s, g0, trow * 128, bar, pol_x);
        }
      };
      long long ra, rb;
      ws_left_range(P, vcta, gridDim.x, &ra, &rb);
      const int dp_b = ws_dp_first(P, vcta);
      const int nchunks = KSC > 1 ? cl_len : (int)(rb - ra) + P.q * P.C;
      bool dead = false;
      uint32_t last_ph[kDenseMaxStagesDev];  // parity of the last copy issued into each stage
      uint32_t issued = 0;                   // stages that received a copy (bit mask)
      // The first stages' weights before the dependency wait, their X after it.
      const int pre = nchunks < S ? nchunks : S;
      Cursor q;
      ws_cursor_init(q, P, ra, rb, dp_b);
      Cursor q0 = q;
      DRing rp;
      for (int j = 0; j < pre; ++j) {
        const uint32_t stage = smem_u32(sm + (size_t)rp.st * SB);
        const int trow = q.t / tok_tiles;
        mbar_arrive_expect_tx(full_bar(rp.st), tx_first);
        tma_load_3d(stage + woff, tmap_w, 0, trow * 128, wk_of(q), full_bar(rp.st), pol_w);
        load_scales(stage, q, trow, full_bar(rp.st));
        last_ph[rp.st] = rp.ph;
        issued |= 1u << rp.st;
        ws_cursor_next(q, P, dp_b);
        rp.advance(S);
      }
      // In-kernel L2 lookahead: the weight chunks after the ring's are
      // requested from HBM into L2 (no shared memory needed), kL2Ahead ahead
      // of the copy into the ring, so that the stream's bytes in flight do not
      // depend on the ring depth.
      Cursor qp = q;
      int fpre = pre;
      auto l2_ahead = [&](int upto) {
        for (; fpre < upto && fpre < nchunks; ++fpre) {
          tma_prefetch_3d(tmap_w, 0, (qp.t / tok_tiles) * 128, wk_of(qp));
          ws_cursor_next(qp, P, dp_b);
        }
      };
      pdl_wait();
      pdl_launch_dependents();
      {
        DRing r2;
        Cursor c = q0;
        for (int j = 0; j < pre; ++j) {
          const uint32_t stage = smem_u32(sm + (size_t)r2.st * SB);
          const int jt = c.t % tok_tiles;
          const int kseg = (slice_c0(c.s) + c.kc) * (KC / 64);
          if constexpr (kI8) mbar_arrive_expect_tx(xfull_bar(r2.st), (uint32_t)XB);
          tma_load_3d(stage + XOFF, &xmap_hi, 0, jt * NTOK, kseg, kI8 ? xfull_bar(r2.st) : full_bar(r2.st), pol_x);
          if constexpr (kSplit)
            tma_load_3d(stage + XOFF + (uint32_t)XB, &xmap_lo, 0, jt * NTOK, kseg, full_bar(r2.st), pol_x);
          ws_cursor_next(c, P, dp_b);
          r2.advance(S);
        }
      }
      // (after the first X copies, which would otherwise queue behind it)
      l2_ahead(pre + kL2Ahead);
      for (int j = pre; j < nchunks; ++j) {
        if (!dead) dead = !mbar_wait(empty_bar(rp.st), rp.ph ^ 1, a.status);
        if (dead) break;
        const uint32_t stage = smem_u32(sm + (size_t)rp.st * SB);
        const int trow = q.t / tok_tiles, jt = q.t % tok_tiles;
        const int kseg = (slice_c0(q.s) + q.kc) * (KC / 64);
        mbar_arrive_expect_tx(full_bar(rp.st), tx);
        tma_load_3d(stage + woff, tmap_w, 0, trow * 128, wk_of(q), full_bar(rp.st), pol_w);
        load_scales(stage, q, trow, full_bar(rp.st));
        tma_load_3d(stage + XOFF, &xmap_hi, 0, jt * NTOK, kseg, full_bar(rp.st), pol_x);
        if constexpr (kSplit)
          tma_load_3d(stage + XOFF + (uint32_t)XB, &xmap_lo, 0, jt * NTOK, kseg, full_bar(rp.st), pol_x);
        last_ph[rp.st] = rp.ph;
        issued |= 1u << rp.st;
        ws_cursor_next(q, P, dp_b);
        rp.advance(S);
        // (int8: the ring of 16 KB code stages already holds more than the
        // latency needs, and one more bulk instruction per chunk would cost
        // this thread ~600 cycles that it is short of)
        if constexpr (!kI8) l2_ahead(j + 1 + kL2Ahead);
      }
      // No copy may still be landing in this CTA's shared memory when it
      // exits: wait (bounded) for the last copy of every stage.  Immediate in
      // normal operation, where the MMA thread has consumed them all.
      for (int st = 0; st < S; ++st)
        if ((issued >> st) & 1u) {
          mbar_wait(full_bar(st), last_ph[st], a.status);
          if (kI8) mbar_wait(xfull_bar(st), 0, a.status);  // (every issued stage had a first use)
        }
      // L2 prefetch of the next GEMM's first weight chunks for this CTA index.
      if (a.next_tmap_w != nullptr && blockIdx.x < a.next_plan.ws.grid) {
        const GemvPlan& Pn = a.next_plan.ws;
        long long na, nb;
        ws_left_range(Pn, blockIdx.x, Pn.grid, &na, &nb);
        const int ndp = ws_dp_first(Pn, blockIdx.x);
        int nn = (int)(nb - na) + Pn.q * Pn.C;
        if (nn > 16) nn = 16;
        Cursor c;
        ws_cursor_init(c, Pn, na, nb, ndp);
        for (int j = 0; j < nn; ++j) {
          tma_prefetch_3d(a.next_tmap_w, 0, (c.t / a.next_plan.tok_tiles) * 128, c.kc * a.next_plan.kc / 64);
          ws_cursor_next(c, Pn, ndp);
        }
      }
    }
    if (KSC > 1) {  // the cluster reduction's two barriers (every thread takes part)
      __syncwarp();
      dense_cluster_sync();
      dense_cluster_sync();
    }
  } else if (warp == kDenseMmaWarp || (nis > 1 && warp == dense_mma2_warp(kI8))) {
    // ---------------------------------------------------------- MMA issuer(s)
    // Issuer me of nis (dense_issuers) takes the CTA's chunks j with
    // j % nis == me -- with two issuers exactly those of its ring stages
    // (fp16 / bf16) or W tiles (int8), so it observes every phase of the
    // barriers it waits on in order (a waiter that skipped a phase would take
    // an older completion for the one it waits for) -- into its own
    // accumulator pair (columns 2 NTOK me ..); the epilogue sums them.
    pdl_launch_dependents();
    const int me = warp == kDenseMmaWarp ? 0 : 1;
    static_assert(kDenseWTiles % 4 == 0 && kDenseWTiles % 2 == 0, "int8: issuer i owns the W tiles i, i + nis, ...");
    if (lane == 0) {
      const uint32_t idesc = umma_idesc(kSplit, NTOK);
      DRing rp;
      int seg = 0;
      int wj = 0;  // int8: chunks so far (W tile wj % kDenseWTiles, its use wj / kDenseWTiles)
      bool dead = false;
      for_segments([&](int u, int kc0, int kc1, int) {
        (void)u;
        const int buf = seg & 1;
        if (seg >= 2 && !dead) dead = !mbar_wait(acce_bar(buf), ((seg >> 1) - 1) & 1, a.status);
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)((2 * me + buf) * NTOK);
        bool first = true;  // this issuer's first chunk of the tile: overwrite the accumulator
        for (int kc = kc0; kc < kc1; ++kc) {
          const int wslot = wj % kDenseWTiles;
          if (wj % nis == me) {
            // int8: the converters have waited for this stage and filled W tile wslot
            if (kI8 && !dead) dead = !mbar_wait(wfull_bar(wslot), (uint32_t)((wj / kDenseWTiles) & 1), a.status);
            // the stage's X (int8: its codes were waited for by the converters)
            if (!dead) dead = !mbar_wait((kI8 && wj < S) ? xfull_bar(rp.st) : full_bar(rp.st), rp.ph, a.status);
            if (!dead) {
              tc_fence_after();
              // Descriptors built once per chunk and advanced by their address
              // field (16-byte units; a stage never crosses the field's range):
              // per-MMA operand arithmetic would add to the issue time.
              const uint32_t sbase = smem_u32(sm + (size_t)rp.st * SB);
              const uint64_t xd0 = umma_desc_sw128(sbase + XOFF);
              const uint64_t wd0 = umma_desc_sw128(sbase);
              const uint32_t acc0 = first ? 0u : 1u;
              // int8: W tile wslot in tensor memory, 8 columns per K step of 16
              const uint32_t wcol = tmem + (uint32_t)(2 * nis * NTOK + wslot * kDenseWTileCols);
#pragma unroll 1
              for (int kb = 0; kb < KC / 64; ++kb) {
                const uint64_t xk = xd0 + (uint64_t)(kb * NTOK * 8);  // NTOK rows of 128 B per 64 K
                const uint64_t wk = wd0 + (uint64_t)(kb * 1024);      // 128 rows of 128 B per 64 K
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16) {
                  const uint32_t acc = (kb > 0 || k16 > 0) ? 1u : acc0;
                  const uint64_t xd = xk + (uint64_t)(2 * k16);      // 32 bytes per K step of 16
                  if constexpr (kI8) {
                    umma_f16_tmem_a(d, wcol + (uint32_t)(8 * (4 * kb + k16)), xd, idesc, acc);
                  } else {
                    const uint64_t dw = wk + (uint64_t)(2 * k16);
                    umma_f16(d, dw, xd, idesc, acc);
                    if constexpr (kSplit) umma_f16(d, dw, xd + (uint64_t)(XB >> 4), idesc, 1u);
                  }
                }
              }
              umma_commit(empty_bar(rp.st));
              if (kI8) umma_commit(wempty_bar(wslot));
            }
            first = false;
          }
          rp.advance(S);
          ++wj;
        }
        if (!dead) umma_commit(accf_bar(buf));
        ++seg;
      });
    }
    if (KSC > 1) {
      __syncwarp();
      dense_cluster_sync();
      dense_cluster_sync();
    }
  } else if (kI8 && warp >= kDenseConvWarp0 && warp < kDenseConvWarp0 + kDenseConvWarps) {
    // ---------------------------------------------------------- int8 dequantisation
    // Thread (row r, half h): weight row r = 32 (warp % 4) + lane -- the TMEM
    // lane its warp may write -- and half h of a stage's 128 codes (the two
    // warps of a lane quarter take one half each).  Stage layout of the codes:
    // [128 rows][128 B], 16-byte chunk c of row r at physical chunk
    // c ^ (r & 7); the thread reads chunks 4h .. 4h + 3 of its row (the 32
    // rows of a warp spread over the 8 physical positions: no bank conflict
    // beyond the 4 wavefronts of 512 bytes), converts the 64 codes to fp16,
    // multiplies them by their group's scale (a group of 64 or more codes
    // covers the half) and stores the 32 columns of fp16 pairs into W tile
    // j % kDenseWTiles once the MMAs of chunk j - kDenseWTiles have released it.
    const int cw = warp - kDenseConvWarp0;
    const int h = cw >> 2;
    const int r = 32 * (warp & 3) + lane;
    const uint32_t rx = (uint32_t)(r & 7);
    const int qshift = 31 - __clz(a.qgroup);
    const uint32_t tlane =
        tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(2 * nis * NTOK + 32 * h);
    DRing rp;
    int wj = 0;
    bool dead = false;
    for_segments([&](int u, int kc0, int kc1, int) {
      const int sl = u / P.tiles;
      for (int kc = kc0; kc < kc1; ++kc) {
        const int wslot = wj % kDenseWTiles;
        if (!dead) dead = !mbar_wait(full_bar(rp.st), rp.ph, a.status);
        if (!dead) dead = !mbar_wait(wempty_bar(wslot), (uint32_t)(((wj / kDenseWTiles) & 1) ^ 1), a.status);
        dead = __any_sync(0xffffffffu, dead);  // the TMEM store below is warp-collective
        if (!dead) {
          tc_fence_after();
          const uint32_t sbase = smem_u32(sm + (size_t)rp.st * SB);
          const int k0 = (slice_c0(sl) + kc) * KC + 64 * h;  // K index of the thread's first code
          // its group, as an index into the stage's scale box (the aligned
          // block of kDenseScaleGroups holding the stage's first group)
          const uint32_t g = (uint32_t)((k0 >> qshift) & (kDenseScaleGroups - 1));
          const uint32_t sv = lds_u16(sbase + SOFF + (uint32_t)r * (2u * kDenseScaleGroups) + 2u * g);
          const uint32_t s2u = sv | (sv << 16);
          const __half2 s2 = *reinterpret_cast<const __half2*>(&s2u);
          uint32_t hv[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = lds_u128(sbase + (uint32_t)r * 128u + (((uint32_t)(4 * h + i) ^ rx) * 16u));
            i8x4_to_half2x2(v.x, hv[8 * i + 0], hv[8 * i + 1]);
            i8x4_to_half2x2(v.y, hv[8 * i + 2], hv[8 * i + 3]);
            i8x4_to_half2x2(v.z, hv[8 * i + 4], hv[8 * i + 5]);
            i8x4_to_half2x2(v.w, hv[8 * i + 6], hv[8 * i + 7]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const __half2 y = __hmul2(*reinterpret_cast<const __half2*>(&hv[j]), s2);
            hv[j] = *reinterpret_cast<const uint32_t*>(&y);
          }
          tmem_st32(tlane + (uint32_t)(wslot * kDenseWTileCols), hv);
          tmem_wait_st();
        }
        // the W tile is read by the tensor cores once every converter warp arrived
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(wfull_bar(wslot));
        rp.advance(S);
        ++wj;
      }
    });
    if (KSC > 1) {
      __syncwarp();
      dense_cluster_sync();
      dense_cluster_sync();
    }
  } else {
    // ---------------------------------------------------------- epilogue
    pdl_wait();
    pdl_launch_dependents();
    const int et = threadIdx.x - kDenseEpiWarp0 * 32;  // 0 .. kDenseEpiThreads-1
    const int qd = warp & 3;                            // TMEM lane quarter
    const int r = 32 * qd + lane;                       // weight row within the tile
    const int cbeg = 8 * ((warp - kDenseEpiWarp0) >> 2); // this warp's first 8-column group; stride 16
    const int M = a.M, N = a.N;
    // One output tile as this thread sees it: weight row n, token columns
    // [m0, m0 + mrows), and the row's epilogue invariants.
    struct TileCtx {
      int t, n, m0, mrows;
      float bias;
      float scale;      // expert output weight (residual-MoE), else 1
      ACT* dst;         // R1: the row's KV-cache element of (b, position) 0; R4a / R4b: output column n
      ACT* dst_lo;      // R4a, bf16: operand lo column n
      float* dst_f32;   // R1 (q rows): q column; R3: x1 column n
      bool to_cache;    // R1: this row is a k or v row
    };
    auto tile_ctx = [&](int t) {
      TileCtx c;
      c.t = t;
      c.n = (t / tok_tiles) * 128 + r;
      c.m0 = (t % tok_tiles) * NTOK;
      c.mrows = min(NTOK, M - c.m0);
      const int bsel = a.sel_idx != nullptr ? a.sel_bias_stride * (*a.sel_idx) : 0;
      c.bias = a.bias != nullptr ? Act<ACT>::to_f(static_cast<const ACT*>(a.bias)[bsel + c.n]) : 0.f;
      c.scale = a.sel_scale != nullptr ? *a.sel_scale : 1.0f;
      c.dst = nullptr;
      c.dst_lo = nullptr;
      c.dst_f32 = nullptr;
      c.to_cache = false;
      if constexpr (R == Region::LnQkv) {
        const int part = c.n / a.H, within = c.n - part * a.H;
        if (part == 0) {
          c.dst_f32 = a.out_f32 + within;
        } else {
          const int head = within / a.head_dim, dim = within - head * a.head_dim;
          c.dst = static_cast<ACT*>(part == 1 ? a.k_cache : a.v_cache) + (size_t)head * a.max_len * a.head_dim + dim;
          c.to_cache = true;
        }
      } else if constexpr (R == Region::OprojRes) {
        c.dst_f32 = a.out_f32 + c.n;
      } else if (R == Region::FfnDown && a.out_f32 != nullptr) {
        c.dst_f32 = a.out_f32 + c.n;  // a tensor-sliced rank's partial sum (fp32)
      } else {
        c.dst = static_cast<ACT*>(a.out_act) + c.n;
        if constexpr (R == Region::FfnUp && kSplit) c.dst_lo = static_cast<ACT*>(a.out_lo) + c.n;
      }
      return c;
    };
    // Global operands of 8 token columns (residual, or the cache position),
    // requested one group ahead of their use.
    auto ops_load = [&](const TileCtx& c, int c8, float (&o)[8]) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int mi = c8 + i;
        const int m = c.m0 + (mi < c.mrows ? mi : c.mrows - 1);
        if constexpr (R == Region::LnQkv) {
          const int b = a.T == 1 ? m : m / a.T;
          o[i] = __int_as_float(a.past_len[b] + (m - b * a.T));
        } else if constexpr (R == Region::OprojRes) {
          o[i] = a.resid_act != nullptr ? Act<ACT>::to_f(static_cast<const ACT*>(a.resid_act)[(size_t)m * N + c.n]) : 0.f;
        } else if constexpr (R == Region::FfnDown) {
          o[i] = a.resid_f32 != nullptr ? a.resid_f32[(size_t)m * N + c.n] : 0.f;
        } else {
          o[i] = 0.f;
        }
      }
    };
    // Region epilogue of 8 token columns [m0 + c8, m0 + c8 + 8) of row n.
    auto epi8 = [&](const TileCtx& c, int c8, const float (&v)[8], const float (&op)[8]) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int mi = c8 + i;  // column within the tile
        const int m = c.m0 + mi;
        const bool ok = mi < c.mrows && ds_in_bounds(m < M && c.n < N, a.status);
        float y = (v[i] + c.bias) * c.scale;
        if constexpr (R == Region::LnQkv) {
          if (ok) {
            if (!c.to_cache) {
              c.dst_f32[(size_t)m * a.H] = y;
            } else {
              const int b = a.T == 1 ? m : m / a.T;
              const int pos = __float_as_int(op[i]);
              if (pos >= 0 && pos < a.max_len) {
                if (ds_in_bounds(b < a.B && c.n < 3 * a.H, a.status))
                  c.dst[((size_t)b * a.heads * a.max_len + pos) * a.head_dim] = Act<ACT>::from_f(y);
              }
              else
                atomicOr(a.status, kFlagCacheOverflow);
            }
          }
        } else if constexpr (R == Region::FfnUp) {
          if (ok) {
            y = gelu_tanh(y);
            const ACT h = Act<ACT>::from_f(y);
            c.dst[(size_t)m * N] = h;
            if constexpr (kSplit) c.dst_lo[(size_t)m * N] = Act<ACT>::from_f(y - Act<ACT>::to_f(h));
          }
        } else {
          y += op[i];
          if (R == Region::OprojRes || c.dst_f32 != nullptr) {
            if (ok) c.dst_f32[(size_t)m * N] = y;
          } else {
            const ACT h = Act<ACT>::from_f(y);
            if (ok) c.dst[(size_t)m * N] = h;
            y = Act<ACT>::to_f(h);
          }
          if constexpr (kStats) {
            // (sum, M2) over each 16-row group of the tile (lanes 0..15, 16..31)
            if (a.stats_out != nullptr && ok) {
              float s = y;
#pragma unroll
              for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
              const float mean = s * (1.0f / 16.0f);
              float dd = (y - mean) * (y - mean);
#pragma unroll
              for (int o = 8; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
              if ((lane & 15) == 0) {
                float* so = a.stats_out + ((size_t)(c.n >> 4) * M + m) * 2;
                so[0] = s;
                so[1] = dd;
              }
            }
          }
        }
      }
    };
    // Split-K partials: [partial tile][KS * maxc slots][ntok][128] fp32, one
    // contiguous block per contributor; partial tiles are all tiles when K is
    // sliced, else only the leftover tiles (u >= U_dp).
    const size_t slot_floats = (size_t)NTOK * 128;
    const int tiles = P.tiles;
    auto partial_base = [&](int t) {
      const int pt = P.KS > 1 ? t : t - P.U_dp;
      return a.partials + (size_t)pt * P.KS * P.maxc * slot_floats;
    };
    // The idx-th contribution to tile t (slice order, then CTA order) -> its slot.
    auto slot_of = [&](int t, int idx) {
      int sl = 0;
      for (;;) {
        const int nj = ws_unit_contrib(sl * tiles + t, P, gridDim.x);
        if (idx < nj) return sl * P.maxc + idx;
        idx -= nj;
        ++sl;
      }
    };
    const uint32_t st = smem_u32(sm);  // fix-up staging slots: slot k at st + k * slot_stride
    const uint32_t slot_stride = (uint32_t)(slot_floats * 4);
    // Residual rows staged in shared memory by a fix-up: row col of the tile
    // (128 features) at ops_sm + col * kResidRowBytes.
    constexpr uint32_t kResidRowBytes = R == Region::OprojRes ? 128 * sizeof(ACT) : 128 * 4;
    auto ops_from_smem = [&](uint32_t ops_sm, int c8, float (&o)[8]) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t e = ops_sm + (uint32_t)(c8 + i) * kResidRowBytes;
        if constexpr (R == Region::OprojRes) {
          unsigned short u;
          asm volatile("ld.shared.u16 %0, [%1];" : "=h"(u) : "r"(e + (uint32_t)r * 2u) : "memory");
          o[i] = Act<ACT>::to_f(*reinterpret_cast<const ACT*>(&u));
        } else {
          o[i] = lds_f32(e + (uint32_t)r * 4u);
        }
      }
    };
    // A tile's accumulator, 8 columns from c8 (tensor memory at tb): the sum
    // of the MMA issuers' accumulators that the segment wrote (mask bit i:
    // issuer i took one of its chunks; warp-uniform, the loads are
    // warp-collective).
    static_assert(kDenseMaxIssuers == 2, "the accumulator sum below takes two issuers");
    auto acc_ld8 = [&](uint32_t tb, int c8, int mask, float (&v)[8]) {
      if (mask == 1) {
        tmem_ld8(tb + (uint32_t)c8, v);
      } else if (mask == 2) {
        tmem_ld8(tb + (uint32_t)(2 * NTOK + c8), v);
      } else {
        float w[8];
        tmem_ld8(tb + (uint32_t)c8, v);
        tmem_ld8(tb + (uint32_t)(2 * NTOK + c8), w);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] += w[i];
      }
    };
    // The issuers whose accumulators a segment of n chunks starting at the
    // CTA's chunk j0 wrote (issuer i takes the chunks j with j % 2 == i).
    auto acc_mask = [&](int j0, int n) { return nis == 1 ? 1 : (n >= 2 ? 3 : 1 << (j0 & 1)); };
    int seg_mask = 1;  // acc_mask of the segment being finished
    // Finishes the 8-column groups c0, c0 + cstep, ... of one tile, the
    // accumulator taken from tensor memory (src 0), from nk staged partial
    // slots in shared memory (src 1), from nk partials in global memory
    // (src 2) or from the partial tiles of the nk CTAs of this cluster (src 3,
    // summed in rank order); the residual from shared memory when
    // ops_sm != 0, else from global memory (group c0's operands already in
    // `pre` when given: loaded before the accumulator was ready).
    auto finish_tile = [&](const TileCtx& c, int src, uint32_t tbase, int nk, const float* pg, uint32_t ops_sm,
                           int c0, int cstep, const float* pre) {
      float opn[8];
      if (pre != nullptr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) opn[i] = pre[i];
      } else if (ops_sm == 0 && c0 < c.mrows) {
        ops_load(c, c0, opn);
      }
#pragma unroll 1
      for (int c8 = c0; c8 < c.mrows; c8 += cstep) {
        float v[8], op[8];
        if (ops_sm != 0) {
          ops_from_smem(ops_sm, c8, op);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) op[i] = opn[i];
          if (c8 + cstep < c.mrows) ops_load(c, c8 + cstep, opn);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
        if (src == 0) {
          acc_ld8(tbase, c8, seg_mask, v);
        } else if (src == 1) {
          const uint32_t e0 = st + (uint32_t)(c8 * 128 + r) * 4u;
#pragma unroll 1
          for (int k = 0; k < nk; ++k) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] += lds_f32(e0 + (uint32_t)k * slot_stride + (uint32_t)i * 512u);
          }
        } else if (src == 2) {
#pragma unroll 1
          for (int k = 0; k < nk; ++k) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (c8 + i < c.mrows) v[i] += ld_cg(pg + (size_t)k * slot_floats + (size_t)(c8 + i) * 128 + r);
          }
        } else {
          const uint32_t e0 = st + (uint32_t)(c8 * 128 + r) * 4u;
#pragma unroll 1
          for (int k = 0; k < nk; ++k) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (c8 + i < c.mrows) v[i] += ld_cluster_f32(e0 + (uint32_t)i * 512u, (uint32_t)k);
          }
        }
        epi8(c, c8, v, op);
      }
    };
    // Tiles this CTA finishes as their last contributor; done after its last
    // segment, when the ring is idle and can stage the partials (a CTA's
    // range has at most two partial segments: its first and its last unit).
    if (KSC > 1) {
      // One K slice of one tile per CTA; the cluster's slices are summed
      // through distributed shared memory.  Each CTA stores its partial tile
      // in its idle ring ([column][128 rows] fp32; every copy into the ring
      // has been consumed by the MMAs the accumulator barrier waits for), then
      // finishes the 8-column groups rank, rank + KSC, ... of the tile (the
      // two warps of a lane quarter alternating) from all the partial tiles in
      // rank order: deterministic, nothing through global memory.
      const int t = (int)(blockIdx.x / KSC), rank = (int)(blockIdx.x % KSC);
      const TileCtx c = tile_ctx(t);
      const int half = (warp - kDenseEpiWarp0) >> 2;
      const int g0 = 8 * (rank + KSC * half);  // this thread's first 8-column group to finish
      float pre[8];
      if (g0 < c.mrows) ops_load(c, g0, pre);  // residual / positions: before the accumulator is ready
      bool dead = !mbar_wait(accf_bar(0), 0, a.status);
      dead = __any_sync(0xffffffffu, dead);  // (the loads below are warp-collective either way)
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(32 * qd) << 16);
#pragma unroll 1
      for (int c8 = cbeg; c8 < c.mrows; c8 += 16) {
        float v[8];
        acc_ld8(tbase, c8, acc_mask(0, cl_len), v);  // (one whole K slice per CTA)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c8 + i < c.mrows) sts_f32(st + (uint32_t)((c8 + i) * 128 + r) * 4u, v[i]);
      }
      tc_fence_before();
      dense_cluster_sync();  // every slice's partial tile is in place
      finish_tile(c, 3, 0u, KSC, nullptr, 0u, g0, 16 * KSC, g0 < c.mrows ? pre : nullptr);
      dense_cluster_sync();  // the other CTAs have read this CTA's partial tile
    } else {
    int pend_t0 = 0, pend_c0 = 0, pend_t1 = 0, pend_c1 = 0, npend = 0;
    const int nstage_slots = (int)(((size_t)S * SB) / (slot_floats * 4));  // staging slots in the ring
    int seg = 0;
    bool dead = false;
    int j0 = 0;  // the CTA's chunks before this segment
    for_segments([&](int u, int kc0, int kc1, int j_slot) {
      seg_mask = acc_mask(j0, kc1 - kc0);
      j0 += kc1 - kc0;
      const int buf = seg & 1;
      const int sl = u / tiles, t = u - sl * tiles;   // K slice, output tile
      const int target = ws_tile_target(t, P, gridDim.x);  // contributions that complete the tile
      const TileCtx c = tile_ctx(t);
      // a tile finished here: its first operands before the accumulator is ready
      float pre[8];
      const bool pre_ok = target == 1 && cbeg < c.mrows;
      if (pre_ok) ops_load(c, cbeg, pre);
      if (!dead) dead = !mbar_wait(accf_bar(buf), (seg >> 1) & 1, a.status);
      dead = __any_sync(0xffffffffu, dead);  // tcgen05.ld below is warp-collective
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(buf * NTOK);
      if (target == 1) {
        finish_tile(c, 0, tbase, 0, nullptr, 0u, cbeg, 16, pre_ok ? pre : nullptr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(buf));
      } else {
        // publish this CTA's partial tile and count; the last contributor
        // finishes the tile (only leftover tiles, u >= U_dp, have several)
        float* pb = partial_base(t) + (size_t)(sl * P.maxc + j_slot) * slot_floats + r;
#pragma unroll 1
        for (int c8 = cbeg; c8 < c.mrows; c8 += 16) {
          float v[8];
          acc_ld8(tbase, c8, seg_mask, v);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (c8 + i < c.mrows) pb[(size_t)(c8 + i) * 128] = v[i];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(buf));
        // every epilogue thread's partial stores, then one release-acquire arrival
        __threadfence();
        named_bar_sync(kDenseBarEpi, kDenseEpiThreads);
        if (et == 0) *last_flag = (atomic_add_acq_rel_gpu(&a.counters[t], 1) == target - 1);
        named_bar_sync(kDenseBarEpi, kDenseEpiThreads);
        const bool last = *last_flag != 0;
        named_bar_sync(kDenseBarEpi, kDenseEpiThreads);  // last_flag is read before the next segment writes it
        if (last) {
          if (npend == 0) {
            pend_t0 = t;
            pend_c0 = target;
          } else {
            pend_t1 = t;
            pend_c1 = target;
          }
          ++npend;
        }
      }
      ++seg;
    });
    // Deferred fix-ups: the ring is idle now (every copy into it has been
    // consumed by the MMAs).  The contributors' partials are bulk-copied into
    // the ring (one round trip for up to nstage_slots of them) and summed in
    // slot order (deterministic), then the epilogue runs.
    uint32_t fph = 0;
#pragma unroll 1
    for (int pi = 0; pi < npend && pi < 2; ++pi) {
      const int t = pi == 0 ? pend_t0 : pend_t1;
      const int contrib = pi == 0 ? pend_c0 : pend_c1;
      const TileCtx c = tile_ctx(t);
      const float* pbase = partial_base(t);
      const uint32_t slot_bytes = (uint32_t)(c.mrows * 128 * 4);
      if (nstage_slots < 2) {
        // a slot larger than half the ring: sum from global memory (the plans
        // give contiguous slots: one K slice, or one CTA per slice)
        finish_tile(c, 2, 0u, contrib, pbase, 0u, cbeg, 16, nullptr);
      } else {
        // Rounds of up to nstage_slots partials (one round in the common
        // case); with more, slot 0 carries the running sum between rounds.
        for (int js = 0; js < contrib;) {
          const int dst0 = js == 0 ? 0 : 1;
          const int nr = min(contrib - js, nstage_slots - dst0);
          // the last round also stages the tile's residual rows behind the
          // partials when they fit (the epilogue then reads no global memory)
          uint32_t ops_sm = 0;
          if constexpr (R == Region::OprojRes || R == Region::FfnDown) {
            const uint32_t off = (uint32_t)(dst0 + nr) * slot_stride;
            const bool has_resid = R == Region::OprojRes ? a.resid_act != nullptr : a.resid_f32 != nullptr;
            if (has_resid && js + nr == contrib && (size_t)off + (size_t)c.mrows * kResidRowBytes <= (size_t)S * SB)
              ops_sm = st + off;
          }
          if (et < 32) {  // the first epilogue warp issues the copies
            // this thread's acquire (the arrival counter) orders the other
            // contributors' partial stores; the proxy fence orders them before
            // the async-proxy (bulk copy) reads
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint64_t pol = l2_evict_first_policy();
            if (et == 0) {
              mbar_arrive_expect_tx(fix_bar, (uint32_t)nr * slot_bytes + (ops_sm ? (uint32_t)c.mrows * kResidRowBytes : 0u));
              for (int k = 0; k < nr; ++k)
                bulk_g2s(st + (uint32_t)(dst0 + k) * slot_stride, pbase + (size_t)slot_of(t, js + k) * slot_floats,
                         slot_bytes, fix_bar, pol);
            }
            __syncwarp();
            if (ops_sm != 0) {
              const int n0 = c.n - r;
              for (int col = et; col < c.mrows; col += 32) {
                const void* src_row;
                if constexpr (R == Region::OprojRes)
                  src_row = static_cast<const ACT*>(a.resid_act) + (size_t)(c.m0 + col) * N + n0;
                else
                  src_row = a.resid_f32 + (size_t)(c.m0 + col) * N + n0;
                bulk_g2s(ops_sm + (uint32_t)col * kResidRowBytes, src_row, kResidRowBytes, fix_bar, pol);
              }
            }
          }
          if (!dead) dead = !mbar_wait(fix_bar, fph, a.status);
          fph ^= 1;
          js += nr;
          const int nk = dst0 + nr;  // slots holding data: 0 .. nk-1
          if (js < contrib) {
            // more rounds follow: fold this round into slot 0 (this thread's row)
#pragma unroll 1
            for (int c8 = cbeg; c8 < c.mrows; c8 += 16) {  // this warp's 8-column groups
              for (int col = c8; col < c8 + 8 && col < c.mrows; ++col) {
                const uint32_t e = st + (uint32_t)(col * 128 + r) * 4u;
                float acc = lds_f32(e);
                for (int k = 1; k < nk; ++k) acc += lds_f32(e + (uint32_t)k * slot_stride);
                sts_f32(e, acc);
              }
            }
            named_bar_sync(kDenseBarEpi, kDenseEpiThreads);  // staging slots free for the next round
          } else {
            finish_tile(c, 1, 0u, nk, nullptr, ops_sm, cbeg, 16, nullptr);
          }
        }
      }
      if (et == 0) a.counters[t] = 0;
      named_bar_sync(kDenseBarEpi, kDenseEpiThreads);  // the staging slots are read before the next fix-up
    }
    }  // KSC == 1
    if constexpr (R == Region::FfnDown) {
      if (a.seq_len_inc != nullptr && blockIdx.x == 0 && warp == kDenseEpiWarp0)
        for (int b = lane; b < a.B; b += 32) a.seq_len_inc[b] += 1;
    }
    // every tensor-memory read of this warp is done: let the MMA warp free it
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(done_bar);
  }
  // Warp 1 frees the tensor memory once the eight epilogue warps are done with
  // it (an mbarrier, not a CTA barrier: the roles reach the end on different
  // paths).
  if (warp == kDenseMmaWarp) {
    if (lane == 0) mbar_wait(done_bar, 0, a.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

}  // namespace ds
