// Region 2 for prompt chunks (T new tokens per sequence, T >= 16): causal
// attention of every new token over the cache and the new tokens before it,
// as tiled tensor-core flash attention.
//
// Pages cited:
//   [P1] "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核
//        与 MoQ 量化支持", §3.2 region 2: the attention GEMMs merged with the
//        transform, the head-split layout read by index arithmetic.
//   [P3] "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、PR-MoE 优化与
//        init_inference 全解析", table "推理配置参数详解": triangular_masking.
//
// What it computes, per sequence b, new token t (query position past[b] + t)
// and head h:  o = softmax_j(q . k_j / sqrt(d)) v_j over keys j <= past[b] + t.
//
// Design: one CTA (4 warps) takes 64 queries of one (b, h); each warp owns 16
// query rows.  Key / value blocks of 64 rows are copied from the cache into
// shared memory with cp.async (double-buffered, 16-byte chunks XOR-swizzled
// so that ldmatrix reads are conflict-free).  S = Q K^T and O += P V run as
// mma.sync m16n8k16 with fp32 accumulation; the softmax is online (running
// max and sum per row, log2 domain), the S accumulators turning into the P
// operand in registers.  bf16 splits Q and P into hi + lo operands (two MMAs
// each), so that the rounding of the operands stays near fp32's; fp16 uses
// single operands (11 significant bits).  Blocks past the causal frontier are
// skipped; the diagonal blocks are masked.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kFaThreads = 128;
constexpr int kFaBQ = 64;  // queries per CTA
constexpr int kFaBK = 64;  // keys per block

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Byte offset of 16-byte chunk c of row r in a [rows][D] 16-bit tile whose
// rows are D * 2 bytes: chunk index XOR (r mod 8).
template <int D>
__device__ __forceinline__ uint32_t fa_off(int r, int c) {
  return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

template <typename T> struct FaMma;
template <> struct FaMma<__half> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    mma_f16(d, a[0], a[1], a[2], a[3], b0, b1);
  }
};
template <> struct FaMma<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    mma_bf16(d, a[0], a[1], a[2], a[3], b0, b1);
  }
};

template <typename ACT, int D>
__global__ void __launch_bounds__(kFaThreads) attn_prefill_kernel(const AttnArgs a) {
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;
  constexpr int NCH = D / 8;        // 16-byte chunks per row
  constexpr int KSTEPS = D / 16;    // k steps of S = Q K^T
  constexpr int NT = D / 8;         // n tiles of O (8 dims each)
  constexpr size_t TILE = (size_t)kFaBK * D * 2;
  extern __shared__ __align__(128) unsigned char fsm[];
  // [Q hi][Q lo (bf16)][K 0][V 0][K 1][V 1]
  unsigned char* q_hi = fsm;
  unsigned char* q_lo = fsm + TILE;
  unsigned char* kv = fsm + (kSplit ? 2 : 1) * TILE;
  const uint32_t s_qhi = smem_u32(q_hi), s_qlo = smem_u32(q_lo), s_kv = smem_u32(kv);

  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, cq = lane & 3;
  const int T = a.T;
  pdl_wait();
  pdl_launch_dependents();
  const int past = a.past_len[b];
  const int q0 = qb * kFaBQ;                      // first query (new-token index) of this CTA
  const int qn = min(kFaBQ, T - q0);              // queries in this CTA
  int kend = past + q0 + qn;                      // keys the last query sees
  if (kend > a.max_len) kend = a.max_len;
  const int nkb = (kend + kFaBK - 1) / kFaBK;
  const size_t head_row0 = ((size_t)b * a.heads + h) * a.max_len;
  const ACT* Kc = static_cast<const ACT*>(a.k_cache) + head_row0 * D;
  const ACT* Vc = static_cast<const ACT*>(a.v_cache) + head_row0 * D;

  // K / V block kb into buffer buf: 64 rows x NCH chunks each, rows past the
  // end clamped to the last key (masked below).
  auto load_kv = [&](int kb, int buf) {
    const uint32_t dk = s_kv + (uint32_t)(2 * buf) * (uint32_t)TILE, dv = dk + (uint32_t)TILE;
    for (int i = tid; i < kFaBK * NCH; i += kFaThreads) {
      const int r = i / NCH, c = i - (i / NCH) * NCH;
      int key = kb * kFaBK + r;
      if (key >= kend) key = kend - 1;
      cp_async16(dk + fa_off<D>(r, c), Kc + (size_t)key * D + c * 8);
      cp_async16(dv + fa_off<D>(r, c), Vc + (size_t)key * D + c * 8);
    }
  };
  if (nkb > 0) load_kv(0, 0);
  cp_async_commit();

  // Q block: fp32 q scaled by log2(e)/sqrt(d), as operand hi (and lo).
  for (int i = tid; i < kFaBQ * NCH; i += kFaThreads) {
    const int r = i / NCH, c = i - (i / NCH) * NCH;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (r < qn) {
      const float* qp = a.q + (size_t)(b * T + q0 + r) * a.H + h * D + c * 8;
      const float4 x0 = *reinterpret_cast<const float4*>(qp), x1 = *reinterpret_cast<const float4*>(qp + 4);
      v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w; v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    }
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float f0 = v[2 * j] * a.scale_log2, f1 = v[2 * j + 1] * a.scale_log2;
      hw[j] = Act<ACT>::pack2(f0, f1);
      if constexpr (kSplit) {
        const float2 hh = Act<ACT>::unpack2(hw[j]);
        lw[j] = Act<ACT>::pack2(f0 - hh.x, f1 - hh.y);
      }
    }
    *reinterpret_cast<uint4*>(q_hi + fa_off<D>(r, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if constexpr (kSplit) *reinterpret_cast<uint4*>(q_lo + fa_off<D>(r, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  __syncthreads();
  // This warp's Q fragments (A operand, rows 16 warp .. +15), kept in registers.
  uint32_t qa[KSTEPS][4], ql[KSTEPS][4];
  {
    const int r = warp * 16 + (lane & 15);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      const int c = 2 * ks + (lane >> 4);
      ldsm_x4(s_qhi + fa_off<D>(r, c), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
      if constexpr (kSplit) ldsm_x4(s_qlo + fa_off<D>(r, c), ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3]);
    }
  }
  (void)ql;

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  // query positions of this thread's two rows (g and g + 8 of the warp's 16)
  const int tq0 = q0 + warp * 16 + g, tq1 = tq0 + 8;
  const int lim0 = past + tq0, lim1 = past + tq1;  // last key each row sees

  for (int kb = 0; kb < nkb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nkb) load_kv(kb + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t sk = s_kv + (uint32_t)(2 * buf) * (uint32_t)TILE, sv = sk + (uint32_t)TILE;
    // S = Q K^T for this warp's 16 rows x 64 keys (8 n-tiles of 8 keys)
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // pairs of key n-tiles
        uint32_t b0, b1, b2, b3;
        const int kr = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = 2 * ks + ((lane >> 3) & 1);
        ldsm_x4(sk + fa_off<D>(kr, c), b0, b1, b2, b3);
        FaMma<ACT>::run(s[2 * np], qa[ks], b0, b1);
        FaMma<ACT>::run(s[2 * np + 1], qa[ks], b2, b3);
        if constexpr (kSplit) {
          FaMma<ACT>::run(s[2 * np], ql[ks], b0, b1);
          FaMma<ACT>::run(s[2 * np + 1], ql[ks], b2, b3);
        }
      }
    }
    // causal mask, running max
    float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int j = kb * kFaBK + nt * 8 + 2 * cq;
      if (j > lim0 || j >= kend) s[nt][0] = -INFINITY;
      if (j + 1 > lim0 || j + 1 >= kend) s[nt][1] = -INFINITY;
      if (j > lim1 || j >= kend) s[nt][2] = -INFINITY;
      if (j + 1 > lim1 || j + 1 >= kend) s[nt][3] = -INFINITY;
      mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
    }
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      alpha[i] = (mx[i] == -INFINITY) ? 1.f : exp2f(mrow[i] - mx[i]);
      mrow[i] = mx[i];
      lrow[i] *= alpha[i];
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // P = exp2(S - m), row sums, P as the A operand of O += P V
    uint32_t ph[4][4], pl[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = (s[nt][0] == -INFINITY) ? 0.f : exp2f(s[nt][0] - mrow[0]);
      const float p1 = (s[nt][1] == -INFINITY) ? 0.f : exp2f(s[nt][1] - mrow[0]);
      const float p2 = (s[nt][2] == -INFINITY) ? 0.f : exp2f(s[nt][2] - mrow[1]);
      const float p3 = (s[nt][3] == -INFINITY) ? 0.f : exp2f(s[nt][3] - mrow[1]);
      lrow[0] += p0 + p1;
      lrow[1] += p2 + p3;
      const int kk = nt >> 1, hf = nt & 1;  // k step of 16 keys, half
      const uint32_t u01 = Act<ACT>::pack2(p0, p1), u23 = Act<ACT>::pack2(p2, p3);
      ph[kk][hf * 2 + 0] = u01;
      ph[kk][hf * 2 + 1] = u23;
      if constexpr (kSplit) {
        const float2 h01 = Act<ACT>::unpack2(u01), h23 = Act<ACT>::unpack2(u23);
        pl[kk][hf * 2 + 0] = Act<ACT>::pack2(p0 - h01.x, p1 - h01.y);
        pl[kk][hf * 2 + 1] = Act<ACT>::pack2(p2 - h23.x, p3 - h23.y);
      }
    }
    (void)pl;
    // O += P V: k steps over 16 keys, n tiles over 8 dims; V read transposed
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t pa[4] = {ph[kk][0], ph[kk][1], ph[kk][2], ph[kk][3]};
      uint32_t pb[4];
      if constexpr (kSplit) {
        pb[0] = pl[kk][0]; pb[1] = pl[kk][1]; pb[2] = pl[kk][2]; pb[3] = pl[kk][3];
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {  // pairs of dim n-tiles
        uint32_t b0, b1, b2, b3;
        const int vr = kk * 16 + (lane & 15);
        const int c = 2 * np + (lane >> 4);
        ldsm_x4_t(sv + fa_off<D>(vr, c), b0, b1, b2, b3);
        FaMma<ACT>::run(o[2 * np], pa, b0, b1);
        FaMma<ACT>::run(o[2 * np + 1], pa, b2, b3);
        if constexpr (kSplit) {
          FaMma<ACT>::run(o[2 * np], pb, b0, b1);
          FaMma<ACT>::run(o[2 * np + 1], pb, b2, b3);
        }
      }
    }
    __syncthreads();  // this buffer is overwritten by the load two blocks on
  }
  cp_async_wait<0>();
  // row sums over the quad, normalise, store
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 1);
    lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 2);
  }
  const float inv0 = lrow[0] > 0.f ? 1.f / lrow[0] : 0.f, inv1 = lrow[1] > 0.f ? 1.f / lrow[1] : 0.f;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int t = hrow ? tq1 : tq0;
      if (t >= T) continue;
      const float inv = hrow ? inv1 : inv0;
      const float v0 = o[n][2 * hrow] * inv, v1 = o[n][2 * hrow + 1] * inv;
      const size_t oi = (size_t)(b * T + t) * a.H + h * D + n * 8 + 2 * cq;
      if (a.out_hi != nullptr) {
        const uint32_t hv = Act<ACT>::pack2(v0, v1);
        *reinterpret_cast<uint32_t*>(static_cast<ACT*>(a.out_hi) + oi) = hv;
        if (a.out_lo != nullptr) {
          const float2 hh = Act<ACT>::unpack2(hv);
          *reinterpret_cast<uint32_t*>(static_cast<ACT*>(a.out_lo) + oi) = Act<ACT>::pack2(v0 - hh.x, v1 - hh.y);
        }
      } else {
        *reinterpret_cast<float2*>(a.out + oi) = make_float2(v0, v1);
      }
    }
  }
}

size_t attn_prefill_smem_bytes(ActKind ak, int head_dim) {
  const size_t tile = (size_t)kFaBK * head_dim * 2;
  return (ak == ActKind::BF16 ? 2 : 1) * tile + 4 * tile;
}

cudaError_t launch_attention_prefill(ActKind ak, const AttnArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.T + kFaBQ - 1) / kFaBQ, a.heads, a.B);
  cfg.blockDim = dim3(kFaThreads);
  cfg.dynamicSmemBytes = attn_prefill_smem_bytes(ak, a.head_dim);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (ak == ActKind::F16) {
    if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<__half, 64>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<__half, 128>, a);
  } else {
    if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<__nv_bfloat16, 64>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<__nv_bfloat16, 128>, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_attention_prefill_kernels(int max_smem) {
  cudaError_t e = cudaSuccess;
#define DS_PREP_FA(T, D)                                                                                \
  if (e == cudaSuccess)                                                                                 \
  e = cudaFuncSetAttribute(attn_prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem)
  DS_PREP_FA(__half, 64);
  DS_PREP_FA(__half, 128);
  DS_PREP_FA(__nv_bfloat16, 64);
  DS_PREP_FA(__nv_bfloat16, 128);
#undef DS_PREP_FA
  return e;
}

}  // namespace ds
