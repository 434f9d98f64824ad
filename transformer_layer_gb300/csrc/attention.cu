// Region 2: decode attention over the KV cache with scale, causal mask and
// softmax fused (split-KV, combined at the reduction boundary).
//
// Pages cited:
//   [P1] "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核
//        与 MoQ 量化支持", §3.2 region 2: transform and attention merged, the
//        head-split layout read through index arithmetic ("implicit matrix
//        transformation") instead of being materialised.
//   [P3] "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、PR-MoE 优化与
//        init_inference 全解析", table "推理配置参数详解": triangular_masking,
//        the causal mask.
//
// What it computes, per sequence b, new token t and head h:
//   s_j = q . k_j / sqrt(d) for j <= past_len[b] + t;  p = softmax(s);  o = sum_j p_j v_j.
//
// GB300 design (not the pages'): at batch 1 a layer has only nh (20-40) heads,
// far fewer than 152 SMs, so each (b, h) is split over `nsplit` CTAs along the
// keys.  Each CTA computes its keys' scores (16-byte loads, a key's d values
// spread over d/8 lanes and reduced with warp shuffles), the local max and sum
// (log2 domain) and the unnormalised p.V; the last CTA of each (b, h) to
// arrive (atomic counter, no waiting) merges the splits with the usual
// log-sum-exp rescaling.  Before griddepcontrol.wait a CTA asks the TMA unit to
// prefetch into L2 the cache rows that the previous kernel does not write.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kAttnThreads = 128;

template <typename ACT, int D>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
  constexpr int LPK = D / 8;               // lanes per key (16 B each)
  constexpr int KPI = kAttnThreads / LPK;  // keys per CTA pass
  extern __shared__ __align__(16) float sm[];
  float* sc = sm;                         // [chunk_cap] scores, then probabilities
  float* ored = sc + a.chunk_cap;         // [KPI][D]
  float* red = ored + KPI * D;            // [32] block-reduction / merge scratch
  int* flag = reinterpret_cast<int*>(red + 32);

  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kq = tid % LPK, kr = tid / LPK;

  const int past = a.past_len[b];
  int S_all = past + a.T;
  if (S_all > a.max_len) S_all = a.max_len;
  if (S_all < 1) S_all = 1;
  const int chunk = (S_all + a.nsplit - 1) / a.nsplit;
  const int lo = sp * chunk;
  const int hi = min(S_all, lo + chunk);
  const size_t head_row0 = ((size_t)b * a.heads + h) * a.max_len;
  const ACT* Kc = static_cast<const ACT*>(a.k_cache) + head_row0 * D;
  const ACT* Vc = static_cast<const ACT*>(a.v_cache) + head_row0 * D;

  if (tid == 0) {
    const int pe = min(hi, past);
    if (pe > lo) {
      prefetch_l2_bulk(Kc + (size_t)lo * D, (uint32_t)((pe - lo) * D * sizeof(ACT)));
      prefetch_l2_bulk(Vc + (size_t)lo * D, (uint32_t)((pe - lo) * D * sizeof(ACT)));
    }
  }
  pdl_wait();
  pdl_launch_dependents();

  for (int t = 0; t < a.T; ++t) {
    const int St = min(past + t + 1, S_all);
    const int n_keys = max(0, min(hi, St) - lo);
    float* dst = a.part + (((size_t)(b * a.T + t) * a.heads + h) * a.nsplit + sp) * (D + 2);
    if (n_keys == 0) {
      if (tid < D) dst[tid] = 0.f;
      if (tid == 0) {
        dst[D] = -INFINITY;
        dst[D + 1] = 0.f;
      }
      continue;
    }
    float qv[8];
    {
      const float* qp = a.q + (size_t)(b * a.T + t) * a.H + h * D + kq * 8;
      const float4 q0 = *reinterpret_cast<const float4*>(qp);
      const float4 q1 = *reinterpret_cast<const float4*>(qp + 4);
      qv[0] = q0.x; qv[1] = q0.y; qv[2] = q0.z; qv[3] = q0.w;
      qv[4] = q1.x; qv[5] = q1.y; qv[6] = q1.z; qv[7] = q1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] *= a.scale_log2;
    }
    // scores (log2 domain)
    float mloc = -INFINITY;
    const int passes = (n_keys + KPI - 1) / KPI;
#pragma unroll 8
    for (int ps = 0; ps < passes; ++ps) {
      const int j = ps * KPI + kr;
      float s = 0.f;
      if (j < n_keys) {
        const uint4 u = *reinterpret_cast<const uint4*>(Kc + (size_t)(lo + j) * D + kq * 8);
        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = Act<ACT>::unpack2(uw[i]);
          s += f.x * qv[2 * i] + f.y * qv[2 * i + 1];
        }
      }
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (j < n_keys) {
        if (kq == 0) sc[j] = s;
        mloc = fmaxf(mloc, s);
      }
    }
    mloc = warp_max(mloc);
    if (lane == 0) red[warp] = mloc;
    __syncthreads();
    const float m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    float lsum = 0.f;
    for (int j = tid; j < n_keys; j += kAttnThreads) {
      const float p = exp2f(sc[j] - m);
      sc[j] = p;
      lsum += p;
    }
    lsum = warp_sum(lsum);
    __syncthreads();  // red reads done, probabilities visible
    if (lane == 0) red[4 + warp] = lsum;
    // o = sum_j p_j v_j
    float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int ps = 0; ps < passes; ++ps) {
      const int j = ps * KPI + kr;
      if (j < n_keys) {
        const float p = sc[j];
        const uint4 u = *reinterpret_cast<const uint4*>(Vc + (size_t)(lo + j) * D + kq * 8);
        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = Act<ACT>::unpack2(uw[i]);
          o8[2 * i] += p * f.x;
          o8[2 * i + 1] += p * f.y;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ored[kr * D + kq * 8 + i] = o8[i];
    __syncthreads();
    if (tid < D) {
      float o = 0.f;
#pragma unroll
      for (int r = 0; r < KPI; ++r) o += ored[r * D + tid];
      dst[tid] = o;
    }
    if (tid == 0) {
      dst[D] = m;
      dst[D + 1] = red[4] + red[5] + red[6] + red[7];
    }
    __syncthreads();  // sc / ored / red reused by the next token
  }

  // Merge the splits of (b, h): the last CTA to arrive does it.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[b * a.heads + h], 1);
    *flag = (prev == a.nsplit - 1);
  }
  __syncthreads();
  if (*flag) {
    __threadfence();
    float* wsm = red;  // [nsplit] merge weights (nsplit <= 32)
    for (int t = 0; t < a.T; ++t) {
      const float* base = a.part + ((size_t)(b * a.T + t) * a.heads + h) * a.nsplit * (D + 2);
      if (warp == 0) {
        const float ms = lane < a.nsplit ? ld_cg(base + lane * (D + 2) + D) : -INFINITY;
        const float ls = lane < a.nsplit ? ld_cg(base + lane * (D + 2) + D + 1) : 0.f;
        const float mx = warp_max(ms);
        const float w = lane < a.nsplit ? exp2f(ms - mx) : 0.f;
        const float lsum = warp_sum(w * ls);
        if (lane < a.nsplit) wsm[lane] = w / lsum;
      }
      __syncthreads();
      if (tid < D) {
        float O = 0.f;
#pragma unroll 8
        for (int s2 = 0; s2 < a.nsplit; ++s2) O += wsm[s2] * ld_cg(base + s2 * (D + 2) + tid);
        a.out[(size_t)(b * a.T + t) * a.H + h * D + tid] = O;
      }
      __syncthreads();
    }
    if (tid == 0) a.counters[b * a.heads + h] = 0;
  }
}

int attn_nsplit(int B, int heads, int max_len, int num_sms) {
  const int bh = B * heads;
  int ns = (2 * num_sms + bh - 1) / bh;
  if (ns < 1) ns = 1;
  if (ns > 32) ns = 32;
  const int cap = (max_len + 15) / 16;  // at least ~16 keys per split
  if (ns > cap) ns = cap < 1 ? 1 : cap;
  return ns;
}

size_t attn_smem_bytes(int head_dim, int chunk_cap) {
  const int kpi = kAttnThreads / (head_dim / 8);
  return sizeof(float) * ((size_t)chunk_cap + (size_t)kpi * head_dim + 32) + 16;
}

cudaError_t launch_attention(ActKind ak, const AttnArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.heads, a.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = a.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (ak == ActKind::F16) {
    if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__half, 64>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__half, 128>, a);
  } else {
    if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__nv_bfloat16, 64>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__nv_bfloat16, 128>, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_attention_kernels(int max_smem) {
  cudaError_t e = cudaSuccess;
#define DS_PREP_ATTN(T, D)                                                                   \
  if (e == cudaSuccess)                                                                      \
    e = cudaFuncSetAttribute(attn_decode_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             max_smem)
  DS_PREP_ATTN(__half, 64);
  DS_PREP_ATTN(__half, 128);
  DS_PREP_ATTN(__nv_bfloat16, 64);
  DS_PREP_ATTN(__nv_bfloat16, 128);
#undef DS_PREP_ATTN
  return e;
}

}  // namespace ds
