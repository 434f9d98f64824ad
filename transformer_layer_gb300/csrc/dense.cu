// Host side of the tensor-core tile path (plan, launch dispatch) and the row
// normalisation kernel that feeds it.
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持", §3.2 regions 1 and 3: the LayerNorm ahead of
// the QKV and FFN-up GEMMs.  On the tile path the normalisation runs as its
// own small kernel (one pass over the M x K activations) that writes the
// tensor-core operand; the statistics still come from the previous GEMM's
// reduction boundary (per-16-feature (sum, M2) partials).
#include <cuda.h>

#include "common.cuh"
#include "dense_impl.cuh"
#include "dense_plan.h"
#include "internal.h"
#include "work_split.h"

namespace ds {

cudaError_t launch_dense_f16(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                             cudaStream_t st, bool pdl);
cudaError_t launch_dense_bf16(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                              cudaStream_t st, bool pdl);
cudaError_t launch_dense_i8(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                            cudaStream_t st, bool pdl);
cudaError_t prepare_dense_f16(int max_smem);
cudaError_t prepare_dense_bf16(int max_smem);
cudaError_t prepare_dense_i8(int max_smem);
int dense_cluster_capacity(int size, int max_smem);


bool dense_make_plan(ActKind ak, int N, int K, int M, int num_sms, int max_smem, DensePlan* plan, bool i8) {
  return dense_make_plan_t(ak, N, K, M, num_sms, max_smem, plan, i8,
                           [&](int size) { return dense_cluster_capacity(size, max_smem); });
}

cudaError_t launch_dense(Region r, ActKind ak, const DenseArgs& a, const void* xmap_hi, const void* xmap_lo,
                         cudaStream_t st, bool pdl) {
  const CUtensorMap* xh = static_cast<const CUtensorMap*>(xmap_hi);
  const CUtensorMap* xl = static_cast<const CUtensorMap*>(xmap_lo != nullptr ? xmap_lo : xmap_hi);
  if (a.plan.i8) return ak == ActKind::F16 ? launch_dense_i8(r, a, xh, xl, st, pdl) : cudaErrorInvalidValue;
  if (ak == ActKind::F16) return launch_dense_f16(r, a, xh, xl, st, pdl);
  return launch_dense_bf16(r, a, xh, xl, st, pdl);
}

cudaError_t prepare_dense_kernels(int max_smem) {
  cudaError_t e = prepare_dense_f16(max_smem);
  if (e == cudaSuccess) e = prepare_dense_bf16(max_smem);
  if (e == cudaSuccess) e = prepare_dense_i8(max_smem);
  return e;
}

// ---------------------------------------------------------------- row normalisation
constexpr int kPrepThreads = 256;
constexpr int kPrepCols = kPrepThreads * 8;  // columns per block

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) s += red[w];
  return s;
}

// Row m = blockIdx.y, columns [blockIdx.x * 2048, +2048): LN(x) with gamma,
// beta, written as the operand hi (and lo for bf16).  Mean and variance come
// from the (sum, M2) partials of 16-feature groups when given (pooled with
// Chan's formula), else from two passes over the row.
template <typename ACT, bool kF32>
__global__ void __launch_bounds__(kPrepThreads) ln_prep_kernel(const LnPrepArgs a) {
  constexpr bool kSplit = std::is_same<ACT, __nv_bfloat16>::value;
  __shared__ float red[kPrepThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.y, K = a.K, M = a.M;
  const int tid = threadIdx.x;
  auto load8 = [&](int k, float (&v)[8]) {
    if constexpr (kF32) {
      const float* p = a.x_f32 + (size_t)m * K + k;
      const float4 p0 = *reinterpret_cast<const float4*>(p), p1 = *reinterpret_cast<const float4*>(p + 4);
      v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
      v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
    } else {
      const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.x_act) + (size_t)m * K + k);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = Act<ACT>::unpack2(w[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
    }
  };
  float mean, m2;
  if (a.stats_in != nullptr) {
    const int tin = K / 16;
    const float2* st2 = reinterpret_cast<const float2*>(a.stats_in);
    float s = 0.f;
    for (int i = tid; i < tin; i += kPrepThreads) s += st2[(size_t)i * M + m].x;
    mean = block_sum(s, red) / (float)K;
    float q = 0.f;
    for (int i = tid; i < tin; i += kPrepThreads) {
      const float2 p = st2[(size_t)i * M + m];
      const float d = p.x * (1.0f / 16.0f) - mean;
      q += p.y + 16.0f * d * d;
    }
    m2 = block_sum(q, red);
  } else {
    float s = 0.f;
    for (int k = tid * 8; k < K; k += kPrepCols) {
      float v[8];
      load8(k, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[i];
    }
    mean = block_sum(s, red) / (float)K;
    float q = 0.f;
    for (int k = tid * 8; k < K; k += kPrepCols) {
      float v[8];
      load8(k, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) q += (v[i] - mean) * (v[i] - mean);
    }
    m2 = block_sum(q, red);
  }
  const float rstd = 1.0f / sqrtf(m2 / (float)K + a.eps);
  const int k = blockIdx.x * kPrepCols + tid * 8;
  if (k >= K) return;
  float v[8];
  load8(k, v);
  const uint4 gu = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_g) + k);
  const uint4 bu = *reinterpret_cast<const uint4*>(static_cast<const ACT*>(a.ln_b) + k);
  const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w}, bw[4] = {bu.x, bu.y, bu.z, bu.w};
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 g = Act<ACT>::unpack2(gw[i]), b = Act<ACT>::unpack2(bw[i]);
    const float y0 = (v[2 * i] - mean) * rstd * g.x + b.x;
    const float y1 = (v[2 * i + 1] - mean) * rstd * g.y + b.y;
    hw[i] = Act<ACT>::pack2(y0, y1);
    if constexpr (kSplit) {
      const float2 h = Act<ACT>::unpack2(hw[i]);
      lw[i] = Act<ACT>::pack2(y0 - h.x, y1 - h.y);
    }
  }
  *reinterpret_cast<uint4*>(static_cast<ACT*>(a.out_hi) + (size_t)m * K + k) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  if constexpr (kSplit)
    *reinterpret_cast<uint4*>(static_cast<ACT*>(a.out_lo) + (size_t)m * K + k) =
        make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

cudaError_t launch_ln_prep(ActKind ak, const LnPrepArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.K + kPrepCols - 1) / kPrepCols, a.M);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const bool f32 = a.x_f32 != nullptr;
  if (ak == ActKind::F16)
    return f32 ? cudaLaunchKernelEx(&cfg, ln_prep_kernel<__half, true>, a)
               : cudaLaunchKernelEx(&cfg, ln_prep_kernel<__half, false>, a);
  return f32 ? cudaLaunchKernelEx(&cfg, ln_prep_kernel<__nv_bfloat16, true>, a)
             : cudaLaunchKernelEx(&cfg, ln_prep_kernel<__nv_bfloat16, false>, a);
}

}  // namespace ds
