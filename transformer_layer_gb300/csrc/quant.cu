// MoQ-style int8 weight quantisation (load-time kernel).
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持", §5.2: int8 inference with the quantisation
// grouping passed as quantization_setting.  Rule implemented (the page fixes no
// rounding; this is the reading the library documents): per group of 32, 64
// or 128 consecutive weights along K, s = fp16_rne(float32(max|w|) / 127) and
// q = clamp(rne(w / s), -127, 127) with IEEE float32 division; s = 0 and q = 0
// for an all-zero group.
#include "common.cuh"
#include "internal.h"

namespace ds {

// One warp per group of G = 32 PER weights; lane i owns weights PER i ..
// PER i + PER - 1.
template <int PER>
__global__ void __launch_bounds__(256) quantize_int8_kernel(const __half* __restrict__ w, int n,
                                                            int k, int8_t* __restrict__ codes,
                                                            __half* __restrict__ scales) {
  constexpr int G = 32 * PER;
  const int lane = threadIdx.x & 31;
  const long long gpr = k / G;
  const long long total = (long long)n * gpr;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; gw < total;
       gw += nwarps) {
    const long long row = gw / gpr, grp = gw - (gw / gpr) * gpr;
    const size_t off = (size_t)row * k + (size_t)grp * G + (size_t)PER * lane;
    float f[PER];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      f[i] = __half2float(w[off + i]);
      amax = fmaxf(amax, fabsf(f[i]));
    }
    amax = warp_max(amax);
    const __half s = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float sf = __half2float(s);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      int q = 0;
      if (sf > 0.0f) q = max(-127, min(127, (int)rintf(__fdiv_rn(f[i], sf))));
      codes[off + i] = (int8_t)q;
    }
    if (lane == 0) scales[(size_t)row * gpr + grp] = s;
  }
}

cudaError_t launch_quantize_int8(const void* w, int n, int k, int group, int8_t* codes, void* scales,
                                 cudaStream_t st) {
  const long long groups = (long long)n * (k / group);
  long long blocks = (groups + 7) / 8;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  const __half* wh = static_cast<const __half*>(w);
  __half* sh = static_cast<__half*>(scales);
  // (cudaLaunchKernelEx returns this launch's own error, not an earlier one)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  if (group == 32) return cudaLaunchKernelEx(&cfg, quantize_int8_kernel<1>, wh, n, k, codes, sh);
  if (group == 64) return cudaLaunchKernelEx(&cfg, quantize_int8_kernel<2>, wh, n, k, codes, sh);
  return cudaLaunchKernelEx(&cfg, quantize_int8_kernel<4>, wh, n, k, codes, sh);
}

// Self-test of the bounded-wait path: one thread waits on an mbarrier that
// nothing arrives on, with the same wait routine as the pipeline kernels and
// a budget of budget_ns.  The wait runs out, records kFlagWaitTimeout in
// *status and the kernel returns (no copy is in flight into its shared memory).
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(unsigned* status, unsigned long long budget_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_init_fence();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status, budget_ns);
}

cudaError_t launch_wait_timeout_selftest(unsigned* status, unsigned long long budget_ns, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = st;
  return cudaLaunchKernelEx(&cfg, wait_timeout_selftest_kernel, status, budget_ns);
}

}  // namespace ds
