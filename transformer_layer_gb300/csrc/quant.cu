// MoQ-style int8 weight quantisation (load-time kernel).
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持", §5.2: int8 inference with the quantisation
// grouping passed as quantization_setting.  Rule implemented (the page fixes no
// rounding; this is the reading the library documents): per group of 64
// consecutive weights along K, s = fp16_rne(float32(max|w|) / 127) and
// q = clamp(rne(w / s), -127, 127) with IEEE float32 division; s = 0 and q = 0
// for an all-zero group.
#include "common.cuh"
#include "internal.h"

namespace ds {

// One warp per group of 64 weights; lane i owns weights 2i and 2i+1.
__global__ void __launch_bounds__(256) quantize_int8_kernel(const __half* __restrict__ w, int n,
                                                            int k, int8_t* __restrict__ codes,
                                                            __half* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const long long gpr = k / 64;
  const long long total = (long long)n * gpr;
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; gw < total;
       gw += nwarps) {
    const long long row = gw / gpr, grp = gw - (gw / gpr) * gpr;
    const size_t off = (size_t)row * k + (size_t)grp * 64 + 2 * lane;
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(w + off));
    const float amax = warp_max(fmaxf(fabsf(f.x), fabsf(f.y)));
    const __half s = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float sf = __half2float(s);
    int q0 = 0, q1 = 0;
    if (sf > 0.0f) {
      q0 = (int)rintf(__fdiv_rn(f.x, sf));
      q1 = (int)rintf(__fdiv_rn(f.y, sf));
      q0 = max(-127, min(127, q0));
      q1 = max(-127, min(127, q1));
    }
    char2 out;
    out.x = (signed char)q0;
    out.y = (signed char)q1;
    *reinterpret_cast<char2*>(codes + off) = out;
    if (lane == 0) scales[(size_t)row * gpr + grp] = s;
  }
}

cudaError_t launch_quantize_int8(const void* w, int n, int k, int8_t* codes, void* scales,
                                 cudaStream_t st) {
  const long long groups = (long long)n * (k / 64);
  long long blocks = (groups + 7) / 8;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  quantize_int8_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const __half*>(w), n, k, codes,
                                                         static_cast<__half*>(scales));
  return cudaGetLastError();
}

}  // namespace ds
