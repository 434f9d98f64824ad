// Cooperative launch of the step kernel for one weight / activation pair.
#pragma once
#include "step_impl.cuh"

namespace ds {

template <WKind WK, typename ACT>
cudaError_t launch_step_t(const StepArgs& s, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = step_smem_bytes(s.plan[0].nt, s.stages, s.SB, s.xs_cap);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the grid barrier needs it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (s.plan[0].nt) {
    case 1: return cudaLaunchKernelEx(&cfg, step_kernel<WK, ACT, 1>, s);
    case 2: return cudaLaunchKernelEx(&cfg, step_kernel<WK, ACT, 2>, s);
    case 4: return cudaLaunchKernelEx(&cfg, step_kernel<WK, ACT, 4>, s);
    case 8: return cudaLaunchKernelEx(&cfg, step_kernel<WK, ACT, 8>, s);
  }
  return cudaErrorInvalidValue;
}

// CTAs of the step kernel that fit on one SM with `smem` dynamic shared memory.
template <WKind WK, typename ACT>
int step_blocks_per_sm_t(int nt, size_t smem) {
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (nt) {
    case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<WK, ACT, 1>, kStepThreads, smem); break;
    case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<WK, ACT, 2>, kStepThreads, smem); break;
    case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<WK, ACT, 4>, kStepThreads, smem); break;
    case 8: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<WK, ACT, 8>, kStepThreads, smem); break;
  }
  return e == cudaSuccess ? n : 0;
}

template <WKind WK, typename ACT>
cudaError_t prepare_step_t(int max_smem) {
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(step_kernel<WK, ACT, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(step_kernel<WK, ACT, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(step_kernel<WK, ACT, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(step_kernel<WK, ACT, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  return e;
}

}  // namespace ds
