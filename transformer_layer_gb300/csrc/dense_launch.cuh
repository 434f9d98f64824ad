// Launch and set-up of the tensor-core tile region kernels for one activation
// type (included by dense_f16.cu and dense_bf16.cu).
#pragma once

#include "dense_impl.cuh"

namespace ds {

template <typename ACT, bool kI8 = false>
cudaError_t launch_dense_t(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                           cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan.ws.grid);
  cfg.blockDim = dim3(kI8 ? kDenseThreadsI8 : kDenseThreads);
  cfg.dynamicSmemBytes = a.plan.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (a.plan.cluster > 1) {  // the K slices of one tile: consecutive CTAs, one cluster
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)a.plan.cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  switch (r) {
    case Region::LnQkv: return cudaLaunchKernelEx(&cfg, dense_region_kernel<Region::LnQkv, ACT, kI8>, *xh, *xl, a);
    case Region::OprojRes:
      return cudaLaunchKernelEx(&cfg, dense_region_kernel<Region::OprojRes, ACT, kI8>, *xh, *xl, a);
    case Region::FfnUp: return cudaLaunchKernelEx(&cfg, dense_region_kernel<Region::FfnUp, ACT, kI8>, *xh, *xl, a);
    case Region::FfnDown:
      return cudaLaunchKernelEx(&cfg, dense_region_kernel<Region::FfnDown, ACT, kI8>, *xh, *xl, a);
  }
  return cudaErrorInvalidValue;
}

// Raises the dynamic shared-memory limit of the four region kernels (once per
// device, before any launch or capture).
template <typename ACT, bool kI8 = false>
cudaError_t prepare_dense_t(int max_smem) {
  cudaError_t e = cudaSuccess;
#define DS_PREP_DENSE(REG)                                                                                        \
  if (e == cudaSuccess)                                                                                           \
  e = cudaFuncSetAttribute(dense_region_kernel<REG, ACT, kI8>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           max_smem)
  DS_PREP_DENSE(Region::LnQkv);
  DS_PREP_DENSE(Region::OprojRes);
  DS_PREP_DENSE(Region::FfnUp);
  DS_PREP_DENSE(Region::FfnDown);
#undef DS_PREP_DENSE
  return e;
}

}  // namespace ds
