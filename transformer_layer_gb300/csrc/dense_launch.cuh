// Launch and set-up of the tensor-core tile region kernels for one activation
// type (included by dense_f16.cu, dense_bf16.cu and dense_i8.cu).
#pragma once

#include "dense_impl.cuh"

namespace ds {

using DenseKernel = decltype(&dense_region_kernel<Region::LnQkv, __half, false, 1>);

// The instance of region R for nis MMA issuers (int8 runs two).
template <Region R, typename ACT, bool kI8>
DenseKernel dense_kernel(int nis) {
  if constexpr (kI8) {
    return &dense_region_kernel<R, ACT, true, kDenseMaxIssuers>;
  } else {
    return nis == kDenseMaxIssuers ? &dense_region_kernel<R, ACT, false, kDenseMaxIssuers>
                                   : &dense_region_kernel<R, ACT, false, 1>;
  }
}

template <typename ACT, bool kI8>
DenseKernel dense_kernel(Region r, int nis) {
  switch (r) {
    case Region::LnQkv: return dense_kernel<Region::LnQkv, ACT, kI8>(nis);
    case Region::OprojRes: return dense_kernel<Region::OprojRes, ACT, kI8>(nis);
    case Region::FfnUp: return dense_kernel<Region::FfnUp, ACT, kI8>(nis);
    case Region::FfnDown: return dense_kernel<Region::FfnDown, ACT, kI8>(nis);
  }
  return nullptr;
}

template <typename ACT, bool kI8 = false>
cudaError_t launch_dense_t(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                           cudaStream_t st, bool pdl) {
  const int nis = dense_issuers(a.plan.ntok, a.plan.stages, kI8);
  const DenseKernel k = dense_kernel<ACT, kI8>(r, nis);
  if (k == nullptr) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.plan.ws.grid);
  cfg.blockDim = dim3(dense_threads(kI8, nis));
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
  return cudaLaunchKernelEx(&cfg, k, *xh, *xl, a);
}

// Raises the dynamic shared-memory limit of the region kernels, for every
// issuer count (once per device, before any launch or capture).
template <typename ACT, bool kI8 = false>
cudaError_t prepare_dense_t(int max_smem) {
  cudaError_t e = cudaSuccess;
  for (int r = 0; r < 4; ++r)
    for (int nis = 1; nis <= kDenseMaxIssuers; ++nis) {
      if (kI8 && nis != kDenseMaxIssuers) continue;
      const DenseKernel k = dense_kernel<ACT, kI8>(static_cast<Region>(r), nis);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    }
  return e;
}

}  // namespace ds
