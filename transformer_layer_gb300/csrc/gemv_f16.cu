// Instantiations of the region GEMV kernels for f16 weights (one translation
// unit per weight type so the library builds in parallel).
#include "gemv_impl.cuh"

namespace ds {

cudaError_t launch_region_f16(Region r, ActKind ak, const RegionArgs& a, cudaStream_t st,
                               bool pdl) {
  (void)ak;
  return launch_region_t<WKind::F16, __half>(r, a, st, pdl);
}

cudaError_t prepare_region_f16(int max_smem) {
  return prepare_region_t<WKind::F16, __half>(max_smem);
}

}  // namespace ds
