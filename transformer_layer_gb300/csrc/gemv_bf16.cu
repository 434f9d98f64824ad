// Instantiations of the region GEMV kernels for bf16 weights (one translation
// unit per weight type so the library builds in parallel).
#include "gemv_impl.cuh"

namespace ds {

cudaError_t launch_region_bf16(Region r, ActKind ak, const RegionArgs& a, cudaStream_t st,
                               bool pdl) {
  (void)ak;
  return launch_region_t<WKind::BF16, __nv_bfloat16>(r, a, st, pdl);
}

cudaError_t prepare_region_bf16(int max_smem) {
  return prepare_region_t<WKind::BF16, __nv_bfloat16>(max_smem);
}

}  // namespace ds
