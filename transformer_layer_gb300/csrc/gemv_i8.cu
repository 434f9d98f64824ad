// Instantiations of the region GEMV kernels for i8 weights (one translation
// unit per weight type so the library builds in parallel).
#include "gemv_impl.cuh"

namespace ds {

cudaError_t launch_region_i8_bf16(Region r, const RegionArgs& a, cudaStream_t st, bool pdl);
cudaError_t prepare_region_i8_bf16(int max_smem);

cudaError_t launch_region_i8(Region r, ActKind ak, const RegionArgs& a, cudaStream_t st,
                               bool pdl) {
  if (ak == ActKind::F16) return launch_region_t<WKind::I8, __half>(r, a, st, pdl);
  return launch_region_i8_bf16(r, a, st, pdl);
}

cudaError_t prepare_region_i8(int max_smem) {
  cudaError_t e = prepare_region_t<WKind::I8, __half>(max_smem);
  if (e != cudaSuccess) return e;
  return prepare_region_i8_bf16(max_smem);
}

}  // namespace ds
