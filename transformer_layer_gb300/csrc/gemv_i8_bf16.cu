// Instantiations of the region GEMV kernels for int8 weights with bf16
// activations (own translation unit so the library builds in parallel).
#include "gemv_impl.cuh"

namespace ds {

cudaError_t launch_region_i8_bf16(Region r, const RegionArgs& a, cudaStream_t st, bool pdl) {
  return launch_region_t<WKind::I8, __nv_bfloat16>(r, a, st, pdl);
}

cudaError_t prepare_region_i8_bf16(int max_smem) { return prepare_region_t<WKind::I8, __nv_bfloat16>(max_smem); }

}  // namespace ds
