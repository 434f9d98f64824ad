// Instantiations of the tensor-core tile region kernels for fp16 (one
// translation unit per activation type so the library builds in parallel).
#include "dense_launch.cuh"

namespace ds {

cudaError_t launch_dense_f16(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                             cudaStream_t st, bool pdl) {
  return launch_dense_t<__half>(r, a, xh, xl, st, pdl);
}

cudaError_t prepare_dense_f16(int max_smem) { return prepare_dense_t<__half>(max_smem); }

}  // namespace ds
