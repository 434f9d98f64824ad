// Instantiations of the tensor-core tile region kernels for int8 weight codes
// with fp16 activations (one translation unit, so the library builds in
// parallel).
#include "dense_launch.cuh"

namespace ds {

cudaError_t launch_dense_i8(Region r, const DenseArgs& a, const CUtensorMap* xh, const CUtensorMap* xl,
                            cudaStream_t st, bool pdl) {
  return launch_dense_t<__half, true>(r, a, xh, xl, st, pdl);
}

cudaError_t prepare_dense_i8(int max_smem) { return prepare_dense_t<__half, true>(max_smem); }

}  // namespace ds
