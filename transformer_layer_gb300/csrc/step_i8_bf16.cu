// Instantiations of the persistent step kernel for int8 weights with bf16
// activations (own translation unit so the library builds in parallel).
#include "step_launch.cuh"

namespace ds {

cudaError_t launch_step_i8_bf16(const StepArgs& s, int grid, cudaStream_t st) {
  return launch_step_t<WKind::I8, __nv_bfloat16>(s, grid, st);
}

cudaError_t prepare_step_i8_bf16(int max_smem) { return prepare_step_t<WKind::I8, __nv_bfloat16>(max_smem); }

int step_blocks_per_sm_i8_bf16(int nt, size_t smem) {
  return step_blocks_per_sm_t<WKind::I8, __nv_bfloat16>(nt, smem);
}

}  // namespace ds
