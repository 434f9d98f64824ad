// Instantiations of the persistent step kernel for f16 weights (one
// translation unit per weight type so the library builds in parallel).
#include "step_launch.cuh"

namespace ds {

cudaError_t launch_step_f16(ActKind ak, const StepArgs& s, int grid, cudaStream_t st) {
  (void)ak;
  return launch_step_t<WKind::F16, __half>(s, grid, st);
}

cudaError_t prepare_step_f16(int max_smem) {
  return prepare_step_t<WKind::F16, __half>(max_smem);
}

int step_blocks_per_sm_f16(ActKind ak, int nt, size_t smem) {
  (void)ak;
  return step_blocks_per_sm_t<WKind::F16, __half>(nt, smem);
}

}  // namespace ds
