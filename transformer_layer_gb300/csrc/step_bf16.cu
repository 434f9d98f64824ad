// Instantiations of the persistent step kernel for bf16 weights (one
// translation unit per weight type so the library builds in parallel).
#include "step_launch.cuh"

namespace ds {

cudaError_t launch_step_bf16(ActKind ak, const StepArgs& s, int grid, cudaStream_t st) {
  (void)ak;
  return launch_step_t<WKind::BF16, __nv_bfloat16>(s, grid, st);
}

cudaError_t prepare_step_bf16(int max_smem) {
  return prepare_step_t<WKind::BF16, __nv_bfloat16>(max_smem);
}

int step_blocks_per_sm_bf16(ActKind ak, int nt, size_t smem) {
  (void)ak;
  return step_blocks_per_sm_t<WKind::BF16, __nv_bfloat16>(nt, smem);
}

}  // namespace ds
