// Instantiations of the persistent step kernel for int8 weights with fp16 activations (one
// translation unit per weight type so the library builds in parallel).
#include "step_launch.cuh"

namespace ds {

cudaError_t launch_step_i8_bf16(const StepArgs& s, int grid, cudaStream_t st);
cudaError_t prepare_step_i8_bf16(int max_smem);
int step_blocks_per_sm_i8_bf16(int nt, size_t smem);

cudaError_t launch_step_i8(ActKind ak, const StepArgs& s, int grid, cudaStream_t st) {
  if (ak == ActKind::F16) return launch_step_t<WKind::I8, __half>(s, grid, st);
  return launch_step_i8_bf16(s, grid, st);
}

cudaError_t prepare_step_i8(int max_smem) {
  cudaError_t e = prepare_step_t<WKind::I8, __half>(max_smem);
  if (e != cudaSuccess) return e;
  return prepare_step_i8_bf16(max_smem);
}

int step_blocks_per_sm_i8(ActKind ak, int nt, size_t smem) {
  (void)ak;
  if (ak == ActKind::F16) return step_blocks_per_sm_t<WKind::I8, __half>(nt, smem);
  return step_blocks_per_sm_i8_bf16(nt, smem);
}

}  // namespace ds
