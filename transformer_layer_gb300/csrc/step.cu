// Host side of the persistent decode-step kernel: ring geometry shared by all
// phases, attention split count, cooperative launch.
#include "step_impl.cuh"

namespace ds {

cudaError_t launch_step_f16(ActKind ak, const StepArgs& s, int grid, cudaStream_t st);
cudaError_t launch_step_bf16(ActKind ak, const StepArgs& s, int grid, cudaStream_t st);
cudaError_t launch_step_i8(ActKind ak, const StepArgs& s, int grid, cudaStream_t st);
cudaError_t prepare_step_f16(int max_smem);
cudaError_t prepare_step_bf16(int max_smem);
cudaError_t prepare_step_i8(int max_smem);
int step_blocks_per_sm_f16(ActKind ak, int nt, size_t smem);
int step_blocks_per_sm_bf16(ActKind ak, int nt, size_t smem);
int step_blocks_per_sm_i8(ActKind ak, int nt, size_t smem);

int step_blocks_per_sm(WKind wk, ActKind ak, int nt, size_t smem) {
  switch (wk) {
    case WKind::F16: return step_blocks_per_sm_f16(ak, nt, smem);
    case WKind::BF16: return step_blocks_per_sm_bf16(ak, nt, smem);
    case WKind::I8: return step_blocks_per_sm_i8(ak, nt, smem);
  }
  return 0;
}

// Key splits per (b, h): enough items for two attention groups per CTA, at
// most one item per group, each split at least ~16 keys.
int step_attn_nsplit(int B, int heads, int max_len, int grid) {
  const int bh = B * heads;
  int ns = (2 * grid) / bh;
  if (ns < 1) ns = 1;
  if (ns > 16) ns = 16;
  const int cap = (max_len + 15) / 16;
  if (ns > cap) ns = cap < 1 ? 1 : cap;
  return ns;
}

size_t step_smem_bytes(int nt, int stages, size_t SB, size_t xs_cap) {
  switch (nt) {
    case 1: return gemv_smem_bytes<1>(stages, SB, xs_cap, kAttnScratchFloats);
    case 2: return gemv_smem_bytes<2>(stages, SB, xs_cap, kAttnScratchFloats);
    case 4: return gemv_smem_bytes<4>(stages, SB, xs_cap, kAttnScratchFloats);
    default: return gemv_smem_bytes<8>(stages, SB, xs_cap, kAttnScratchFloats);
  }
}

// One ring for all phases: stage stride = the largest phase's stage, staged-x
// space = the largest phase's slice; as many stages as fit (up to kMaxStages).
bool step_geometry(WKind wk, ActKind ak, int M, int max_smem, StepArgs* s) {
  const bool i8 = (wk == WKind::I8);
  const int esize = i8 ? 1 : 2, pad = i8 ? 8 : 32;
  const bool split = (ak == ActKind::BF16);
  size_t SB = 0, xs = 0;
  for (int i = 0; i < 4; ++i) {
    const GemvPlan& p = s->plan[i];
    const size_t sb = SmemLayout<1>::stage_bytes(p.chunk_k, esize, i8);
    const size_t x = SmemLayout<1>::xs_bytes(M, p.K_S, pad, split);
    if (sb > SB) SB = sb;
    if (x > xs) xs = x;
  }
  const int nt = s->plan[0].nt;
  int stages = kMaxStages;
  while (stages >= 3 && step_smem_bytes(nt, stages, SB, xs) > (size_t)max_smem) --stages;
  if (stages < 3) return false;
  s->stages = stages;
  s->SB = SB;
  s->xs_cap = xs;
  return true;
}

cudaError_t launch_step(WKind wk, ActKind ak, const StepArgs& s, int grid, cudaStream_t st) {
  switch (wk) {
    case WKind::F16: return launch_step_f16(ak, s, grid, st);
    case WKind::BF16: return launch_step_bf16(ak, s, grid, st);
    case WKind::I8: return launch_step_i8(ak, s, grid, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_step_kernels(int max_smem) {
  cudaError_t e = prepare_step_f16(max_smem);
  if (e == cudaSuccess) e = prepare_step_bf16(max_smem);
  if (e == cudaSuccess) e = prepare_step_i8(max_smem);
  return e;
}

}  // namespace ds
