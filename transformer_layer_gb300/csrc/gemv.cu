// Work split and dispatch of the region GEMV kernels (host side).
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持", §3 intro (skinny GEMM tuned for small batch).
#include "gemv_impl.cuh"

namespace ds {

cudaError_t launch_region_f16(Region r, ActKind ak, const RegionArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_region_bf16(Region r, ActKind ak, const RegionArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_region_i8(Region r, ActKind ak, const RegionArgs& a, cudaStream_t st, bool pdl);
cudaError_t prepare_region_f16(int max_smem);
cudaError_t prepare_region_bf16(int max_smem);
cudaError_t prepare_region_i8(int max_smem);

// Bytes of shared memory the staged x slice may use (two CTAs share an SM).
static constexpr size_t kXBudget = 80 * 1024;

static size_t xs_bytes_nt(int nt, int M, int K_S, int pad, bool split) {
  switch (nt) {
    case 1: return SmemLayout<1>::xs_bytes(M, K_S, pad, split);
    case 2: return SmemLayout<2>::xs_bytes(M, K_S, pad, split);
    case 4: return SmemLayout<4>::xs_bytes(M, K_S, pad, split);
    default: return SmemLayout<8>::xs_bytes(M, K_S, pad, split);
  }
}
static size_t fixed_nt(int nt, int M, int K_S, int pad, bool split) {
  switch (nt) {
    case 1: return SmemLayout<1>::fixed(M, K_S, pad, split);
    case 2: return SmemLayout<2>::fixed(M, K_S, pad, split);
    case 4: return SmemLayout<4>::fixed(M, K_S, pad, split);
    default: return SmemLayout<8>::fixed(M, K_S, pad, split);
  }
}

bool gemv_make_plan(WKind wk, ActKind ak, int N, int K, int M, int num_sms, int max_smem, GemvPlan* plan) {
  const bool i8 = (wk == WKind::I8);
  const int blk_k = i8 ? 64 : 32;
  const int pad = i8 ? 8 : 32;
  const int esize = i8 ? 1 : 2;
  const bool split = (ak == ActKind::BF16);
  const int nt = M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 32 ? 4 : 8));
  auto xs = [&](int K_S) { return xs_bytes_nt(nt, M, K_S, pad, split); };
  if (!ws_make_plan(N, K, M, num_sms, blk_k, kProducers, kXBudget, xs, plan))
    return false;
  // As deep a weight ring as the rest of shared memory allows (up to kMaxStages).
  const size_t fixed = fixed_nt(plan->nt, M, plan->K_S, pad, split);
  const size_t stage = SmemLayout<1>::stage_bytes(plan->chunk_k, esize, i8) + 16;
  if ((size_t)max_smem <= fixed + 1024) return false;
  size_t s = ((size_t)max_smem - fixed - 1024) / stage;
  if (s > (size_t)kMaxStages) s = kMaxStages;
  if (s < 2) return false;
  plan->stages = (int)s;
  plan->smem = 1024 + fixed + s * stage;  // + alignment of the ring to 1024 bytes
  return true;
}

cudaError_t launch_region(Region r, WKind wk, ActKind ak, const RegionArgs& a, cudaStream_t st,
                          bool pdl) {
  switch (wk) {
    case WKind::F16: return launch_region_f16(r, ak, a, st, pdl);
    case WKind::BF16: return launch_region_bf16(r, ak, a, st, pdl);
    case WKind::I8: return launch_region_i8(r, ak, a, st, pdl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_region_kernels(int max_smem) {
  cudaError_t e = prepare_region_f16(max_smem);
  if (e == cudaSuccess) e = prepare_region_bf16(max_smem);
  if (e == cudaSuccess) e = prepare_region_i8(max_smem);
  return e;
}

}  // namespace ds
