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

// Bytes of shared memory the staged x slice may use.
static constexpr size_t kXBudget = 96 * 1024;

// Chooses K slice length and grid so that every CTA gets the same number of
// items to within one.  Items are 16 rows x K_S; the score is the fraction of
// the grid's item slots that hold work, preferring longer slices on ties
// (fewer split-K partials to reduce).
bool gemv_make_plan(WKind wk, ActKind ak, int N, int K, int M, int num_sms, int ctas_per_sm,
                    GemvPlan* plan) {
  if (N <= 0 || K <= 0 || M < 1 || M > 64 || (N % 16) != 0) return false;
  GemvPlan p;
  p.nt = M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 32 ? 4 : 8));
  const int blk_k = (wk == WKind::I8) ? 64 : 32;
  const int pad = (wk == WKind::I8) ? 8 : 32;
  const bool split = (ak == ActKind::BF16);
  p.nblk = (K % (kWarps * 2 * blk_k) == 0) ? 2 : 1;
  const int unit = kWarps * p.nblk * blk_k;
  if (K % unit != 0) return false;
  p.tiles = N / 16;
  const int G = num_sms * ctas_per_sm;
  double best = -1.0;
  int best_ks = 0;
  for (int d = 1; d <= K / unit; ++d) {  // K_S = K / d, longest first
    if ((K / unit) % d != 0) continue;
    const int K_S = K / d;
    size_t xs = 0;
    switch (p.nt) {
      case 1: xs = SmemLayout<1>::xs_bytes(K_S, pad, split); break;
      case 2: xs = SmemLayout<2>::xs_bytes(K_S, pad, split); break;
      case 4: xs = SmemLayout<4>::xs_bytes(K_S, pad, split); break;
      default: xs = SmemLayout<8>::xs_bytes(K_S, pad, split); break;
    }
    if (xs > kXBudget) continue;
    const long long items = (long long)d * p.tiles;
    const long long g = items < G ? items : G;
    const long long per = (items + g - 1) / g;
    const double eff = (double)items / ((double)G * (double)per);
    if (eff > best + 0.01) {
      best = eff;
      best_ks = K_S;
    }
  }
  if (best_ks == 0) return false;
  p.K_S = best_ks;
  p.KS = K / best_ks;
  p.items = p.KS * p.tiles;
  p.grid = p.items < G ? p.items : G;
  switch (p.nt) {
    case 1: p.smem = SmemLayout<1>::total(p.K_S, pad, split); break;
    case 2: p.smem = SmemLayout<2>::total(p.K_S, pad, split); break;
    case 4: p.smem = SmemLayout<4>::total(p.K_S, pad, split); break;
    default: p.smem = SmemLayout<8>::total(p.K_S, pad, split); break;
  }
  *plan = p;
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
