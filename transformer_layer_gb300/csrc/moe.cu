// Residual-MoE (PR-MoE) FFN block on one GPU: the FFN of a layer replaced by
// a dense MLP plus one expert chosen per token by a gate.
//
// Page cited as [P3]: "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、PR-MoE
// 优化与 init_inference 全解析", section "用 PR-MoE 结构进一步提速并降低推理成本"
// (mlp_type 'residual', per-layer expert counts) and the configuration table
// (moe.type standard / residual, moe_experts).  The page gives no formula; the
// reading taken (the plainest one for a residual MoE with top-1 routing):
//   h = LN2(x);  p = softmax(h W_g^T) over the E experts;  e = argmax p (ties:
//   the lowest index);  y = x + MLP(h) + p_e * Expert_e(h),
// where MLP and every expert are GeLU FFNs of the layer's shape (W1 [F][H] +
// b1, GeLU, W2 [H][F] + b2) and W_g is [E][H] without bias.
//
// Launch chain (programmatic dependent launch throughout):
//   1. row LayerNorm of x -> h (tensor-core operand format);
//   2. gate: logits in fp32 (one CTA per row), softmax, argmax -> e[m], p_e[m];
//   3. dense FFN-up (tile kernel, GeLU) -> g;  4. dense FFN-down with the
//      residual -> y_d = x + MLP(h) (fp32);
//   5. per row m: expert FFN-up of expert e[m] on row m, then expert
//      FFN-down scaled by p_e[m] with residual y_d[m] -> y[m].  The expert's
//      weights are chosen on the device (tile kernel with a tensor-map table
//      indexed by e[m], read after the dependency wait): no host sync.
#include <cuda.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "ds_layer.h"
#include "internal.h"

namespace ds {

constexpr int kGateThreads = 256;

// One CTA per row m: logits[e] = h[m] . W_g[e] (h = hi + lo of the operand),
// then the softmax weight and the argmax (lowest index on ties).
template <typename ACT>
__global__ void __launch_bounds__(kGateThreads) moe_gate_kernel(const ACT* __restrict__ h_hi, const ACT* __restrict__ h_lo,
                                                               const ACT* __restrict__ wg, int E, int H,
                                                               int32_t* __restrict__ idx, float* __restrict__ pw) {
  extern __shared__ float gsm[];
  float* hs = gsm;          // [H]
  float* lg = gsm + H;      // [E]
  __shared__ float red_v[kGateThreads / 32];
  __shared__ int red_i[kGateThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int k = tid; k < H; k += kGateThreads) {
    float v = Act<ACT>::to_f(h_hi[(size_t)m * H + k]);
    if (h_lo != nullptr) v += Act<ACT>::to_f(h_lo[(size_t)m * H + k]);
    hs[k] = v;
  }
  __syncthreads();
  // one warp per expert row of W_g (coalesced), lanes split H
  for (int e = warp; e < E; e += kGateThreads / 32) {
    float s = 0.f;
    const ACT* w = wg + (size_t)e * H;
    for (int k = lane * 8; k < H; k += 256) {
      const uint4 u = *reinterpret_cast<const uint4*>(w + k);
      const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = Act<ACT>::unpack2(uw[j]);
        s += f.x * hs[k + 2 * j] + f.y * hs[k + 2 * j + 1];
      }
    }
    s = warp_sum(s);
    if (lane == 0) lg[e] = s;
  }
  __syncthreads();
  // argmax (largest logit, lowest index on ties)
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int e = tid; e < E; e += kGateThreads) {
    const float v = lg[e];
    if (v > bv || (v == bv && e < bi)) {
      bv = v;
      bi = e;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if (lane == 0) {
    red_v[warp] = bv;
    red_i[warp] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kGateThreads / 32; ++w)
      if (red_v[w] > red_v[0] || (red_v[w] == red_v[0] && red_i[w] < red_i[0])) {
        red_v[0] = red_v[w];
        red_i[0] = red_i[w];
      }
  }
  __syncthreads();
  const float mx = red_v[0];
  float z = 0.f;
  for (int e = tid; e < E; e += kGateThreads) z += expf(lg[e] - mx);
  z = warp_sum(z);
  __syncthreads();
  if (lane == 0) red_v[warp] = z;
  __syncthreads();
  if (tid == 0) {
    float zz = 0.f;
    for (int w = 0; w < kGateThreads / 32; ++w) zz += red_v[w];
    idx[m] = red_i[0];
    pw[m] = 1.0f / zz;  // softmax weight of the argmax: exp(0) / sum
  }
}

cudaError_t launch_moe_gate(ActKind ak, const void* h_hi, const void* h_lo, const void* wg, int M, int E, int H,
                            int32_t* idx, float* pw, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(kGateThreads);
  cfg.dynamicSmemBytes = (size_t)(H + E) * 4;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (ak == ActKind::F16)
    return cudaLaunchKernelEx(&cfg, moe_gate_kernel<__half>, static_cast<const __half*>(h_hi),
                              static_cast<const __half*>(h_lo), static_cast<const __half*>(wg), E, H, idx, pw);
  return cudaLaunchKernelEx(&cfg, moe_gate_kernel<__nv_bfloat16>, static_cast<const __nv_bfloat16*>(h_hi),
                            static_cast<const __nv_bfloat16*>(h_lo), static_cast<const __nv_bfloat16*>(wg), E, H,
                            idx, pw);
}

// Raises the gate kernel's dynamic shared-memory limit to what its static
// shared memory leaves of the per-block maximum.
cudaError_t prepare_moe_kernels(int max_smem) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, moe_gate_kernel<__half>);
  if (e != cudaSuccess) return e;
  const int dyn = max_smem - (int)fa.sharedSizeBytes;
  e = cudaFuncSetAttribute(moe_gate_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(moe_gate_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  return e;
}

}  // namespace ds

using namespace ds;

struct ds_moe_ffn {
  ds_moe_config cfg;
  ds_moe_weights w;
  int device = 0, sms = 0, max_smem = 0;
  // Tensor maps in device memory, 128 bytes each: [0..3] the dense W1, W2 for
  // ring stages of 64 and 128 along K; then the experts' W1 maps (E for
  // stages of 64, E for 128), then their W2 maps likewise.
  unsigned char* tmaps = nullptr;
  const unsigned char* dense_map(int which, int kc) const { return tmaps + (size_t)(2 * which + (kc == 128)) * 128; }
  const unsigned char* expert_table(int which, int kc) const {
    const int E = cfg.experts;
    return tmaps + (size_t)(4 + (2 * which + (kc == 128)) * E) * 128;
  }
};

namespace {

ds_status moe_fail(ds_status s, const char* msg) {
  set_last_error(msg);
  return s;
}
bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct MoePlans {
  DensePlan up, down, eup, edown;  // dense FFN-up (M rows), FFN-down (M rows), expert ones (1 row)
};

bool moe_plans(const ds_moe_ffn& m, int M, MoePlans* p) {
  const ActKind ak = m.cfg.act_dtype == DS_BF16 ? ActKind::BF16 : ActKind::F16;
  const int H = m.cfg.hidden, F = m.cfg.ffn;
  return dense_make_plan(ak, F, H, M, m.sms, m.max_smem, &p->up) &&
         dense_make_plan(ak, H, F, M, m.sms, m.max_smem, &p->down) &&
         dense_make_plan(ak, F, H, 1, m.sms, m.max_smem, &p->eup) &&
         dense_make_plan(ak, H, F, 1, m.sms, m.max_smem, &p->edown);
}

struct MoeWs {
  size_t status, cnt, h_hi, h_lo, g_hi, g_lo, ge_hi, ge_lo, yd, idx, pw, partials, total;
};

MoeWs moe_ws(const ds_moe_ffn& m, int M, const MoePlans& p) {
  const int H = m.cfg.hidden, F = m.cfg.ffn;
  const bool split = m.cfg.act_dtype == DS_BF16;
  MoeWs w{};
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t o = off;
    off += up256(b);
    return o;
  };
  w.status = take(256);
  size_t tiles = 0, part = 0;
  for (const DensePlan* d : {&p.up, &p.down, &p.eup, &p.edown}) {
    tiles = std::max(tiles, (size_t)d->ws.tiles);
    const size_t pt = d->ws.KS > 1 ? (size_t)d->ws.tiles : (size_t)(d->ws.units - d->ws.U_dp);
    part = std::max(part, pt * d->ws.KS * d->ws.maxc * d->ntok * 128 * 4);
  }
  w.cnt = take(tiles * 4);
  w.h_hi = take((size_t)M * H * 2);
  w.h_lo = split ? take((size_t)M * H * 2) : 0;
  w.g_hi = take((size_t)M * F * 2);
  w.g_lo = split ? take((size_t)M * F * 2) : 0;
  w.ge_hi = take((size_t)M * F * 2);
  w.ge_lo = split ? take((size_t)M * F * 2) : 0;
  w.yd = take((size_t)M * H * 4);
  w.idx = take((size_t)M * 4);
  w.pw = take((size_t)M * 4);
  w.partials = take(part);
  w.total = off;
  return w;
}

}  // namespace

extern "C" {

ds_status ds_moe_ffn_create(const ds_moe_config* cfg, const ds_moe_weights* w, ds_moe_ffn** out) {
  if (out == nullptr) return moe_fail(DS_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  if (cfg == nullptr || w == nullptr) return moe_fail(DS_ERR_INVALID_ARG, "config or weights are null");
  if (cfg->hidden <= 0 || cfg->ffn <= 0 || cfg->hidden % 256 != 0 || cfg->ffn % 256 != 0)
    return moe_fail(DS_ERR_UNSUPPORTED, "hidden and ffn must be positive multiples of 256");
  if (cfg->experts < 1 || cfg->experts > 1024) return moe_fail(DS_ERR_UNSUPPORTED, "experts must be in 1..1024");
  if (cfg->act_dtype != DS_F16 && cfg->act_dtype != DS_BF16)
    return moe_fail(DS_ERR_INVALID_ARG, "act_dtype must be DS_F16 or DS_BF16");
  if (!(cfg->ln_eps > 0.0f) || !std::isfinite(cfg->ln_eps)) return moe_fail(DS_ERR_INVALID_ARG, "ln_eps must be positive");
  const void* ptrs[11] = {w->ln2_g, w->ln2_b, w->w_gate, w->w_fc1, w->b_fc1, w->w_fc2, w->b_fc2,
                          w->we_fc1, w->be_fc1, w->we_fc2, w->be_fc2};
  for (const void* p : ptrs)
    if (!al16(p)) return moe_fail(DS_ERR_INVALID_ARG, "weight pointers must be non-null and 16-byte aligned");
  int dev = 0, sms = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return moe_fail(DS_ERR_CUDA, "device attributes");
  // the tile and row kernels' limits are raised by ds_layer_create's device set-up; do it here as well
  if (prepare_dense_kernels(max_smem) != cudaSuccess || prepare_moe_kernels(max_smem) != cudaSuccess)
    return moe_fail(DS_ERR_CUDA, "cudaFuncSetAttribute (tile / gate kernels)");
  ds_moe_ffn* m = new ds_moe_ffn();
  m->cfg = *cfg;
  m->w = *w;
  m->device = dev;
  m->sms = sms;
  m->max_smem = max_smem;
  const int H = cfg->hidden, F = cfg->ffn, E = cfg->experts;
  std::vector<unsigned char> host((size_t)(4 + 4 * E) * 128, 0);
  bool ok = true;
  for (int j = 0; j < 2 && ok; ++j) {
    const int kc = j ? 128 : 64;
    ok = encode_tile_map(host.data() + (size_t)(0 + j) * 128, w->w_fc1, F, H, 128, kc) &&
         encode_tile_map(host.data() + (size_t)(2 + j) * 128, w->w_fc2, H, F, 128, kc);
    for (int e = 0; e < E && ok; ++e) {
      const char* w1 = static_cast<const char*>(w->we_fc1) + (size_t)e * F * H * 2;
      const char* w2 = static_cast<const char*>(w->we_fc2) + (size_t)e * H * F * 2;
      ok = encode_tile_map(host.data() + (size_t)(4 + (0 + j) * E + e) * 128, w1, F, H, 128, kc) &&
           encode_tile_map(host.data() + (size_t)(4 + (2 + j) * E + e) * 128, w2, H, F, 128, kc);
    }
  }
  if (!ok) {
    delete m;
    return moe_fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an MoE weight matrix");
  }
  if (cudaMalloc(&m->tmaps, host.size()) != cudaSuccess ||
      cudaMemcpy(m->tmaps, host.data(), host.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    if (m->tmaps != nullptr) cudaFree(m->tmaps);
    delete m;
    return moe_fail(DS_ERR_CUDA, "tensor map upload");
  }
  MoePlans p;
  if (!moe_plans(*m, 1, &p)) {
    cudaFree(m->tmaps);
    delete m;
    return moe_fail(DS_ERR_UNSUPPORTED, "no tile split for this shape");
  }
  *out = m;
  return DS_OK;
}

ds_status ds_moe_ffn_destroy(ds_moe_ffn* m) {
  if (m != nullptr && m->tmaps != nullptr) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(m->device);
    cudaFree(m->tmaps);
    cudaSetDevice(cur);
  }
  delete m;
  return DS_OK;
}

size_t ds_moe_ffn_workspace_bytes(const ds_moe_ffn* m, int rows) {
  if (m == nullptr || rows < 1 || rows > 4096) return 0;
  MoePlans p;
  if (!moe_plans(*m, rows, &p)) return 0;
  return moe_ws(*m, rows, p).total;
}

ds_status ds_moe_ffn_forward(ds_moe_ffn* m, const void* x_in, void* x_out, int rows, int32_t* expert_out,
                             void* workspace, size_t ws_bytes, void* stream) {
  if (m == nullptr) return moe_fail(DS_ERR_INVALID_ARG, "moe is null");
  if (!al16(x_in) || !al16(x_out) || x_in == x_out)
    return moe_fail(DS_ERR_INVALID_ARG, "x_in / x_out must be 16-byte aligned, non-null and not alias");
  if (rows < 1 || rows > 4096) return moe_fail(DS_ERR_UNSUPPORTED, "rows must be in 1..4096");
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return moe_fail(DS_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (expert_out != nullptr && (reinterpret_cast<uintptr_t>(expert_out) & 3u) != 0)
    return moe_fail(DS_ERR_INVALID_ARG, "expert_out must be int32-aligned");
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != m->device)
    return moe_fail(DS_ERR_INVALID_ARG, "the current device is not the device the block was created on");
  const int M = rows, H = m->cfg.hidden, F = m->cfg.ffn, E = m->cfg.experts;
  if ((size_t)(H + E) * 4 + 1024 > (size_t)m->max_smem) return moe_fail(DS_ERR_UNSUPPORTED, "gate shared memory");
  MoePlans p;
  if (!moe_plans(*m, M, &p)) return moe_fail(DS_ERR_UNSUPPORTED, "no tile split for this shape");
  const MoeWs wl = moe_ws(*m, M, p);
  if (ws_bytes < wl.total) return moe_fail(DS_ERR_WORKSPACE, "workspace smaller than ds_moe_ffn_workspace_bytes()");
  const ActKind ak = m->cfg.act_dtype == DS_BF16 ? ActKind::BF16 : ActKind::F16;
  const bool split = ak == ActKind::BF16;
  char* b = static_cast<char*>(workspace);
  auto at = [&](size_t off) -> void* { return off ? static_cast<void*>(b + off) : nullptr; };
  unsigned* status = reinterpret_cast<unsigned*>(b + wl.status);
  int* cnt = reinterpret_cast<int*>(b + wl.cnt);
  void *h_hi = at(wl.h_hi), *h_lo = at(wl.h_lo), *g_hi = at(wl.g_hi), *g_lo = at(wl.g_lo);
  char *ge_hi = static_cast<char*>(at(wl.ge_hi)), *ge_lo = static_cast<char*>(at(wl.ge_lo));
  float* yd = static_cast<float*>(at(wl.yd));
  int32_t* idx = static_cast<int32_t*>(at(wl.idx));
  float* pw = static_cast<float*>(at(wl.pw));
  float* partials = static_cast<float*>(at(wl.partials));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // activation operand maps: h [M][H], g [M][F]; per row: h row, ge row
  alignas(64) unsigned char mh[2][128], mg[2][128];
  std::memset(mh, 0, sizeof(mh));
  std::memset(mg, 0, sizeof(mg));
  const int nt = p.up.ntok, kc = p.up.kc;
  bool ok = encode_tile_map(mh[0], h_hi, M, H, nt, kc) && encode_tile_map(mg[0], g_hi, M, F, p.down.ntok, p.down.kc);
  if (ok && split)
    ok = encode_tile_map(mh[1], h_lo, M, H, nt, kc) && encode_tile_map(mg[1], g_lo, M, F, p.down.ntok, p.down.kc);
  if (!ok) return moe_fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation operand");
  cudaError_t e;
  // 1. LN2 rows -> h
  LnPrepArgs lp;
  lp.M = M;
  lp.K = H;
  lp.eps = m->cfg.ln_eps;
  lp.x_act = x_in;
  lp.ln_g = m->w.ln2_g;
  lp.ln_b = m->w.ln2_b;
  lp.out_hi = h_hi;
  lp.out_lo = h_lo;
  if ((e = launch_ln_prep(ak, lp, st, false)) != cudaSuccess) return moe_fail(DS_ERR_CUDA, "row LayerNorm launch");
  // 2. gate
  if ((e = launch_moe_gate(ak, h_hi, h_lo, m->w.w_gate, M, E, H, idx, pw, st)) != cudaSuccess)
    return moe_fail(DS_ERR_CUDA, "gate launch");
  DenseArgs base;
  base.B = M;
  base.T = 1;
  base.partials = partials;
  base.counters = cnt;
  base.status = status;
  base.H = H;
  // 3. dense FFN-up + GeLU -> g
  DenseArgs u = base;
  u.tmap_w = m->dense_map(0, p.up.kc);
  u.N = F;
  u.K = H;
  u.M = M;
  u.plan = p.up;
  u.bias = m->w.b_fc1;
  u.out_act = g_hi;
  u.out_lo = g_lo;
  if ((e = launch_dense(Region::FfnUp, ak, u, mh[0], split ? mh[1] : nullptr, st, true)) != cudaSuccess)
    return moe_fail(DS_ERR_CUDA, "dense FFN-up launch");
  // 4. dense FFN-down + bias + residual x -> y_d (fp32)
  DenseArgs d = base;
  d.tmap_w = m->dense_map(1, p.down.kc);
  d.N = H;
  d.K = F;
  d.M = M;
  d.plan = p.down;
  d.bias = m->w.b_fc2;
  d.resid_act = x_in;
  d.out_f32 = yd;
  if ((e = launch_dense(Region::OprojRes, ak, d, mg[0], split ? mg[1] : nullptr, st, true)) != cudaSuccess)
    return moe_fail(DS_ERR_CUDA, "dense FFN-down launch");
  // 5. per row: the chosen expert's FFN, weighted, added to y_d
  for (int r = 0; r < M; ++r) {
    alignas(64) unsigned char rh[2][128], rg[2][128];
    std::memset(rh, 0, sizeof(rh));
    std::memset(rg, 0, sizeof(rg));
    char* hr_hi = static_cast<char*>(h_hi) + (size_t)r * H * 2;
    char* hr_lo = split ? static_cast<char*>(h_lo) + (size_t)r * H * 2 : nullptr;
    char* gr_hi = ge_hi + (size_t)r * F * 2;
    char* gr_lo = split ? ge_lo + (size_t)r * F * 2 : nullptr;
    ok = encode_tile_map(rh[0], hr_hi, 1, H, p.eup.ntok, p.eup.kc) &&
         encode_tile_map(rg[0], gr_hi, 1, F, p.edown.ntok, p.edown.kc);
    if (ok && split)
      ok = encode_tile_map(rh[1], hr_lo, 1, H, p.eup.ntok, p.eup.kc) &&
           encode_tile_map(rg[1], gr_lo, 1, F, p.edown.ntok, p.edown.kc);
    if (!ok) return moe_fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an expert operand");
    DenseArgs eu = base;
    eu.tmap_table = m->expert_table(0, p.eup.kc);
    eu.sel_idx = idx + r;
    eu.sel_bias_stride = F;
    eu.N = F;
    eu.K = H;
    eu.M = 1;
    eu.plan = p.eup;
    eu.bias = m->w.be_fc1;
    eu.out_act = gr_hi;
    eu.out_lo = gr_lo;
    if ((e = launch_dense(Region::FfnUp, ak, eu, rh[0], split ? rh[1] : nullptr, st, true)) != cudaSuccess)
      return moe_fail(DS_ERR_CUDA, "expert FFN-up launch");
    DenseArgs ed = base;
    ed.tmap_table = m->expert_table(1, p.edown.kc);
    ed.sel_idx = idx + r;
    ed.sel_scale = pw + r;
    ed.sel_bias_stride = H;
    ed.N = H;
    ed.K = F;
    ed.M = 1;
    ed.plan = p.edown;
    ed.bias = m->w.be_fc2;
    ed.resid_f32 = yd + (size_t)r * H;
    ed.out_act = static_cast<char*>(x_out) + (size_t)r * H * 2;
    if ((e = launch_dense(Region::FfnDown, ak, ed, rg[0], split ? rg[1] : nullptr, st, true)) != cudaSuccess)
      return moe_fail(DS_ERR_CUDA, "expert FFN-down launch");
  }
  add_launches(4ull + 2ull * (unsigned long long)M);
  if (expert_out != nullptr) {
    e = cudaMemcpyAsync(expert_out, idx, (size_t)M * 4, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return moe_fail(DS_ERR_CUDA, "expert index copy");
  }
  return DS_OK;
}

}  // extern "C"
