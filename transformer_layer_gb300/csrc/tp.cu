// Tensor-sliced (Megatron-style) layer: one rank's share of a layer step,
// split at the two all-reduce boundaries.
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持".  §3.2: the Attn and FF blocks are split across
// GPUs (Megatron-LM style), each followed by one cross-GPU all-reduce; §3.1,
// second fusion principle: fuse up to every all-reduce boundary, since the
// partial results must be reduced before anything after them can run; the
// injection-policy passage: the attention output GEMM and the layer output
// GEMM are the two linear layers whose results are reduced across ranks.
//
// Fusion regions of one rank (each a chain of programmatic-dependent launches):
//   attention partial: row LayerNorm1 -> QKV tile GEMM of the rank's heads
//     (bias, KV append) -> attention over the rank's heads -> O-proj tile GEMM
//     over the rank's Hl inputs whose epilogue writes the fp32 partial sum
//     (rank 0 also adds b_o and the residual x);
//   [all-reduce x1, by the caller]
//   FFN partial: row LayerNorm2 of the reduced x1 (two passes: statistics of
//     a sum cannot come from the ranks' partial statistics) -> FFN-up tile GEMM
//     of the rank's Fl features (bias, GeLU) -> FFN-down tile GEMM over those
//     features, fp32 partial (rank 0 adds b_2 and x1);
//   [all-reduce y, by the caller]
//   finish: y -> activation dtype.
#include <cuda.h>

#include <cmath>
#include <cstring>
#include <string>

#include "common.cuh"
#include "ds_layer.h"
#include "internal.h"

namespace ds {

constexpr int kFinishThreads = 256;

// y (fp32) -> out (activation dtype), 8 elements per thread and step.
template <typename ACT>
__global__ void __launch_bounds__(kFinishThreads) tp_finish_kernel(const float* __restrict__ y, ACT* __restrict__ out,
                                                                   size_t n8) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t stride = (size_t)gridDim.x * kFinishThreads;
  for (size_t i = (size_t)blockIdx.x * kFinishThreads + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(y)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(y)[2 * i + 1];
    uint4 o;
    o.x = Act<ACT>::pack2(a.x, a.y);
    o.y = Act<ACT>::pack2(a.z, a.w);
    o.z = Act<ACT>::pack2(b.x, b.y);
    o.w = Act<ACT>::pack2(b.z, b.w);
    reinterpret_cast<uint4*>(out)[i] = o;
  }
}

}  // namespace ds

using namespace ds;

struct ds_tp_layer {
  ds_tp_config cfg;
  ds_layer_weights w;
  int device = 0, sms = 0, max_smem = 0;
  // Tile tensor maps in device memory, 128 bytes each: QKV, O-proj, FFN-up,
  // FFN-down shards, each for ring stages of 64 and of 128 along K.
  unsigned char* tmaps = nullptr;
  const unsigned char* map(int r, int kc) const { return tmaps + (size_t)(2 * r + (kc == 128)) * 128; }
};

namespace {

ds_status tp_fail(ds_status s, const std::string& msg) {
  set_last_error(msg.c_str());
  return s;
}
ds_status launch_fail(const char* what, cudaError_t e) {
  return tp_fail(DS_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e));
}
bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr int kTpMaxRows = 4096;
constexpr int kTpBlocks = 10;

// Shape checks shared by every entry point; "" when the config is valid.
std::string tp_config_error(const ds_tp_config* c) {
  if (c == nullptr) return "config is null";
  const ds_layer_config& l = c->layer;
  if (l.hidden <= 0 || l.heads <= 0 || l.ffn <= 0 || l.hidden % l.heads != 0)
    return "hidden, heads and ffn must be positive with hidden % heads == 0";
  const int d = l.hidden / l.heads;
  if (d != 64 && d != 128) return "head_dim must be 64 or 128";
  if (!(l.ln_eps > 0.0f) || !std::isfinite(l.ln_eps)) return "ln_eps must be positive and finite";
  if (l.act_dtype != DS_F16 && l.act_dtype != DS_BF16) return "act_dtype must be DS_F16 or DS_BF16";
  if (l.weight_dtype != l.act_dtype) return "the tensor-sliced layer takes fp16 / bf16 weights of the activation dtype";
  if (c->tp_size < 1 || c->tp_size > 64) return "tp_size must be in 1..64";
  if (c->tp_rank < 0 || c->tp_rank >= c->tp_size) return "tp_rank must be in 0..tp_size-1";
  if (l.heads % c->tp_size != 0) return "tp_size must divide heads";
  if (l.hidden % 256 != 0 || l.ffn % 256 != 0) return "hidden and ffn must be multiples of 256";
  if ((l.hidden / c->tp_size) % 128 != 0 || (l.ffn / c->tp_size) % 128 != 0)
    return "hidden / tp_size and ffn / tp_size must be multiples of 128";
  return "";
}

// The rank's blocks of the full matrices (see ds_tp_block).
int tp_blocks(const ds_tp_config& c, ds_tp_block* out) {
  const int H = c.layer.hidden, F = c.layer.ffn, W = c.tp_size, r = c.tp_rank;
  const int Hl = H / W, Fl = F / W;
  int n = 0;
  for (int part = 0; part < 3; ++part)  // q, k, v rows of the rank's heads
    out[n++] = ds_tp_block{DS_TP_W_QKV, part * H + r * Hl, 0, Hl, H, H, part * Hl};
  for (int part = 0; part < 3; ++part)
    out[n++] = ds_tp_block{DS_TP_B_QKV, part * H + r * Hl, 0, Hl, 1, 1, part * Hl};
  out[n++] = ds_tp_block{DS_TP_W_O, 0, r * Hl, H, Hl, H, 0};      // inputs from the rank's heads
  out[n++] = ds_tp_block{DS_TP_W_FC1, r * Fl, 0, Fl, H, H, 0};    // the rank's FFN features
  out[n++] = ds_tp_block{DS_TP_B_FC1, r * Fl, 0, Fl, 1, 1, 0};
  out[n++] = ds_tp_block{DS_TP_W_FC2, 0, r * Fl, H, Fl, F, 0};
  return n;
}

struct TpPlans {
  DensePlan tq, to, tu, td;
};

bool tp_plans(const ds_tp_layer& L, int M, TpPlans* p) {
  const ActKind ak = L.cfg.layer.act_dtype == DS_BF16 ? ActKind::BF16 : ActKind::F16;
  const int H = L.cfg.layer.hidden, F = L.cfg.layer.ffn, W = L.cfg.tp_size;
  const int Hl = H / W, Fl = F / W;
  return dense_make_plan(ak, 3 * Hl, H, M, L.sms, L.max_smem, &p->tq) &&
         dense_make_plan(ak, H, Hl, M, L.sms, L.max_smem, &p->to) &&
         dense_make_plan(ak, Fl, H, M, L.sms, L.max_smem, &p->tu) &&
         dense_make_plan(ak, H, Fl, M, L.sms, L.max_smem, &p->td);
}

struct TpWs {
  size_t status, cnt, q, a_hi, a_lo, b_hi, b_lo, partials, total;
};

// Workspace regions (256-byte aligned): status word and arrival counters
// first (zero-filled once), q [M][Hl] fp32, operand A [M][H] (LayerNorm
// outputs), operand B [M][max(Hl, Fl)] (attention / GeLU outputs), split-K
// partials.
TpWs tp_ws(const ds_tp_layer& L, int M, const TpPlans& p) {
  const int H = L.cfg.layer.hidden, F = L.cfg.layer.ffn, W = L.cfg.tp_size;
  const int Hl = H / W, Fl = F / W;
  const bool split = L.cfg.layer.act_dtype == DS_BF16;
  TpWs w{};
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t o = off;
    off += up256(b);
    return o;
  };
  w.status = take(256);
  size_t tiles = 0, part = 0;
  for (const DensePlan* d : {&p.tq, &p.to, &p.tu, &p.td}) {
    tiles = std::max(tiles, (size_t)d->ws.tiles);
    const size_t pt = d->ws.KS > 1 ? (size_t)d->ws.tiles : (size_t)(d->ws.units - d->ws.U_dp);
    part = std::max(part, pt * d->ws.KS * d->ws.maxc * d->ntok * 128 * 4);
  }
  w.cnt = take(tiles * 4);
  w.q = take((size_t)M * Hl * 4);
  w.a_hi = take((size_t)M * H * 2);
  w.a_lo = split ? take((size_t)M * H * 2) : 0;
  const size_t bw = (size_t)std::max(Hl, Fl);
  w.b_hi = take((size_t)M * bw * 2);
  w.b_lo = split ? take((size_t)M * bw * 2) : 0;
  w.partials = take(part);
  w.total = off;
  return w;
}

ds_status check_current_device(const ds_tp_layer* L) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != L->device)
    return tp_fail(DS_ERR_INVALID_ARG, "the current device is not the device the layer was created on");
  return DS_OK;
}

}  // namespace

extern "C" {

int ds_tp_shard_blocks(const ds_tp_config* cfg, ds_tp_block* out, int cap) {
  const std::string why = tp_config_error(cfg);
  if (!why.empty()) {
    set_last_error(why.c_str());
    return -1;
  }
  if (out == nullptr || cap < kTpBlocks) {
    set_last_error("out is null or cap < 10");
    return -1;
  }
  return tp_blocks(*cfg, out);
}

ds_status ds_tp_shard_weights(const ds_tp_config* cfg, const ds_layer_weights* full, const ds_layer_weights* shard,
                              void* stream) {
  const std::string why = tp_config_error(cfg);
  if (!why.empty()) return tp_fail(DS_ERR_INVALID_ARG, why);
  if (full == nullptr || shard == nullptr) return tp_fail(DS_ERR_INVALID_ARG, "weights are null");
  const void* src[6] = {full->w_qkv, full->b_qkv, full->w_o, full->w_fc1, full->b_fc1, full->w_fc2};
  const void* dst[6] = {shard->w_qkv, shard->b_qkv, shard->w_o, shard->w_fc1, shard->b_fc1, shard->w_fc2};
  for (int i = 0; i < 6; ++i)
    if (src[i] == nullptr || dst[i] == nullptr) return tp_fail(DS_ERR_INVALID_ARG, "a sliced weight pointer is null");
  ds_tp_block b[kTpBlocks];
  const int n = tp_blocks(*cfg, b);
  const size_t es = 2;  // fp16 / bf16
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < n; ++i) {
    const char* s = static_cast<const char*>(src[b[i].matrix]) + ((size_t)b[i].src_row * b[i].src_cols + b[i].src_col) * es;
    char* d = static_cast<char*>(const_cast<void*>(dst[b[i].matrix])) + (size_t)b[i].dst_row * b[i].cols * es;
    const cudaError_t e = cudaMemcpy2DAsync(d, (size_t)b[i].cols * es, s, (size_t)b[i].src_cols * es,
                                            (size_t)b[i].cols * es, (size_t)b[i].rows, cudaMemcpyDefault, st);
    if (e != cudaSuccess)
      return tp_fail(DS_ERR_CUDA, std::string("cudaMemcpy2DAsync: ") + cudaGetErrorName(e));
  }
  return DS_OK;
}

ds_status ds_tp_layer_create(const ds_tp_config* cfg, const ds_layer_weights* w, ds_tp_layer** out) {
  if (out == nullptr) return tp_fail(DS_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  const std::string why = tp_config_error(cfg);
  if (!why.empty()) return tp_fail(DS_ERR_INVALID_ARG, why);
  if (w == nullptr) return tp_fail(DS_ERR_INVALID_ARG, "weights are null");
  const void* need[12] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o,
                          w->ln2_g, w->ln2_b, w->w_fc1, w->b_fc1, w->w_fc2, w->b_fc2};
  for (const void* p : need)
    if (!al16(p)) return tp_fail(DS_ERR_INVALID_ARG, "weight pointers must be non-null and 16-byte aligned");
  int dev = 0, sms = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return tp_fail(DS_ERR_CUDA, "device attributes");
  if (prepare_dense_kernels(max_smem) != cudaSuccess || prepare_attention_kernels(max_smem) != cudaSuccess ||
      prepare_attention_prefill_kernels(max_smem) != cudaSuccess)
    return tp_fail(DS_ERR_CUDA, "cudaFuncSetAttribute (tile / attention kernels)");
  ds_tp_layer* L = new ds_tp_layer();
  L->cfg = *cfg;
  L->w = *w;
  L->device = dev;
  L->sms = sms;
  L->max_smem = max_smem;
  const int H = cfg->layer.hidden, F = cfg->layer.ffn, W = cfg->tp_size;
  const int Hl = H / W, Fl = F / W;
  unsigned char host[8 * 128];
  std::memset(host, 0, sizeof(host));
  bool ok = true;
  for (int j = 0; j < 2 && ok; ++j) {
    const int kc = j ? 128 : 64;
    ok = encode_tile_map(host + (0 + j) * 128, w->w_qkv, 3 * Hl, H, 128, kc) &&
         encode_tile_map(host + (2 + j) * 128, w->w_o, H, Hl, 128, kc) &&
         encode_tile_map(host + (4 + j) * 128, w->w_fc1, Fl, H, 128, kc) &&
         encode_tile_map(host + (6 + j) * 128, w->w_fc2, H, Fl, 128, kc);
  }
  if (!ok) {
    delete L;
    return tp_fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight shard");
  }
  if (cudaMalloc(&L->tmaps, sizeof(host)) != cudaSuccess ||
      cudaMemcpy(L->tmaps, host, sizeof(host), cudaMemcpyHostToDevice) != cudaSuccess) {
    if (L->tmaps != nullptr) cudaFree(L->tmaps);
    delete L;
    return tp_fail(DS_ERR_CUDA, "tensor map upload");
  }
  TpPlans p;
  if (!tp_plans(*L, 1, &p)) {
    cudaFree(L->tmaps);
    delete L;
    return tp_fail(DS_ERR_UNSUPPORTED, "no tile split for this shape");
  }
  *out = L;
  return DS_OK;
}

ds_status ds_tp_layer_destroy(ds_tp_layer* L) {
  if (L != nullptr && L->tmaps != nullptr) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(L->device);
    cudaFree(L->tmaps);
    cudaSetDevice(cur);
  }
  delete L;
  return DS_OK;
}

size_t ds_tp_layer_workspace_bytes(const ds_tp_layer* L, int batch, int new_tokens) {
  if (L == nullptr || batch < 1 || new_tokens < 1 || (long long)batch * new_tokens > kTpMaxRows) return 0;
  TpPlans p;
  if (!tp_plans(*L, batch * new_tokens, &p)) return 0;
  return tp_ws(*L, batch * new_tokens, p).total;
}

ds_status ds_tp_attention_partial(ds_tp_layer* L, const void* x_in, float* x1_part, int batch, int new_tokens,
                                  void* k_cache, void* v_cache, int max_len, const int32_t* past_len,
                                  void* workspace, size_t ws_bytes, void* stream) {
  if (L == nullptr) return tp_fail(DS_ERR_INVALID_ARG, "layer is null");
  if (!al16(x_in) || !al16(x1_part) || !al16(k_cache) || !al16(v_cache))
    return tp_fail(DS_ERR_INVALID_ARG, "x_in, x1_part and the caches must be non-null and 16-byte aligned");
  if (past_len == nullptr || (reinterpret_cast<uintptr_t>(past_len) & 3u) != 0)
    return tp_fail(DS_ERR_INVALID_ARG, "past_len must be non-null and int32-aligned");
  if (batch < 1 || new_tokens < 1 || (long long)batch * new_tokens > kTpMaxRows)
    return tp_fail(DS_ERR_UNSUPPORTED, "batch * new_tokens must be in 1..4096");
  if (max_len < new_tokens) return tp_fail(DS_ERR_INVALID_ARG, "max_len must be at least new_tokens");
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return tp_fail(DS_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (const ds_status s = check_current_device(L); s != DS_OK) return s;
  const int B = batch, T = new_tokens, M = B * T;
  TpPlans p;
  if (!tp_plans(*L, M, &p)) return tp_fail(DS_ERR_UNSUPPORTED, "no tile split for this shape");
  const TpWs wl = tp_ws(*L, M, p);
  if (ws_bytes < wl.total) return tp_fail(DS_ERR_WORKSPACE, "workspace smaller than ds_tp_layer_workspace_bytes()");
  const ds_layer_config& c = L->cfg.layer;
  const int H = c.hidden, W = L->cfg.tp_size, r = L->cfg.tp_rank;
  const int Hl = H / W, nhl = c.heads / W, d = H / c.heads;
  const ActKind ak = c.act_dtype == DS_BF16 ? ActKind::BF16 : ActKind::F16;
  const bool split = ak == ActKind::BF16;
  char* b = static_cast<char*>(workspace);
  auto at = [&](size_t off) -> void* { return off ? static_cast<void*>(b + off) : nullptr; };
  unsigned* status = reinterpret_cast<unsigned*>(b + wl.status);
  int* cnt = reinterpret_cast<int*>(b + wl.cnt);
  float* q = static_cast<float*>(at(wl.q));
  void *a_hi = at(wl.a_hi), *a_lo = at(wl.a_lo), *b_hi = at(wl.b_hi), *b_lo = at(wl.b_lo);
  float* partials = static_cast<float*>(at(wl.partials));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  alignas(64) unsigned char ma[2][128], mb[2][128];
  std::memset(ma, 0, sizeof(ma));
  std::memset(mb, 0, sizeof(mb));
  bool ok = encode_tile_map(ma[0], a_hi, M, H, p.tq.ntok, p.tq.kc) &&
            encode_tile_map(mb[0], b_hi, M, Hl, p.to.ntok, p.to.kc);
  if (ok && split)
    ok = encode_tile_map(ma[1], a_lo, M, H, p.tq.ntok, p.tq.kc) && encode_tile_map(mb[1], b_lo, M, Hl, p.to.ntok, p.to.kc);
  if (!ok) return tp_fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation operand");
  cudaError_t e;
  // LayerNorm1 rows -> operand A (first launch of the call: no programmatic
  // overlap with whatever precedes it, e.g. the caller's collective)
  LnPrepArgs lp;
  lp.M = M;
  lp.K = H;
  lp.eps = c.ln_eps;
  lp.x_act = x_in;
  lp.ln_g = L->w.ln1_g;
  lp.ln_b = L->w.ln1_b;
  lp.out_hi = a_hi;
  lp.out_lo = a_lo;
  if ((e = launch_ln_prep(ak, lp, st, false)) != cudaSuccess) return launch_fail("row LayerNorm launch", e);
  DenseArgs base;
  base.M = M;
  base.B = B;
  base.T = T;
  base.partials = partials;
  base.counters = cnt;
  base.status = status;
  base.H = Hl;
  // QKV of the rank's heads + bias + KV append
  DenseArgs r1 = base;
  r1.tmap_w = L->map(0, p.tq.kc);
  r1.N = 3 * Hl;
  r1.K = H;
  r1.plan = p.tq;
  r1.bias = L->w.b_qkv;
  r1.out_f32 = q;
  r1.k_cache = k_cache;
  r1.v_cache = v_cache;
  r1.heads = nhl;
  r1.head_dim = d;
  r1.max_len = max_len;
  r1.past_len = past_len;
  if ((e = launch_dense(Region::LnQkv, ak, r1, ma[0], split ? ma[1] : nullptr, st, true)) != cudaSuccess)
    return launch_fail("QKV launch", e);
  // attention over the rank's heads, output in the operand format
  AttnArgs ra;
  ra.q = q;
  ra.k_cache = k_cache;
  ra.v_cache = v_cache;
  ra.past_len = past_len;
  ra.B = B;
  ra.T = T;
  ra.heads = nhl;
  ra.head_dim = d;
  ra.max_len = max_len;
  ra.H = Hl;
  ra.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  attn_configure(ra, L->cfg.layer.act_dtype == DS_BF16 ? ActKind::BF16 : ActKind::F16, L->sms, L->max_smem);
  ra.status = status;
  ra.out_hi = b_hi;
  ra.out_lo = b_lo;
  e = T >= kPrefillMinTokens ? launch_attention_prefill(ak, ra, st, true) : launch_attention(ak, ra, st, true);
  if (e != cudaSuccess) return launch_fail("attention launch", e);
  // O-proj over the rank's inputs: the fp32 partial sum (rank 0: + b_o + x)
  DenseArgs r3 = base;
  r3.tmap_w = L->map(1, p.to.kc);
  r3.N = H;
  r3.K = Hl;
  r3.plan = p.to;
  r3.bias = r == 0 ? L->w.b_o : nullptr;
  r3.resid_act = r == 0 ? x_in : nullptr;
  r3.out_f32 = x1_part;
  if ((e = launch_dense(Region::OprojRes, ak, r3, mb[0], split ? mb[1] : nullptr, st, true)) != cudaSuccess)
    return launch_fail("O-proj launch", e);
  add_launches(4);
  return DS_OK;
}

ds_status ds_tp_ffn_partial(ds_tp_layer* L, const float* x1, float* y_part, int rows, void* workspace,
                            size_t ws_bytes, void* stream) {
  if (L == nullptr) return tp_fail(DS_ERR_INVALID_ARG, "layer is null");
  if (!al16(x1) || !al16(y_part) || x1 == y_part)
    return tp_fail(DS_ERR_INVALID_ARG, "x1 and y_part must be non-null, 16-byte aligned and not alias");
  if (rows < 1 || rows > kTpMaxRows) return tp_fail(DS_ERR_UNSUPPORTED, "rows must be in 1..4096");
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return tp_fail(DS_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (const ds_status s = check_current_device(L); s != DS_OK) return s;
  const int M = rows;
  TpPlans p;
  if (!tp_plans(*L, M, &p)) return tp_fail(DS_ERR_UNSUPPORTED, "no tile split for this shape");
  const TpWs wl = tp_ws(*L, M, p);
  if (ws_bytes < wl.total) return tp_fail(DS_ERR_WORKSPACE, "workspace smaller than ds_tp_layer_workspace_bytes()");
  const ds_layer_config& c = L->cfg.layer;
  const int H = c.hidden, W = L->cfg.tp_size, r = L->cfg.tp_rank;
  const int Fl = c.ffn / W;
  const ActKind ak = c.act_dtype == DS_BF16 ? ActKind::BF16 : ActKind::F16;
  const bool split = ak == ActKind::BF16;
  char* b = static_cast<char*>(workspace);
  auto at = [&](size_t off) -> void* { return off ? static_cast<void*>(b + off) : nullptr; };
  unsigned* status = reinterpret_cast<unsigned*>(b + wl.status);
  int* cnt = reinterpret_cast<int*>(b + wl.cnt);
  void *a_hi = at(wl.a_hi), *a_lo = at(wl.a_lo), *b_hi = at(wl.b_hi), *b_lo = at(wl.b_lo);
  float* partials = static_cast<float*>(at(wl.partials));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  alignas(64) unsigned char ma[2][128], mb[2][128];
  std::memset(ma, 0, sizeof(ma));
  std::memset(mb, 0, sizeof(mb));
  bool ok = encode_tile_map(ma[0], a_hi, M, H, p.tu.ntok, p.tu.kc) &&
            encode_tile_map(mb[0], b_hi, M, Fl, p.td.ntok, p.td.kc);
  if (ok && split)
    ok = encode_tile_map(ma[1], a_lo, M, H, p.tu.ntok, p.tu.kc) && encode_tile_map(mb[1], b_lo, M, Fl, p.td.ntok, p.td.kc);
  if (!ok) return tp_fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation operand");
  cudaError_t e;
  // LayerNorm2 of the reduced x1 (statistics by two passes over each row)
  LnPrepArgs lp;
  lp.M = M;
  lp.K = H;
  lp.eps = c.ln_eps;
  lp.x_f32 = x1;
  lp.ln_g = L->w.ln2_g;
  lp.ln_b = L->w.ln2_b;
  lp.out_hi = a_hi;
  lp.out_lo = a_lo;
  if ((e = launch_ln_prep(ak, lp, st, false)) != cudaSuccess) return launch_fail("row LayerNorm launch", e);
  DenseArgs base;
  base.M = M;
  base.B = M;
  base.T = 1;
  base.partials = partials;
  base.counters = cnt;
  base.status = status;
  base.H = H;
  // FFN-up of the rank's features + bias + GeLU -> operand B
  DenseArgs u = base;
  u.tmap_w = L->map(2, p.tu.kc);
  u.N = Fl;
  u.K = H;
  u.plan = p.tu;
  u.bias = L->w.b_fc1;
  u.out_act = b_hi;
  u.out_lo = b_lo;
  if ((e = launch_dense(Region::FfnUp, ak, u, ma[0], split ? ma[1] : nullptr, st, true)) != cudaSuccess)
    return launch_fail("FFN-up launch", e);
  // FFN-down over the rank's features: the fp32 partial sum (rank 0: + b_2 + x1)
  DenseArgs dn = base;
  dn.tmap_w = L->map(3, p.td.kc);
  dn.N = H;
  dn.K = Fl;
  dn.plan = p.td;
  dn.bias = r == 0 ? L->w.b_fc2 : nullptr;
  dn.resid_f32 = r == 0 ? x1 : nullptr;
  dn.out_f32 = y_part;
  if ((e = launch_dense(Region::FfnDown, ak, dn, mb[0], split ? mb[1] : nullptr, st, true)) != cudaSuccess)
    return launch_fail("FFN-down launch", e);
  add_launches(3);
  return DS_OK;
}

ds_status ds_tp_finish(ds_tp_layer* L, const float* y, void* x_out, int rows, void* stream) {
  if (L == nullptr) return tp_fail(DS_ERR_INVALID_ARG, "layer is null");
  if (!al16(y) || !al16(x_out)) return tp_fail(DS_ERR_INVALID_ARG, "y and x_out must be non-null and 16-byte aligned");
  if (rows < 1 || rows > kTpMaxRows) return tp_fail(DS_ERR_UNSUPPORTED, "rows must be in 1..4096");
  if (const ds_status s = check_current_device(L); s != DS_OK) return s;
  const size_t n8 = (size_t)rows * L->cfg.layer.hidden / 8;
  cudaLaunchConfig_t cfg = {};
  const size_t blocks = (n8 + kFinishThreads - 1) / kFinishThreads;
  cfg.gridDim = dim3((unsigned)std::min<size_t>(blocks, (size_t)L->sms * 8));
  cfg.blockDim = dim3(kFinishThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (L->cfg.layer.act_dtype == DS_BF16)
    e = cudaLaunchKernelEx(&cfg, tp_finish_kernel<__nv_bfloat16>, y, static_cast<__nv_bfloat16*>(x_out), n8);
  else
    e = cudaLaunchKernelEx(&cfg, tp_finish_kernel<__half>, y, static_cast<__half*>(x_out), n8);
  if (e != cudaSuccess) return tp_fail(DS_ERR_CUDA, std::string("finish launch: ") + cudaGetErrorName(e));
  add_launches(1);
  return DS_OK;
}

}  // extern "C"
