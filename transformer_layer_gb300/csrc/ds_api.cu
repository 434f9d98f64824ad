// C-ABI entry points of libdslayer.so (declared and documented in ds_layer.h).
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持".  A layer runs as the four fusion regions of
// §3.2; region 3 of the page (intermediate FF + LayerNorm + bias + residual +
// GeLU) is launched as two kernels, O-proj + residual + LayerNorm2 statistics
// and LayerNorm2 + FFN-up + GeLU, and region 4 (bias + residual) is fused into
// the FFN-down kernel's epilogue.  The all-reduce boundaries of §3.1 collapse on
// one GPU; they remain as the kernel boundaries.
//
// Host-side responsibilities here: argument validation before any launch,
// workspace layout, the per-GEMV work split, the launch chain with
// programmatic dependent launch, CUDA-graph capture/replay of a stack step,
// and per-region event timing in profile mode.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ds_layer.h"
#include "internal.h"

using namespace ds;

namespace {

thread_local std::string g_err;
std::atomic<unsigned long long> g_launches{0};

ds_status fail(ds_status s, const std::string& msg) {
  g_err = msg;
  return s;
}
ds_status cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return DS_ERR_CUDA;
}
bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DevInfo {
  bool ready = false;
  int sms = 0;
  int max_smem = 0;     // opt-in shared memory of one block
  int smem_per_sm = 0;  // shared memory of one SM (shared by its resident blocks)
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

// Queries the current device once and raises the kernels' shared-memory limit.
ds_status device_info(int* dev_out, DevInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(DS_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    e = cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(max smem)");
    e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem per SM)");
    e = prepare_region_kernels(d.max_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(region kernels)");
    e = prepare_attention_kernels(d.max_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention kernel)");
    e = prepare_step_kernels(d.max_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(step kernel)");
    d.ready = true;
  }
  *dev_out = dev;
  *out = d;
  return DS_OK;
}

int ctas_per_sm_knob() {
  const char* s = std::getenv("DS_GEMV_CTAS_PER_SM");
  if (s == nullptr) return 1;
  const int v = std::atoi(s);
  return (v >= 1 && v <= 4) ? v : 1;
}

// A stack step runs as the chain of region kernels (graph-captured, PDL
// overlapped); DS_STEP_KERNEL=1 selects the persistent step kernel instead
// where it can run (one cooperative launch per step; measured slower on
// GB300, kept for comparison).
bool step_kernel_knob() {
  const char* s = std::getenv("DS_STEP_KERNEL");
  return s != nullptr && std::atoi(s) != 0;
}

WKind wkind(ds_dtype d) { return d == DS_I8 ? WKind::I8 : (d == DS_BF16 ? WKind::BF16 : WKind::F16); }
ActKind akind(ds_dtype d) { return d == DS_BF16 ? ActKind::BF16 : ActKind::F16; }

}  // namespace

struct ds_layer {
  ds_layer_config cfg;
  ds_layer_weights w;
  int device = 0;
  int sms = 0;
  int max_smem = 0;
  int smem_per_sm = 0;
  int ctas_per_sm = 1;
  // TMA tensor maps in device memory, kTensorMapBytes each: weights of QKV,
  // O-proj, FFN-up, FFN-down, then (int8) their scales in the same order, one
  // map per k-blocks-per-step choice (1, 2, 4): a map's box is one chunk.
  unsigned char* tmaps = nullptr;
  static int nblk_index(int nblk) { return nblk == 4 ? 2 : (nblk == 2 ? 1 : 0); }
  const void* tmap_w(int r, int nblk) const { return tmaps + (size_t)(3 * r + nblk_index(nblk)) * kTensorMapBytes; }
  const void* tmap_s(int r, int nblk) const {
    return cfg.weight_dtype == DS_I8 ? tmaps + (size_t)(12 + 3 * r + nblk_index(nblk)) * kTensorMapBytes : nullptr;
  }
  // int8 scale group length of matrix r (0 QKV, 1 O-proj, 2 FFN-up, 3 FFN-down):
  // the FFN matrices take half the length under mlp_extra_grouping.
  int qgroup(int r) const { return (r >= 2 && cfg.mlp_extra_grouping == 1) ? cfg.quant_group / 2 : cfg.quant_group; }
};

namespace {

struct Plans {
  GemvPlan qkv, o, up, down;  // region kernels (ds_layer_forward, profile mode)
  GemvPlan step[4];           // persistent step kernel: one CTA per SM for every phase
  bool step_ok = false;
};

bool make_plans(const ds_layer& L, int M, int B, Plans* p) {
  (void)B;
  const int H = L.cfg.hidden, F = L.cfg.ffn;
  const WKind wk = wkind(L.cfg.weight_dtype);
  const ActKind ak = akind(L.cfg.act_dtype);
  // Several CTAs per SM share its shared memory (1 KB of it reserved per CTA).
  const int cps = L.ctas_per_sm;
  const int smem = cps == 1 ? L.max_smem : std::min(L.max_smem, L.smem_per_sm / cps - 1024);
  if (!gemv_make_plan(wk, ak, 3 * H, H, M, L.sms, cps, smem, &p->qkv)) return false;
  if (!gemv_make_plan(wk, ak, H, H, M, L.sms, cps, smem, &p->o)) return false;
  if (!gemv_make_plan(wk, ak, F, H, M, L.sms, cps, smem, &p->up)) return false;
  if (!gemv_make_plan(wk, ak, H, F, M, L.sms, cps, smem, &p->down)) return false;
  if (wk == WKind::I8) {  // the scale box of a chunk must hold at least 8 groups
    const GemvPlan* pl[4] = {&p->qkv, &p->o, &p->up, &p->down};
    for (int i = 0; i < 4; ++i)
      if (pl[i]->chunk_k / L.qgroup(i) < 8) return false;
  }
  const int NK[4][2] = {{3 * H, H}, {H, H}, {F, H}, {H, F}};
  p->step_ok = true;
  for (int i = 0; i < 4; ++i)
    if (!gemv_make_plan(wk, ak, NK[i][0], NK[i][1], M, L.sms, 1, L.max_smem, &p->step[i], true) ||
        (wk == WKind::I8 && p->step[i].chunk_k / L.qgroup(i) < 8))
      p->step_ok = false;
  return true;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t status, cnt_gemv, grid_bar, attn_cnt, q, o, x1, g, stats_a, stats_b, partials, attn_part, act,
      total;
};

// Workspace regions, each 256-byte aligned.  Counters first so that a
// zero-fill of the first bytes is enough to reset them.
WsLayout ws_layout(const ds_layer& L, int B, int T, const Plans& p) {
  const int H = L.cfg.hidden, F = L.cfg.ffn, nh = L.cfg.heads, d = H / nh;
  const size_t M = (size_t)B * T;
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up256(bytes);
    return o;
  };
  w.status = take(256);
  const size_t tiles_max = (size_t)std::max(3 * H, F) / 16;
  w.cnt_gemv = take(tiles_max * sizeof(int));
  w.grid_bar = take(sizeof(unsigned));
  w.attn_cnt = take((size_t)B * nh * sizeof(int));
  w.q = take(M * H * 4);
  w.o = take(M * H * 4);
  w.x1 = take(M * H * 4);
  w.g = take(M * F * 4);
  w.stats_a = take((size_t)(H / 16) * M * 2 * 4);
  w.stats_b = take((size_t)(H / 16) * M * 2 * 4);
  size_t part = 0;
  const GemvPlan* ps[4] = {&p.qkv, &p.o, &p.up, &p.down};
  for (int i = 0; i < 4; ++i) {
    part = std::max(part, (size_t)ps[i]->tiles * ps[i]->KS * ps[i]->maxc * 16 * M * 4);
    const GemvPlan& q = p.step[i];
    if (p.step_ok) part = std::max(part, (size_t)q.tiles * q.KS * q.maxc * 16 * M * 4);
  }
  w.partials = take(part);
  w.attn_part = take((size_t)B * nh * step_attn_nsplit(B, nh, 1 << 30, L.sms) * (d + 2) * 4);
  w.act = take(2 * M * H * 2);
  w.total = off;
  return w;
}

ds_status validate_config(const ds_layer_config* c) {
  if (c == nullptr) return fail(DS_ERR_INVALID_ARG, "config is null");
  if (c->hidden <= 0 || c->heads <= 0 || c->ffn <= 0 || c->hidden % c->heads != 0)
    return fail(DS_ERR_INVALID_ARG, "hidden, heads and ffn must be positive with hidden % heads == 0");
  const int d = c->hidden / c->heads;
  if (d != 64 && d != 128) return fail(DS_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (!(c->ln_eps > 0.0f) || !std::isfinite(c->ln_eps))
    return fail(DS_ERR_INVALID_ARG, "ln_eps must be positive and finite");
  if (c->act_dtype != DS_F16 && c->act_dtype != DS_BF16)
    return fail(DS_ERR_INVALID_ARG, "act_dtype must be DS_F16 or DS_BF16");
  if (c->weight_dtype == DS_I8) {
    // One MMA sums 16 codes spread over a 64-code block, so a scale must be
    // uniform over each block: groups of 64 or 128 (32 would need the scale
    // applied before the MMA).
    if (c->quant_group != 64 && c->quant_group != 128)
      return fail(DS_ERR_UNSUPPORTED, "quant_group must be 64 or 128 for the layer (32 only for ds_quantize_int8)");
    if (c->mlp_extra_grouping != 0 && c->mlp_extra_grouping != 1)
      return fail(DS_ERR_INVALID_ARG, "mlp_extra_grouping must be 0 or 1");
    const int g_mlp = c->mlp_extra_grouping == 1 ? c->quant_group / 2 : c->quant_group;
    if (g_mlp < 64)
      return fail(DS_ERR_UNSUPPORTED, "mlp_extra_grouping needs quant_group 128 (FFN groups of 64)");
    // a weight chunk (8 warps x blocks of 64 codes) spans at least 8 scale
    // groups: each matrix's K is a multiple of 8 groups and of 512
    const int kmul_h = std::max(512, 8 * c->quant_group), kmul_f = std::max(512, 8 * g_mlp);
    if (c->hidden % kmul_h != 0 || c->ffn % kmul_f != 0)
      return fail(DS_ERR_UNSUPPORTED, "int8 weights need hidden and ffn multiples of 512 (of 1024 for groups of 128)");
  } else if (c->weight_dtype == c->act_dtype) {
    if (c->hidden % 256 != 0 || c->ffn % 256 != 0)
      return fail(DS_ERR_UNSUPPORTED, "hidden and ffn must be multiples of 256");
  } else {
    return fail(DS_ERR_UNSUPPORTED, "fp16/bf16 weights must have the activation dtype");
  }
  return DS_OK;
}

struct Bufs {
  unsigned* status;
  int* cnt_gemv;
  unsigned* grid_bar;
  int* attn_cnt;
  float *q, *o, *x1, *g, *stats_a, *stats_b, *partials, *attn_part;
  char* act;
};

Bufs bufs_of(void* ws, const WsLayout& w) {
  char* b = static_cast<char*>(ws);
  Bufs r;
  r.status = reinterpret_cast<unsigned*>(b + w.status);
  r.cnt_gemv = reinterpret_cast<int*>(b + w.cnt_gemv);
  r.grid_bar = reinterpret_cast<unsigned*>(b + w.grid_bar);
  r.attn_cnt = reinterpret_cast<int*>(b + w.attn_cnt);
  r.attn_part = reinterpret_cast<float*>(b + w.attn_part);
  r.q = reinterpret_cast<float*>(b + w.q);
  r.o = reinterpret_cast<float*>(b + w.o);
  r.x1 = reinterpret_cast<float*>(b + w.x1);
  r.g = reinterpret_cast<float*>(b + w.g);
  r.stats_a = reinterpret_cast<float*>(b + w.stats_a);
  r.stats_b = reinterpret_cast<float*>(b + w.stats_b);
  r.partials = reinterpret_cast<float*>(b + w.partials);
  r.act = b + w.act;
  return r;
}

// Optional per-kernel event pairs (profile mode).
struct EventSink {
  std::vector<cudaEvent_t>* ev = nullptr;  // 2 per launch
  size_t next = 0;
};

cudaError_t record(EventSink* es, cudaStream_t st) {
  if (es == nullptr || es->ev == nullptr) return cudaSuccess;
  if (es->next >= es->ev->size()) return cudaErrorInvalidValue;
  return cudaEventRecord((*es->ev)[es->next++], st);
}

// Enqueues the five region kernels of one layer.
cudaError_t enqueue_layer(const ds_layer& L, const Plans& P, const Bufs& bf, const void* x_in,
                          void* x_out, int B, int T, void* kc, void* vc, int max_len,
                          const int32_t* past_len, const float* stats_in, float* stats_out,
                          int32_t* seq_inc, const ds_layer* next, bool first, cudaStream_t st,
                          bool pdl, EventSink* es) {
  const ds_layer_config& c = L.cfg;
  const int H = c.hidden, F = c.ffn, nh = c.heads, d = H / nh, M = B * T;
  const WKind wk = wkind(c.weight_dtype);
  const ActKind ak = akind(c.act_dtype);
  cudaError_t e;

  RegionArgs base;
  base.M = M;
  base.B = B;
  base.T = T;
  base.partials = bf.partials;
  base.counters = bf.cnt_gemv;
  base.eps = c.ln_eps;
  base.status = bf.status;
  base.H = H;

  // R1: LayerNorm1 + QKV + bias + KV append
  RegionArgs r1 = base;
  r1.W = L.w.w_qkv;
  r1.tmap_w = L.tmap_w(0, P.qkv.nblk);
  r1.tmap_s = L.tmap_s(0, P.qkv.nblk);
  r1.Wscale = static_cast<const __half*>(L.w.s_qkv);
  r1.next_tmap_w = L.tmap_w(1, P.o.nblk);
  r1.next_tmap_s = L.tmap_s(1, P.o.nblk);
  r1.next_plan = P.o;
  r1.qgroup = L.qgroup(0);
  r1.next_qgroup = L.qgroup(1);
  r1.N = 3 * H;
  r1.K = H;
  r1.plan = P.qkv;
  r1.bias = L.w.b_qkv;
  r1.x_act = x_in;
  r1.ln_g = L.w.ln1_g;
  r1.ln_b = L.w.ln1_b;
  r1.stats_in = stats_in;
  r1.out_f32 = bf.q;
  r1.k_cache = kc;
  r1.v_cache = vc;
  r1.heads = nh;
  r1.head_dim = d;
  r1.max_len = max_len;
  r1.past_len = past_len;
  if ((e = record(es, st)) != cudaSuccess) return e;
  // The first kernel of an enqueue waits for everything before it (no
  // programmatic overlap): later kernels may then read past_len early.
  if ((e = launch_region(Region::LnQkv, wk, ak, r1, st, pdl && !first)) != cudaSuccess) return e;
  if ((e = record(es, st)) != cudaSuccess) return e;

  // R2: attention
  AttnArgs ra;
  ra.q = bf.q;
  ra.k_cache = kc;
  ra.v_cache = vc;
  ra.past_len = past_len;
  ra.B = B;
  ra.T = T;
  ra.heads = nh;
  ra.head_dim = d;
  ra.max_len = max_len;
  ra.H = H;
  ra.nsplit = attn_nsplit(B, nh, max_len, L.sms);
  ra.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  ra.stage_keys = attn_stage_keys(d, max_len, ra.nsplit);
  ra.smem = attn_smem_bytes(d, ra.stage_keys);
  ra.out = bf.o;
  ra.status = bf.status;
  if ((e = record(es, st)) != cudaSuccess) return e;
  if ((e = launch_attention(ak, ra, st, pdl)) != cudaSuccess) return e;
  if ((e = record(es, st)) != cudaSuccess) return e;

  // R3: O-proj + bias + residual + LayerNorm2 statistics
  RegionArgs r3 = base;
  r3.W = L.w.w_o;
  r3.tmap_w = L.tmap_w(1, P.o.nblk);
  r3.tmap_s = L.tmap_s(1, P.o.nblk);
  r3.Wscale = static_cast<const __half*>(L.w.s_o);
  r3.next_tmap_w = L.tmap_w(2, P.up.nblk);
  r3.next_tmap_s = L.tmap_s(2, P.up.nblk);
  r3.next_plan = P.up;
  r3.qgroup = L.qgroup(1);
  r3.next_qgroup = L.qgroup(2);
  r3.N = H;
  r3.K = H;
  r3.plan = P.o;
  r3.bias = L.w.b_o;
  r3.x_f32 = bf.o;
  r3.out_f32 = bf.x1;
  r3.resid_act = x_in;
  r3.stats_out = bf.stats_a;
  if ((e = record(es, st)) != cudaSuccess) return e;
  if ((e = launch_region(Region::OprojRes, wk, ak, r3, st, pdl)) != cudaSuccess) return e;
  if ((e = record(es, st)) != cudaSuccess) return e;

  // R4a: LayerNorm2 + FFN-up + bias + GeLU
  RegionArgs r4 = base;
  r4.W = L.w.w_fc1;
  r4.tmap_w = L.tmap_w(2, P.up.nblk);
  r4.tmap_s = L.tmap_s(2, P.up.nblk);
  r4.Wscale = static_cast<const __half*>(L.w.s_fc1);
  r4.next_tmap_w = L.tmap_w(3, P.down.nblk);
  r4.next_tmap_s = L.tmap_s(3, P.down.nblk);
  r4.next_plan = P.down;
  r4.qgroup = L.qgroup(2);
  r4.next_qgroup = L.qgroup(3);
  r4.N = F;
  r4.K = H;
  r4.plan = P.up;
  r4.bias = L.w.b_fc1;
  r4.x_f32 = bf.x1;
  r4.ln_g = L.w.ln2_g;
  r4.ln_b = L.w.ln2_b;
  r4.stats_in = bf.stats_a;
  r4.out_f32 = bf.g;
  if ((e = record(es, st)) != cudaSuccess) return e;
  if ((e = launch_region(Region::FfnUp, wk, ak, r4, st, pdl)) != cudaSuccess) return e;
  if ((e = record(es, st)) != cudaSuccess) return e;

  // R4b: FFN-down + bias + residual (+ next LayerNorm statistics)
  RegionArgs r5 = base;
  r5.W = L.w.w_fc2;
  r5.tmap_w = L.tmap_w(3, P.down.nblk);
  r5.tmap_s = L.tmap_s(3, P.down.nblk);
  r5.Wscale = static_cast<const __half*>(L.w.s_fc2);
  if (next != nullptr) {
    r5.next_tmap_w = next->tmap_w(0, P.qkv.nblk);
    r5.next_tmap_s = next->tmap_s(0, P.qkv.nblk);
    r5.next_plan = P.qkv;
    r5.next_qgroup = next->qgroup(0);
  }
  r5.qgroup = L.qgroup(3);
  r5.N = H;
  r5.K = F;
  r5.plan = P.down;
  r5.bias = L.w.b_fc2;
  r5.x_f32 = bf.g;
  r5.resid_f32 = bf.x1;
  r5.out_act = x_out;
  r5.stats_out = stats_out;
  r5.seq_len_inc = seq_inc;
  if ((e = record(es, st)) != cudaSuccess) return e;
  if ((e = launch_region(Region::FfnDown, wk, ak, r5, st, pdl)) != cudaSuccess) return e;
  if ((e = record(es, st)) != cudaSuccess) return e;
  return cudaSuccess;
}

ds_status check_forward_args(const void* x_in, const void* x_out, int batch, int T, const void* kc,
                             const void* vc, int max_len, const void* len, const void* ws) {
  if (!aligned16(x_in) || !aligned16(x_out))
    return fail(DS_ERR_INVALID_ARG, "x_in / x_out must be non-null and 16-byte aligned");
  if (x_in == x_out) return fail(DS_ERR_INVALID_ARG, "x_out must not alias x_in");
  if (batch < 1 || T < 1 || (long long)batch * T > 64)
    return fail(DS_ERR_UNSUPPORTED, "batch * new_tokens must be in 1..64");
  if (!aligned16(kc) || !aligned16(vc))
    return fail(DS_ERR_INVALID_ARG, "KV caches must be non-null and 16-byte aligned");
  if (max_len < 1 || max_len < T) return fail(DS_ERR_INVALID_ARG, "max_len must be >= new_tokens");
  if (len == nullptr || (reinterpret_cast<uintptr_t>(len) & 3u) != 0)
    return fail(DS_ERR_INVALID_ARG, "past_len / seq_len must be a non-null int32 device array");
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(DS_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  return DS_OK;
}

ds_status check_attn_smem(const ds_layer& L, int T) {
  (void)T;  // tokens are processed one after another: shared memory does not grow with T
  const int d = L.cfg.hidden / L.cfg.heads;
  if (attn_smem_bytes(d, attn_stage_keys(d, 1 << 30, 1)) > (size_t)L.max_smem)
    return fail(DS_ERR_UNSUPPORTED, "attention kernel's shared memory exceeds the device limit");
  return DS_OK;
}

// Encodes the layer's TMA tensor maps on the host and copies them to device
// memory owned by the layer (freed by ds_layer_destroy).
ds_status make_tensor_maps(ds_layer* L) {
  const ds_layer_config& c = L->cfg;
  const int H = c.hidden, F = c.ffn;
  const size_t esz = (c.weight_dtype == DS_I8) ? 1 : 2;
  const void* W[4] = {L->w.w_qkv, L->w.w_o, L->w.w_fc1, L->w.w_fc2};
  const void* Sc[4] = {L->w.s_qkv, L->w.s_o, L->w.s_fc1, L->w.s_fc2};
  const int rows[4] = {3 * H, H, F, H};
  const int cols[4] = {H, H, H, F};
  const bool i8 = (c.weight_dtype == DS_I8);
  const int nmaps = i8 ? 24 : 12;
  std::vector<unsigned char> host((size_t)nmaps * kTensorMapBytes, 0);
  const int blk_k = i8 ? 64 : 32;  // k per 16-byte lane load
  for (int r = 0; r < 4; ++r) {
    // a chunk is 8 warps x nb blocks of blk_k weights (8 nb blk_k esz bytes per row)
    for (int i = 0, nb = 1; i < 3; ++i, nb *= 2) {
      if (cols[r] % (8 * nb * blk_k) != 0) continue;  // no chunk of this width
      if (!encode_weight_map(host.data() + (size_t)(3 * r + i) * kTensorMapBytes, W[r], rows[r],
                             (size_t)cols[r] * esz, (int)(8 * nb * blk_k * esz)))
        return fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight matrix");
      // the scale box (8 nb 64 / group groups) must be 16 bytes or more
      const int grp = L->qgroup(r);
      if (i8 && 8 * nb * 64 / grp >= 8 &&
          !encode_scale_map(host.data() + (size_t)(12 + 3 * r + i) * kTensorMapBytes, Sc[r], rows[r],
                            cols[r] / grp, 8 * nb * 64 / grp))
        return fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for a scale matrix");
    }
  }
  int cur = 0;
  cudaGetDevice(&cur);
  cudaError_t e = cudaSetDevice(L->device);
  if (e == cudaSuccess) e = cudaMalloc(&L->tmaps, host.size());
  if (e == cudaSuccess) e = cudaMemcpy(L->tmaps, host.data(), host.size(), cudaMemcpyHostToDevice);
  cudaSetDevice(cur);
  if (e != cudaSuccess) return cuda_fail(e, "tensor map upload");
  return DS_OK;
}

}  // namespace

struct GraphKey {
  const void* x_in = nullptr;
  void* x_out = nullptr;
  int batch = 0;
  std::vector<void*> kc, vc;
  int max_len = 0;
  int32_t* seq = nullptr;
  void* ws = nullptr;
  bool operator==(const GraphKey& o) const {
    return x_in == o.x_in && x_out == o.x_out && batch == o.batch && kc == o.kc && vc == o.vc &&
           max_len == o.max_len && seq == o.seq && ws == o.ws;
  }
};

struct ds_stack {
  std::vector<ds_layer*> layers;
  bool have_graph = false;
  GraphKey key;
  cudaGraphExec_t exec = nullptr;
  int graph_kernels = 0;
  bool profiling = false;
  std::vector<cudaEvent_t> events;
  double acc_ms[5] = {0, 0, 0, 0, 0};
  int acc_n[5] = {0, 0, 0, 0, 0};
};

extern "C" {

const char* ds_status_string(ds_status s) {
  switch (s) {
    case DS_OK: return "DS_OK";
    case DS_ERR_INVALID_ARG: return "DS_ERR_INVALID_ARG";
    case DS_ERR_UNSUPPORTED: return "DS_ERR_UNSUPPORTED";
    case DS_ERR_CUDA: return "DS_ERR_CUDA";
    case DS_ERR_WORKSPACE: return "DS_ERR_WORKSPACE";
    case DS_ERR_DEVICE: return "DS_ERR_DEVICE";
  }
  return "unknown ds_status";
}

const char* ds_last_error(void) { return g_err.c_str(); }

uint64_t ds_launch_count(void) { return (uint64_t)g_launches.load(); }

ds_status ds_layer_create(const ds_layer_config* cfg, const ds_layer_weights* w, ds_layer** out) {
  if (out == nullptr) return fail(DS_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  ds_status s = validate_config(cfg);
  if (s != DS_OK) return s;
  if (w == nullptr) return fail(DS_ERR_INVALID_ARG, "weights are null");
  const void* ptrs[12] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o,   w->b_o,
                          w->ln2_g, w->ln2_b, w->w_fc1, w->b_fc1, w->w_fc2, w->b_fc2};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(DS_ERR_INVALID_ARG, "weight pointers must be non-null and 16-byte aligned");
  if (cfg->weight_dtype == DS_I8) {
    const void* sp[4] = {w->s_qkv, w->s_o, w->s_fc1, w->s_fc2};
    for (const void* p : sp)
      if (!aligned16(p)) return fail(DS_ERR_INVALID_ARG, "int8 scale pointers must be non-null and 16-byte aligned");
  }
  int dev = 0;
  DevInfo di;
  s = device_info(&dev, &di);
  if (s != DS_OK) return s;
  ds_layer* L = new ds_layer();
  L->cfg = *cfg;
  if (cfg->weight_dtype != DS_I8) {  // the int8 fields are ignored: keep them inert
    L->cfg.quant_group = 64;
    L->cfg.mlp_extra_grouping = 0;
  }
  L->w = *w;
  L->device = dev;
  L->sms = di.sms;
  L->max_smem = di.max_smem;
  L->smem_per_sm = di.smem_per_sm;
  L->ctas_per_sm = ctas_per_sm_knob();
  Plans p;
  if (!make_plans(*L, 1, 1, &p)) {
    delete L;
    return fail(DS_ERR_UNSUPPORTED, "no GEMV work split for this shape");
  }
  s = make_tensor_maps(L);
  if (s != DS_OK) {
    delete L;
    return s;
  }
  *out = L;
  return DS_OK;
}

ds_status ds_layer_destroy(ds_layer* layer) {
  if (layer != nullptr && layer->tmaps != nullptr) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(layer->device);
    cudaFree(layer->tmaps);
    cudaSetDevice(cur);
  }
  delete layer;
  return DS_OK;
}

size_t ds_layer_workspace_bytes(const ds_layer* layer, int batch, int new_tokens) {
  if (layer == nullptr || batch < 1 || new_tokens < 1 || (long long)batch * new_tokens > 64) return 0;
  Plans p;
  if (!make_plans(*layer, batch * new_tokens, batch, &p)) return 0;
  return ws_layout(*layer, batch, new_tokens, p).total;
}

ds_status ds_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (workspace == nullptr || ws_bytes == 0) return fail(DS_ERR_INVALID_ARG, "workspace is null or empty");
  cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
  return DS_OK;
}

ds_status ds_layer_forward(ds_layer* layer, const void* x_in, void* x_out, int batch, int new_tokens,
                           void* k_cache, void* v_cache, int max_len, const int32_t* past_len,
                           void* workspace, size_t ws_bytes, void* stream) {
  if (layer == nullptr) return fail(DS_ERR_INVALID_ARG, "layer is null");
  ds_status s = check_forward_args(x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len,
                                   past_len, workspace);
  if (s != DS_OK) return s;
  if ((s = check_attn_smem(*layer, new_tokens)) != DS_OK) return s;
  Plans p;
  if (!make_plans(*layer, batch * new_tokens, batch, &p))
    return fail(DS_ERR_UNSUPPORTED, "no GEMV work split for this shape");
  const WsLayout wl = ws_layout(*layer, batch, new_tokens, p);
  if (ws_bytes < wl.total) return fail(DS_ERR_WORKSPACE, "workspace smaller than ds_layer_workspace_bytes()");
  const Bufs bf = bufs_of(workspace, wl);
  cudaError_t e = enqueue_layer(*layer, p, bf, x_in, x_out, batch, new_tokens, k_cache, v_cache,
                                max_len, past_len, nullptr, nullptr, nullptr, nullptr, true,
                                static_cast<cudaStream_t>(stream), true, nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "region kernel launch");
  g_launches += 5;
  return DS_OK;
}

}  // extern "C"

namespace ds {
void set_last_error(const char* msg) { g_err = msg; }

// Bytes at the start of a workspace that must be zero before a call (status
// word and arrival counters); 0 for invalid arguments.
size_t layer_workspace_zero_prefix(const ds_layer* layer, int batch, int new_tokens) {
  if (layer == nullptr || batch < 1 || new_tokens < 1 || (long long)batch * new_tokens > 64) return 0;
  Plans p;
  if (!make_plans(*layer, batch * new_tokens, batch, &p)) return 0;
  return ws_layout(*layer, batch, new_tokens, p).q;
}
}  // namespace ds

extern "C" {

ds_status ds_stack_create(ds_layer* const* layers, int n_layers, ds_stack** out) {
  if (out == nullptr) return fail(DS_ERR_INVALID_ARG, "out is null");
  *out = nullptr;
  if (layers == nullptr || n_layers < 1) return fail(DS_ERR_INVALID_ARG, "need at least one layer");
  for (int i = 0; i < n_layers; ++i) {
    if (layers[i] == nullptr) return fail(DS_ERR_INVALID_ARG, "null layer in stack");
    const ds_layer_config& a = layers[0]->cfg;
    const ds_layer_config& b = layers[i]->cfg;
    if (a.hidden != b.hidden || a.heads != b.heads || a.ffn != b.ffn || a.act_dtype != b.act_dtype ||
        a.weight_dtype != b.weight_dtype || a.ln_eps != b.ln_eps || layers[i]->device != layers[0]->device ||
        (a.weight_dtype == DS_I8 &&
         (a.quant_group != b.quant_group || a.mlp_extra_grouping != b.mlp_extra_grouping)))
      return fail(DS_ERR_INVALID_ARG, "all layers of a stack must share one config and device");
  }
  ds_stack* S = new ds_stack();
  S->layers.assign(layers, layers + n_layers);
  *out = S;
  return DS_OK;
}

ds_status ds_stack_destroy(ds_stack* stack) {
  if (stack == nullptr) return DS_OK;
  if (stack->exec != nullptr) cudaGraphExecDestroy(stack->exec);
  for (cudaEvent_t ev : stack->events) cudaEventDestroy(ev);
  delete stack;
  return DS_OK;
}

size_t ds_stack_workspace_bytes(const ds_stack* stack, int batch) {
  if (stack == nullptr) return 0;
  return ds_layer_workspace_bytes(stack->layers[0], batch, 1);
}

namespace {

// Arguments of the persistent step kernel; false when it cannot run this
// configuration (too many layers, no ring geometry, or not co-resident).
bool build_step_args(const ds_stack* S, const Plans& p, const Bufs& bf, const void* x_in, void* x_out, int B,
                     void* const* kc, void* const* vc, int max_len, int32_t* seq, StepArgs* a) {
  const int L = (int)S->layers.size();
  if (!p.step_ok || L > kStepMaxLayers || !step_kernel_knob()) return false;
  const ds_layer& L0 = *S->layers[0];
  const ds_layer_config& c = L0.cfg;
  const WKind wk = wkind(c.weight_dtype);
  const ActKind ak = akind(c.act_dtype);
  a->L = L;
  a->B = B;
  a->H = c.hidden;
  a->F = c.ffn;
  a->heads = c.heads;
  a->head_dim = c.hidden / c.heads;
  a->max_len = max_len;
  a->eps = c.ln_eps;
  for (int i = 0; i < 4; ++i) a->qgroup[i] = L0.qgroup(i);
  a->scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)a->head_dim));
  a->nsplit = step_attn_nsplit(B, c.heads, max_len, L0.sms);
  for (int i = 0; i < 4; ++i) a->plan[i] = p.step[i];
  if (!step_geometry(wk, ak, B, L0.max_smem, a)) return false;
  if (step_blocks_per_sm(wk, ak, a->plan[0].nt, step_smem_bytes(a->plan[0].nt, a->stages, a->SB, a->xs_cap)) < 1)
    return false;
  a->x_in = x_in;
  a->x_out = x_out;
  a->seq = seq;
  a->status = bf.status;
  a->counters = bf.cnt_gemv;
  a->grid_bar = bf.grid_bar;
  a->attn_cnt = bf.attn_cnt;
  a->q = bf.q;
  a->o = bf.o;
  a->x1 = bf.x1;
  a->g = bf.g;
  a->stats_a = bf.stats_a;
  a->stats_b = bf.stats_b;
  a->partials = bf.partials;
  a->attn_part = bf.attn_part;
  a->act = bf.act;
  for (int l = 0; l < L; ++l) {
    const ds_layer_weights& w = S->layers[l]->w;
    StepLayer& y = a->layer[l];
    y.w[0] = w.w_qkv;
    y.w[1] = w.w_o;
    y.w[2] = w.w_fc1;
    y.w[3] = w.w_fc2;
    y.sc[0] = static_cast<const __half*>(w.s_qkv);
    y.sc[1] = static_cast<const __half*>(w.s_o);
    y.sc[2] = static_cast<const __half*>(w.s_fc1);
    y.sc[3] = static_cast<const __half*>(w.s_fc2);
    y.bias[0] = w.b_qkv;
    y.bias[1] = w.b_o;
    y.bias[2] = w.b_fc1;
    y.bias[3] = w.b_fc2;
    y.ln1_g = w.ln1_g;
    y.ln1_b = w.ln1_b;
    y.ln2_g = w.ln2_g;
    y.ln2_b = w.ln2_b;
    y.kc = kc[l];
    y.vc = vc[l];
    for (int r = 0; r < 4; ++r) {
      y.tmap_w[r] = S->layers[l]->tmap_w(r, p.step[r].nblk);
      y.tmap_s[r] = S->layers[l]->tmap_s(r, p.step[r].nblk);
    }
  }
  return true;
}

cudaError_t enqueue_stack(ds_stack* S, const Plans& p, const Bufs& bf, const void* x_in, void* x_out,
                          int B, void* const* kc, void* const* vc, int max_len, int32_t* seq,
                          cudaStream_t st, bool pdl, EventSink* es) {
  const int L = (int)S->layers.size();
  const size_t act_bytes = (size_t)B * S->layers[0]->cfg.hidden * 2;
  for (int l = 0; l < L; ++l) {
    const void* xi = (l == 0) ? x_in : static_cast<const void*>(bf.act + ((l - 1) & 1) * act_bytes);
    void* xo = (l == L - 1) ? x_out : static_cast<void*>(bf.act + (l & 1) * act_bytes);
    const float* sin = (l == 0) ? nullptr : bf.stats_b;
    float* sout = (l == L - 1) ? nullptr : bf.stats_b;
    cudaError_t e = enqueue_layer(*S->layers[l], p, bf, xi, xo, B, 1, kc[l], vc[l], max_len, seq, sin,
                                  sout, (l == L - 1) ? seq : nullptr, (l + 1 < L) ? S->layers[l + 1] : nullptr,
                                  l == 0, st, pdl, es);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

ds_status ds_stack_decode_step(ds_stack* stack, const void* x_in, void* x_out, int batch,
                               void* const* k_caches, void* const* v_caches, int max_len,
                               int32_t* seq_len, void* workspace, size_t ws_bytes, void* stream) {
  if (stack == nullptr) return fail(DS_ERR_INVALID_ARG, "stack is null");
  if (k_caches == nullptr || v_caches == nullptr) return fail(DS_ERR_INVALID_ARG, "cache arrays are null");
  const int L = (int)stack->layers.size();
  for (int l = 0; l < L; ++l) {
    ds_status s = check_forward_args(x_in, x_out, batch, 1, k_caches[l], v_caches[l], max_len,
                                     seq_len, workspace);
    if (s != DS_OK) return s;
  }
  const ds_layer& L0 = *stack->layers[0];
  ds_status s = check_attn_smem(L0, 1);
  if (s != DS_OK) return s;
  Plans p;
  if (!make_plans(L0, batch, batch, &p)) return fail(DS_ERR_UNSUPPORTED, "no GEMV work split for this shape");
  const WsLayout wl = ws_layout(L0, batch, 1, p);
  if (ws_bytes < wl.total) return fail(DS_ERR_WORKSPACE, "workspace smaller than ds_stack_workspace_bytes()");
  const Bufs bf = bufs_of(workspace, wl);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int kernels = 5 * L;

  if (stack->profiling) {
    const size_t need = (size_t)2 * kernels;
    while (stack->events.size() < need) {
      cudaEvent_t ev;
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
      stack->events.push_back(ev);
    }
    EventSink es;
    es.ev = &stack->events;
    cudaError_t e = enqueue_stack(stack, p, bf, x_in, x_out, batch, k_caches, v_caches, max_len,
                                  seq_len, st, false, &es);
    if (e != cudaSuccess) return cuda_fail(e, "region kernel launch (profile)");
    g_launches += kernels;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize (profile)");
    for (int k = 0; k < kernels; ++k) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, stack->events[2 * k], stack->events[2 * k + 1]);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
      stack->acc_ms[k % 5] += ms;
      stack->acc_n[k % 5] += 1;
    }
    return DS_OK;
  }

  // Default path: one persistent, cooperative launch for the whole step;
  // otherwise the chain of region kernels.
  static thread_local StepArgs step_args;  // ~10 KB: kept off the call stack
  const bool use_step = build_step_args(stack, p, bf, x_in, x_out, batch, k_caches, v_caches, max_len,
                                        seq_len, &step_args);
  const WKind swk = wkind(L0.cfg.weight_dtype);
  const ActKind sak = akind(L0.cfg.act_dtype);
  auto enqueue = [&]() -> cudaError_t {
    if (use_step) return launch_step(swk, sak, step_args, L0.sms, st);
    return enqueue_stack(stack, p, bf, x_in, x_out, batch, k_caches, v_caches, max_len, seq_len, st, true,
                         nullptr);
  };
  const int launched = use_step ? 1 : kernels;

  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (st != nullptr) {
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  }
  if (st == nullptr || cs != cudaStreamCaptureStatusNone) {
    cudaError_t e = enqueue();
    if (e != cudaSuccess) return cuda_fail(e, use_step ? "step kernel launch" : "region kernel launch");
    g_launches += launched;
    return DS_OK;
  }

  GraphKey key;
  key.x_in = x_in;
  key.x_out = x_out;
  key.batch = batch;
  key.kc.assign(k_caches, k_caches + L);
  key.vc.assign(v_caches, v_caches + L);
  key.max_len = max_len;
  key.seq = seq_len;
  key.ws = workspace;
  if (!stack->have_graph || !(stack->key == key)) {
    if (stack->exec != nullptr) {
      cudaGraphExecDestroy(stack->exec);
      stack->exec = nullptr;
    }
    stack->have_graph = false;
    cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
    cudaError_t el = enqueue();
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(st, &graph);
    if (el != cudaSuccess) {
      if (graph != nullptr) cudaGraphDestroy(graph);
      return cuda_fail(el, "region kernel launch (capture)");
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(&stack->exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      stack->exec = nullptr;
      return cuda_fail(e, "cudaGraphInstantiate");
    }
    stack->key = key;
    stack->have_graph = true;
    stack->graph_kernels = launched;
  }
  cudaError_t e = cudaGraphLaunch(stack->exec, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  g_launches += stack->graph_kernels;
  return DS_OK;
}

ds_status ds_stack_decode_host(ds_stack* stack, const void* x_host, void* y_host, void* x_dev_in,
                               void* x_dev_out, int batch, void* const* k_caches,
                               void* const* v_caches, int max_len, int32_t* seq_len,
                               void* workspace, size_t ws_bytes, void* stream) {
  if (stack == nullptr) return fail(DS_ERR_INVALID_ARG, "stack is null");
  if (x_host == nullptr || y_host == nullptr) return fail(DS_ERR_INVALID_ARG, "host buffers are null");
  if (batch < 1 || batch > 64) return fail(DS_ERR_UNSUPPORTED, "batch must be in 1..64");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)batch * stack->layers[0]->cfg.hidden * 2;
  cudaError_t e = cudaMemcpyAsync(x_dev_in, x_host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(host to device)");
  ds_status s = ds_stack_decode_step(stack, x_dev_in, x_dev_out, batch, k_caches, v_caches, max_len,
                                     seq_len, workspace, ws_bytes, stream);
  if (s != DS_OK) return s;
  e = cudaMemcpyAsync(y_host, x_dev_out, bytes, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(device to host)");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  return DS_OK;
}

ds_status ds_stack_set_profiling(ds_stack* stack, int enabled) {
  if (stack == nullptr) return fail(DS_ERR_INVALID_ARG, "stack is null");
  stack->profiling = (enabled != 0);
  return DS_OK;
}

ds_status ds_stack_region_times(ds_stack* stack, float us_out[5], int launches_out[5]) {
  if (stack == nullptr || us_out == nullptr) return fail(DS_ERR_INVALID_ARG, "null argument");
  for (int i = 0; i < 5; ++i) {
    us_out[i] = stack->acc_n[i] ? (float)(1000.0 * stack->acc_ms[i] / stack->acc_n[i]) : 0.f;
    if (launches_out != nullptr) launches_out[i] = stack->acc_n[i];
    stack->acc_ms[i] = 0.0;
    stack->acc_n[i] = 0;
  }
  return DS_OK;
}

ds_status ds_quantize_int8(const void* w_f16, int n, int k, int group, int8_t* codes, void* scales_f16,
                           void* stream) {
  if (w_f16 == nullptr || codes == nullptr || scales_f16 == nullptr)
    return fail(DS_ERR_INVALID_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(w_f16) & 3u) != 0 || (reinterpret_cast<uintptr_t>(codes) & 1u) != 0 ||
      (reinterpret_cast<uintptr_t>(scales_f16) & 1u) != 0)
    return fail(DS_ERR_INVALID_ARG, "misaligned pointer");
  if (group != 32 && group != 64 && group != 128) return fail(DS_ERR_UNSUPPORTED, "group must be 32, 64 or 128");
  if ((reinterpret_cast<uintptr_t>(w_f16) & (size_t)(group / 16 - 1)) != 0 ||
      (reinterpret_cast<uintptr_t>(codes) & (size_t)(group / 32 - 1)) != 0)
    return fail(DS_ERR_INVALID_ARG, "misaligned pointer for this group length");
  if (n < 1 || k < group || k % group != 0)
    return fail(DS_ERR_INVALID_ARG, "n >= 1 and k a positive multiple of group required");
  cudaError_t e = launch_quantize_int8(w_f16, n, k, group, codes, scales_f16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize_int8 launch");
  g_launches += 1;
  return DS_OK;
}

ds_status ds_workspace_status(void* workspace, uint32_t* flags_out, void* stream) {
  if (workspace == nullptr || flags_out == nullptr) return fail(DS_ERR_INVALID_ARG, "null argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status word");
  if (v != 0) {
    e = cudaMemsetAsync(workspace, 0, sizeof(v), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace status word");
  }
  *flags_out = v;
  if (v != 0) return fail(DS_ERR_DEVICE, "device-side check failed (see flags)");
  return DS_OK;
}

}  // extern "C"
