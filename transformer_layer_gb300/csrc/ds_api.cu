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
// Two GEMM paths serve the regions (§3 intro: the skinny GEMM at small batch):
//  * up to 8 rows (B * T), and for int8 weights up to 64, the streaming GEMV
//    kernels (gemv_impl.cuh) with the LayerNorm fused into their prologue;
//  * from 8 rows (fp16 / bf16 weights, or int8 with fp16 activations), the tensor-core tile kernels
//    (dense_impl.cuh, tcgen05 + TMEM), each LayerNorm run by a small row
//    normalisation kernel that writes the tensor-core operand.
//
// Host-side responsibilities here: argument validation before any launch,
// workspace layout, the work splits, the launch chain with programmatic
// dependent launch, CUDA-graph capture/replay of a stack step, and per-region
// event timing in profile mode.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
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

constexpr int kGemvMaxRows = 64;   // streaming GEMV kernels: up to 8 MMA column tiles
constexpr int kTileMinRows = 8;    // tensor-core tiles from 8 rows (streaming kernels below)
constexpr int kTileMaxRows = 4096; // rows (B * T) of one tile-path call

struct DevInfo {
  bool ready = false;
  int sms = 0;
  int max_smem = 0;  // opt-in shared memory of one block
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
    e = prepare_region_kernels(d.max_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(region kernels)");
    e = prepare_dense_kernels(d.max_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(tile kernels)");
    e = prepare_attention_kernels(d.max_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attention kernel)");
    e = prepare_attention_prefill_kernels(d.max_smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prompt attention kernel)");
    d.ready = true;
  }
  *dev_out = dev;
  *out = d;
  return DS_OK;
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
  // TMA tensor maps in device memory, kTensorMapBytes each: weights of QKV,
  // O-proj, FFN-up, FFN-down for the GEMV path, one map per k-blocks-per-step
  // choice (1, 2, 4: a map's box is one chunk); then (int8) their scales in
  // the same order; then the tile maps of the four matrices: fp16 / bf16 for
  // ring stages of 64 and of 128 along K, int8 the scales' and the codes'.
  unsigned char* tmaps = nullptr;
  static int nblk_index(int nblk) { return nblk == 4 ? 2 : (nblk == 2 ? 1 : 0); }
  const void* tmap_w(int r, int nblk) const { return tmaps + (size_t)(3 * r + nblk_index(nblk)) * kTensorMapBytes; }
  const void* tmap_s(int r, int nblk) const {
    return cfg.weight_dtype == DS_I8 ? tmaps + (size_t)(12 + 3 * r + nblk_index(nblk)) * kTensorMapBytes : nullptr;
  }
  const void* tmap_tile(int r, int kc) const {
    return tmaps + (size_t)(24 + 2 * r + (kc == 128 ? 1 : 0)) * kTensorMapBytes;
  }
  // int8 tiles (stages of 128 codes): the scales' map, in the unused slot of stages of 64
  const void* tmap_tile_s(int r) const {
    return cfg.weight_dtype == DS_I8 ? tmaps + (size_t)(24 + 2 * r) * kTensorMapBytes : nullptr;
  }
  // int8 scale group length of matrix r (0 QKV, 1 O-proj, 2 FFN-up, 3 FFN-down):
  // the FFN matrices take half the length under mlp_extra_grouping.
  int qgroup(int r) const { return (r >= 2 && cfg.mlp_extra_grouping == 1) ? cfg.quant_group / 2 : cfg.quant_group; }
  // tensor-core tiles: fp16 / bf16 weights, and int8 codes with fp16 activations
  bool tile_capable() const { return cfg.weight_dtype != DS_I8 || cfg.act_dtype == DS_F16; }
  int max_rows() const { return tile_capable() ? kTileMaxRows : kGemvMaxRows; }
};

namespace {

struct Plans {
  bool tile = false;          // tensor-core tile path
  GemvPlan qkv, o, up, down;  // streaming GEMV path
  DensePlan tq, to, tu, td;   // tile path
};

bool use_tile_path(const ds_layer& L, int M) { return L.tile_capable() && M >= kTileMinRows; }

bool make_plans(const ds_layer& L, int M, Plans* p) {
  const int H = L.cfg.hidden, F = L.cfg.ffn;
  const WKind wk = wkind(L.cfg.weight_dtype);
  const ActKind ak = akind(L.cfg.act_dtype);
  if (M < 1 || M > L.max_rows()) return false;
  p->tile = use_tile_path(L, M);
  if (p->tile) {
    const bool i8 = wk == WKind::I8;
    return dense_make_plan(ak, 3 * H, H, M, L.sms, L.max_smem, &p->tq, i8) &&
           dense_make_plan(ak, H, H, M, L.sms, L.max_smem, &p->to, i8) &&
           dense_make_plan(ak, F, H, M, L.sms, L.max_smem, &p->tu, i8) &&
           dense_make_plan(ak, H, F, M, L.sms, L.max_smem, &p->td, i8);
  }
  if (!gemv_make_plan(wk, ak, 3 * H, H, M, L.sms, L.max_smem, &p->qkv)) return false;
  if (!gemv_make_plan(wk, ak, H, H, M, L.sms, L.max_smem, &p->o)) return false;
  if (!gemv_make_plan(wk, ak, F, H, M, L.sms, L.max_smem, &p->up)) return false;
  if (!gemv_make_plan(wk, ak, H, F, M, L.sms, L.max_smem, &p->down)) return false;
  if (wk == WKind::I8) {  // the scale box of a chunk must hold at least 8 groups
    const GemvPlan* pl[4] = {&p->qkv, &p->o, &p->up, &p->down};
    for (int i = 0; i < 4; ++i)
      if (pl[i]->chunk_k / L.qgroup(i) < 8) return false;
  }
  return true;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
  size_t status, cnt, q, o, x1, g, stats_a, stats_b, partials, op_a_hi, op_a_lo, op_b_hi, op_b_lo, act, total;
};

// Workspace regions, each 256-byte aligned.  The status word and the arrival
// counters come first so that a zero-fill of the first bytes resets them.
WsLayout ws_layout(const ds_layer& L, int B, int T, const Plans& p) {
  const int H = L.cfg.hidden, F = L.cfg.ffn;
  const size_t M = (size_t)B * T;
  const bool split = L.cfg.act_dtype == DS_BF16;
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up256(bytes);
    return o;
  };
  w.status = take(256);
  size_t tiles = (size_t)std::max(3 * H, F) / 16;
  if (p.tile) {
    const DensePlan* d[4] = {&p.tq, &p.to, &p.tu, &p.td};
    tiles = 0;
    for (const DensePlan* x : d) tiles = std::max(tiles, (size_t)x->ws.tiles);
  }
  w.cnt = take(tiles * sizeof(int));
  w.q = take(M * H * 4);
  w.x1 = take(M * H * 4);
  w.stats_a = take((size_t)(H / 16) * M * 2 * 4);
  w.stats_b = take((size_t)(H / 16) * M * 2 * 4);
  size_t part = 0;
  if (p.tile) {
    w.o = w.g = 0;
    const DensePlan* d[4] = {&p.tq, &p.to, &p.tu, &p.td};
    for (const DensePlan* x : d) {  // all tiles when K is sliced, else only the leftover tiles (u >= U_dp)
      const size_t ptiles = x->ws.KS > 1 ? (size_t)x->ws.tiles : (size_t)(x->ws.units - x->ws.U_dp);
      part = std::max(part, ptiles * x->ws.KS * x->ws.maxc * x->ntok * 128 * 4);
    }
    w.partials = take(part);
    w.op_a_hi = take(M * H * 2);
    w.op_a_lo = split ? take(M * H * 2) : 0;
    w.op_b_hi = take(M * std::max(H, F) * 2);
    w.op_b_lo = split ? take(M * std::max(H, F) * 2) : 0;
  } else {
    w.o = take(M * H * 4);
    w.g = take(M * F * 4);
    const GemvPlan* ps[4] = {&p.qkv, &p.o, &p.up, &p.down};
    for (const GemvPlan* g : ps) part = std::max(part, (size_t)g->tiles * g->KS * g->maxc * 16 * M * 4);
    w.partials = take(part);
    w.op_a_hi = w.op_a_lo = w.op_b_hi = w.op_b_lo = 0;
  }
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
  int* cnt;
  float *q, *o, *x1, *g, *stats_a, *stats_b, *partials;
  void *op_a_hi, *op_a_lo, *op_b_hi, *op_b_lo;
  char* act;
};

Bufs bufs_of(void* ws, const WsLayout& w) {
  char* b = static_cast<char*>(ws);
  auto at = [&](size_t off) -> void* { return off ? static_cast<void*>(b + off) : nullptr; };
  Bufs r;
  r.status = reinterpret_cast<unsigned*>(b + w.status);
  r.cnt = reinterpret_cast<int*>(b + w.cnt);
  r.q = static_cast<float*>(at(w.q));
  r.o = static_cast<float*>(at(w.o));
  r.x1 = static_cast<float*>(at(w.x1));
  r.g = static_cast<float*>(at(w.g));
  r.stats_a = static_cast<float*>(at(w.stats_a));
  r.stats_b = static_cast<float*>(at(w.stats_b));
  r.partials = static_cast<float*>(at(w.partials));
  r.op_a_hi = at(w.op_a_hi);
  r.op_a_lo = at(w.op_a_lo);
  r.op_b_hi = at(w.op_b_hi);
  r.op_b_lo = at(w.op_b_lo);
  r.act = b + w.act;
  return r;
}

// Tensor maps of the tile path's activation operands for one workspace and
// row count: op_a with K = H, op_b with K = H (attention output) and K = F
// (GeLU output); hi and (bf16) lo parts.
struct alignas(64) XMaps {
  unsigned char aq_hi[kTensorMapBytes], aq_lo[kTensorMapBytes];  // LN1 output, read by QKV
  unsigned char au_hi[kTensorMapBytes], au_lo[kTensorMapBytes];  // LN2 output, read by FFN-up
  unsigned char bh_hi[kTensorMapBytes], bh_lo[kTensorMapBytes];  // attention output, read by O-proj
  unsigned char bf_hi[kTensorMapBytes], bf_lo[kTensorMapBytes];  // GeLU output, read by FFN-down
};

// Each map's box is its reader's token tile and ring stage (the four plans
// may differ: a prompt chunk's QKV can take 128-row tiles where the others
// take 256).
bool make_xmaps(const ds_layer& L, const Plans& p, const Bufs& bf, int M, XMaps* x) {
  const int H = L.cfg.hidden, F = L.cfg.ffn;
  const bool split = L.cfg.act_dtype == DS_BF16;
  std::memset(x, 0, sizeof(*x));
  bool ok = encode_tile_map(x->aq_hi, bf.op_a_hi, M, H, p.tq.ntok, p.tq.kc) &&
            encode_tile_map(x->au_hi, bf.op_a_hi, M, H, p.tu.ntok, p.tu.kc) &&
            encode_tile_map(x->bh_hi, bf.op_b_hi, M, H, p.to.ntok, p.to.kc) &&
            encode_tile_map(x->bf_hi, bf.op_b_hi, M, F, p.td.ntok, p.td.kc);
  if (ok && split)
    ok = encode_tile_map(x->aq_lo, bf.op_a_lo, M, H, p.tq.ntok, p.tq.kc) &&
         encode_tile_map(x->au_lo, bf.op_a_lo, M, H, p.tu.ntok, p.tu.kc) &&
         encode_tile_map(x->bh_lo, bf.op_b_lo, M, H, p.to.ntok, p.to.kc) &&
         encode_tile_map(x->bf_lo, bf.op_b_lo, M, F, p.td.ntok, p.td.kc);
  return ok;
}

// Optional per-kernel event pairs (profile mode).
struct EventSink {
  std::vector<cudaEvent_t>* ev = nullptr;  // 2 per region
  size_t next = 0;
};

cudaError_t record(EventSink* es, cudaStream_t st) {
  if (es == nullptr || es->ev == nullptr) return cudaSuccess;
  if (es->next >= es->ev->size()) return cudaErrorInvalidValue;
  return cudaEventRecord((*es->ev)[es->next++], st);
}

// A captured kernel node whose arguments hold the caller's x_in or x_out: the
// graph is kept for these pointers being replaced in place (no re-capture).
struct PatchNode {
  cudaGraphNode_t node = nullptr;
  int arg_index = 0;                 // which kernel parameter is the argument struct
  std::vector<unsigned char> args;   // its bytes as captured
  std::vector<size_t> in_offsets;    // offsets of x_in pointers inside it
  std::vector<size_t> out_offsets;   // offsets of x_out pointers
};

// During stream capture: records the node just added to the capture.
template <typename A>
cudaError_t record_patch(std::vector<PatchNode>* rec, cudaStream_t st, int arg_index, const A& args,
                         std::vector<size_t> in_off, std::vector<size_t> out_off) {
  if (rec == nullptr || (in_off.empty() && out_off.empty())) return cudaSuccess;
  cudaStreamCaptureStatus cs;
  const cudaGraphNode_t* deps = nullptr;
  size_t nd = 0;
  cudaError_t e = cudaStreamGetCaptureInfo(st, &cs, nullptr, nullptr, &deps, nullptr, &nd);
  if (e != cudaSuccess) return e;
  if (cs != cudaStreamCaptureStatusActive || nd != 1) return cudaErrorStreamCaptureUnsupported;
  PatchNode p;
  p.node = deps[0];
  p.arg_index = arg_index;
  p.args.resize(sizeof(A));
  std::memcpy(p.args.data(), &args, sizeof(A));
  p.in_offsets = std::move(in_off);
  p.out_offsets = std::move(out_off);
  rec->push_back(std::move(p));
  return cudaSuccess;
}

struct LayerIO {
  const void* x_in;
  void* x_out;
  bool in_is_caller;   // x_in is the caller's buffer (record for patching)
  bool out_is_caller;  // x_out is the caller's buffer
};

// Enqueues the region kernels of one layer.
cudaError_t enqueue_layer(const ds_layer& L, const Plans& P, const Bufs& bf, const XMaps* xm, const LayerIO& io,
                          int B, int T, void* kc, void* vc, int max_len, const int32_t* past_len,
                          const float* stats_in, float* stats_out, int32_t* seq_inc, const ds_layer* next,
                          bool first, cudaStream_t st, bool pdl, EventSink* es, std::vector<PatchNode>* rec) {
  const ds_layer_config& c = L.cfg;
  const int H = c.hidden, F = c.ffn, nh = c.heads, d = H / nh, M = B * T;
  const WKind wk = wkind(c.weight_dtype);
  const ActKind ak = akind(c.act_dtype);
  const bool split = ak == ActKind::BF16;
  cudaError_t e;
  auto in_if = [&](size_t off) { return io.in_is_caller ? std::vector<size_t>{off} : std::vector<size_t>{}; };
  auto out_if = [&](size_t off) { return io.out_is_caller ? std::vector<size_t>{off} : std::vector<size_t>{}; };

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
  ra.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  attn_configure(ra, akind(L.cfg.act_dtype), L.sms, L.max_smem);
  ra.status = bf.status;
  // prompt chunks: tiled flash attention; decode and short chunks: split-KV
  auto launch_attn = [&](const AttnArgs& x) {
    return T >= kPrefillMinTokens ? launch_attention_prefill(ak, x, st, pdl) : launch_attention(ak, x, st, pdl);
  };

  if (P.tile) {
    // (no L2 prefetch of the next GEMM's weights on this path: the tile
    // kernels end with split-K fix-ups whose L2 traffic it would delay; each
    // tile CTA requests its own first weight chunks before its dependency wait)
    DenseArgs base;
    base.M = M;
    base.B = B;
    base.T = T;
    base.partials = bf.partials;
    base.counters = bf.cnt;
    base.status = bf.status;
    base.H = H;
    // R1: LayerNorm1 (row kernel) + QKV + bias + KV append
    LnPrepArgs p1;
    p1.M = M;
    p1.K = H;
    p1.eps = c.ln_eps;
    p1.x_act = io.x_in;
    p1.stats_in = stats_in;
    p1.ln_g = L.w.ln1_g;
    p1.ln_b = L.w.ln1_b;
    p1.out_hi = bf.op_a_hi;
    p1.out_lo = bf.op_a_lo;
    if ((e = record(es, st)) != cudaSuccess) return e;
    // The first kernel of an enqueue waits for everything before it (no
    // programmatic overlap): later kernels may then read past_len early.
    if ((e = launch_ln_prep(ak, p1, st, pdl && !first)) != cudaSuccess) return e;
    if ((e = record_patch(rec, st, 0, p1, in_if(offsetof(LnPrepArgs, x_act)), {})) != cudaSuccess) return e;
    DenseArgs r1 = base;
    r1.tmap_w = L.tmap_tile(0, P.tq.kc);
    r1.tmap_s = L.tmap_tile_s(0);
    r1.qgroup = L.qgroup(0);
    r1.N = 3 * H;
    r1.K = H;
    r1.plan = P.tq;
    r1.bias = L.w.b_qkv;
    r1.out_f32 = bf.q;
    r1.k_cache = kc;
    r1.v_cache = vc;
    r1.heads = nh;
    r1.head_dim = d;
    r1.max_len = max_len;
    r1.past_len = past_len;
    if ((e = launch_dense(Region::LnQkv, ak, r1, xm->aq_hi, split ? xm->aq_lo : nullptr, st, pdl)) != cudaSuccess)
      return e;
    if ((e = record(es, st)) != cudaSuccess) return e;
    // R2: attention, output in the operand format
    ra.out_hi = bf.op_b_hi;
    ra.out_lo = bf.op_b_lo;
    if ((e = record(es, st)) != cudaSuccess) return e;
    if ((e = launch_attn(ra)) != cudaSuccess) return e;
    if ((e = record(es, st)) != cudaSuccess) return e;
    // R3: O-proj + bias + residual + LayerNorm2 statistics
    DenseArgs r3 = base;
    r3.tmap_w = L.tmap_tile(1, P.to.kc);
    r3.tmap_s = L.tmap_tile_s(1);
    r3.qgroup = L.qgroup(1);
    r3.N = H;
    r3.K = H;
    r3.plan = P.to;
    r3.bias = L.w.b_o;
    r3.resid_act = io.x_in;
    r3.out_f32 = bf.x1;
    r3.stats_out = bf.stats_a;
    if ((e = record(es, st)) != cudaSuccess) return e;
    if ((e = launch_dense(Region::OprojRes, ak, r3, xm->bh_hi, split ? xm->bh_lo : nullptr, st, pdl)) != cudaSuccess)
      return e;
    if ((e = record_patch(rec, st, 2, r3, in_if(offsetof(DenseArgs, resid_act)), {})) != cudaSuccess) return e;
    if ((e = record(es, st)) != cudaSuccess) return e;
    // R4a: LayerNorm2 (row kernel) + FFN-up + bias + GeLU
    LnPrepArgs p2;
    p2.M = M;
    p2.K = H;
    p2.eps = c.ln_eps;
    p2.x_f32 = bf.x1;
    p2.stats_in = bf.stats_a;
    p2.ln_g = L.w.ln2_g;
    p2.ln_b = L.w.ln2_b;
    p2.out_hi = bf.op_a_hi;
    p2.out_lo = bf.op_a_lo;
    if ((e = record(es, st)) != cudaSuccess) return e;
    if ((e = launch_ln_prep(ak, p2, st, pdl)) != cudaSuccess) return e;
    DenseArgs r4 = base;
    r4.tmap_w = L.tmap_tile(2, P.tu.kc);
    r4.tmap_s = L.tmap_tile_s(2);
    r4.qgroup = L.qgroup(2);
    r4.N = F;
    r4.K = H;
    r4.plan = P.tu;
    r4.bias = L.w.b_fc1;
    r4.out_act = bf.op_b_hi;
    r4.out_lo = bf.op_b_lo;
    if ((e = launch_dense(Region::FfnUp, ak, r4, xm->au_hi, split ? xm->au_lo : nullptr, st, pdl)) != cudaSuccess)
      return e;
    if ((e = record(es, st)) != cudaSuccess) return e;
    // R4b: FFN-down + bias + residual (+ next LayerNorm statistics)
    DenseArgs r5 = base;
    r5.tmap_w = L.tmap_tile(3, P.td.kc);
    r5.tmap_s = L.tmap_tile_s(3);
    r5.qgroup = L.qgroup(3);
    r5.N = H;
    r5.K = F;
    r5.plan = P.td;
    r5.bias = L.w.b_fc2;
    r5.resid_f32 = bf.x1;
    r5.out_act = io.x_out;
    r5.stats_out = stats_out;
    r5.seq_len_inc = seq_inc;
    if ((e = record(es, st)) != cudaSuccess) return e;
    if ((e = launch_dense(Region::FfnDown, ak, r5, xm->bf_hi, split ? xm->bf_lo : nullptr, st, pdl)) != cudaSuccess)
      return e;
    if ((e = record_patch(rec, st, 2, r5, {}, out_if(offsetof(DenseArgs, out_act)))) != cudaSuccess) return e;
    return record(es, st);
  }

  RegionArgs base;
  base.M = M;
  base.B = B;
  base.T = T;
  base.partials = bf.partials;
  base.counters = bf.cnt;
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
  r1.x_act = io.x_in;
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
  if ((e = record_patch(rec, st, 0, r1, in_if(offsetof(RegionArgs, x_act)), {})) != cudaSuccess) return e;
  if ((e = record(es, st)) != cudaSuccess) return e;

  // R2: attention
  ra.out = bf.o;
  if ((e = record(es, st)) != cudaSuccess) return e;
  if ((e = launch_attn(ra)) != cudaSuccess) return e;
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
  r3.resid_act = io.x_in;
  r3.stats_out = bf.stats_a;
  if ((e = record(es, st)) != cudaSuccess) return e;
  if ((e = launch_region(Region::OprojRes, wk, ak, r3, st, pdl)) != cudaSuccess) return e;
  if ((e = record_patch(rec, st, 0, r3, in_if(offsetof(RegionArgs, resid_act)), {})) != cudaSuccess) return e;
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
  r5.out_act = io.x_out;
  r5.stats_out = stats_out;
  r5.seq_len_inc = seq_inc;
  if ((e = record(es, st)) != cudaSuccess) return e;
  if ((e = launch_region(Region::FfnDown, wk, ak, r5, st, pdl)) != cudaSuccess) return e;
  if ((e = record_patch(rec, st, 0, r5, {}, out_if(offsetof(RegionArgs, out_act)))) != cudaSuccess) return e;
  return record(es, st);
}

int kernels_per_layer(const Plans& p) { return p.tile ? 7 : 5; }

ds_status check_forward_args(const ds_layer& L, const void* x_in, const void* x_out, int batch, int T, const void* kc,
                             const void* vc, int max_len, const void* len, const void* ws) {
  if (!aligned16(x_in) || !aligned16(x_out))
    return fail(DS_ERR_INVALID_ARG, "x_in / x_out must be non-null and 16-byte aligned");
  if (x_in == x_out) return fail(DS_ERR_INVALID_ARG, "x_out must not alias x_in");
  if (batch < 1 || T < 1 || (long long)batch * T > L.max_rows())
    return fail(DS_ERR_UNSUPPORTED, L.tile_capable() ? "batch * new_tokens must be in 1..4096"
                                                     : "batch * new_tokens must be in 1..64 for int8 weights with "
                                                       "bf16 activations");
  if (!aligned16(kc) || !aligned16(vc))
    return fail(DS_ERR_INVALID_ARG, "KV caches must be non-null and 16-byte aligned");
  if (max_len < 1 || max_len < T) return fail(DS_ERR_INVALID_ARG, "max_len must be >= new_tokens");
  if (len == nullptr || (reinterpret_cast<uintptr_t>(len) & 3u) != 0)
    return fail(DS_ERR_INVALID_ARG, "past_len / seq_len must be a non-null int32 device array");
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(DS_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  return DS_OK;
}

// The library's kernels run on the device a layer was created on, with that
// device current: its weights and tensor maps live there.
ds_status check_device(const ds_layer& L) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != L.device) return fail(DS_ERR_INVALID_ARG, "the current device is not the device the layer was created on");
  return DS_OK;
}

ds_status check_attn_smem(const ds_layer& L) {
  const int d = L.cfg.hidden / L.cfg.heads;
  if (attn_smem_bytes(d, 0) + 1024 > (size_t)L.max_smem ||
      attn_prefill_smem_bytes(akind(L.cfg.act_dtype), d) > (size_t)L.max_smem)
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
  const int nmaps = 32;
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
    if (L->tile_capable()) {
      // fp16 / bf16: ring stages of 64 and 128 along K; int8: the codes (as
      // pairs of 16-bit elements) in stages of 128, then their scales in boxes
      // of 8 groups x 128 rows
      for (int j = 0; j < 2; ++j) {
        unsigned char* m = host.data() + (size_t)(24 + 2 * r + j) * kTensorMapBytes;
        const bool ok = i8 ? (j ? encode_tile_map(m, W[r], rows[r], cols[r] / 2, 128, 64)
                                : encode_scale_map(m, Sc[r], rows[r], cols[r] / L->qgroup(r), 8, 128))
                           : encode_tile_map(m, W[r], rows[r], cols[r], 128, j ? 128 : 64);
        if (!ok) return fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight tile map");
      }
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
  int batch = 0;
  std::vector<void*> kc, vc;
  int max_len = 0;
  int32_t* seq = nullptr;
  void* ws = nullptr;
  bool operator==(const GraphKey& o) const {
    return batch == o.batch && kc == o.kc && vc == o.vc && max_len == o.max_len && seq == o.seq && ws == o.ws;
  }
};

struct ds_stack {
  std::vector<ds_layer*> layers;
  bool have_graph = false;
  GraphKey key;
  cudaGraph_t graph = nullptr;   // kept alive for in-place updates of its kernel nodes
  cudaGraphExec_t exec = nullptr;
  std::vector<PatchNode> patch;  // nodes holding x_in / x_out
  const void* x_in = nullptr;    // the pointers the executable graph currently uses
  void* x_out = nullptr;
  int graph_kernels = 0;
  unsigned long long captures = 0;  // graph captures since creation
  bool profiling = false;
  std::vector<cudaEvent_t> events;
  double acc_ms[5] = {0, 0, 0, 0, 0};
  int acc_n[5] = {0, 0, 0, 0, 0};
};

namespace ds {
void set_last_error(const char* msg) { g_err = msg; }
int layer_device(const ds_layer* layer) { return layer->device; }
void add_launches(unsigned long long n) { g_launches += n; }

// Validates a ds_layer_forward call (nothing is enqueued).  On success
// *zero_prefix is the number of leading workspace bytes (status word and
// counters) that must be zero before the call.
ds_status layer_forward_check(const ds_layer* layer, const void* x_in, const void* x_out, int batch, int new_tokens,
                              const void* k_cache, const void* v_cache, int max_len, const int32_t* past_len,
                              const void* workspace, size_t ws_bytes, size_t* zero_prefix) {
  if (layer == nullptr) return fail(DS_ERR_INVALID_ARG, "layer is null");
  ds_status s = check_forward_args(*layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len,
                                   workspace);
  if (s != DS_OK) return s;
  if ((s = check_device(*layer)) != DS_OK) return s;
  if ((s = check_attn_smem(*layer)) != DS_OK) return s;
  Plans p;
  if (!make_plans(*layer, batch * new_tokens, &p)) return fail(DS_ERR_UNSUPPORTED, "no GEMM work split for this shape");
  const WsLayout wl = ws_layout(*layer, batch, new_tokens, p);
  if (ws_bytes < wl.total) return fail(DS_ERR_WORKSPACE, "workspace smaller than ds_layer_workspace_bytes()");
  if (zero_prefix != nullptr) *zero_prefix = wl.q;
  return DS_OK;
}

// Enqueues a ds_layer_forward call that layer_forward_check accepted.
ds_status layer_forward_enqueue(ds_layer* layer, const void* x_in, void* x_out, int batch, int new_tokens,
                                void* k_cache, void* v_cache, int max_len, const int32_t* past_len, void* workspace,
                                void* stream) {
  Plans p;
  make_plans(*layer, batch * new_tokens, &p);
  const WsLayout wl = ws_layout(*layer, batch, new_tokens, p);
  const Bufs bf = bufs_of(workspace, wl);
  XMaps xm;
  if (p.tile && !make_xmaps(*layer, p, bf, batch * new_tokens, &xm))
    return fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation operand");
  const LayerIO io{x_in, x_out, false, false};
  cudaError_t e = enqueue_layer(*layer, p, bf, &xm, io, batch, new_tokens, k_cache, v_cache, max_len, past_len,
                                nullptr, nullptr, nullptr, nullptr, true, static_cast<cudaStream_t>(stream), true,
                                nullptr, nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "region kernel launch");
  g_launches += kernels_per_layer(p);
  return DS_OK;
}
}  // namespace ds

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
  Plans p;
  if (!make_plans(*L, 1, &p)) {
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
  if (layer == nullptr || batch < 1 || new_tokens < 1 || (long long)batch * new_tokens > layer->max_rows()) return 0;
  Plans p;
  if (!make_plans(*layer, batch * new_tokens, &p)) return 0;
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
  ds_status s = layer_forward_check(layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len,
                                    workspace, ws_bytes, nullptr);
  if (s != DS_OK) return s;
  return layer_forward_enqueue(layer, x_in, x_out, batch, new_tokens, k_cache, v_cache, max_len, past_len, workspace,
                               stream);
}

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

}  // extern "C"

namespace {

void drop_graph(ds_stack* S) {
  if (S->exec != nullptr) cudaGraphExecDestroy(S->exec);
  if (S->graph != nullptr) cudaGraphDestroy(S->graph);
  S->exec = nullptr;
  S->graph = nullptr;
  S->patch.clear();
  S->have_graph = false;
}

cudaError_t enqueue_stack(ds_stack* S, const Plans& p, const Bufs& bf, const XMaps* xm, const void* x_in, void* x_out,
                          int B, void* const* kc, void* const* vc, int max_len, int32_t* seq, cudaStream_t st,
                          bool pdl, EventSink* es, std::vector<PatchNode>* rec, int T = 1, bool advance = true) {
  const int L = (int)S->layers.size();
  const size_t act_bytes = (size_t)B * T * S->layers[0]->cfg.hidden * 2;
  for (int l = 0; l < L; ++l) {
    LayerIO io;
    io.x_in = (l == 0) ? x_in : static_cast<const void*>(bf.act + ((l - 1) & 1) * act_bytes);
    io.x_out = (l == L - 1) ? x_out : static_cast<void*>(bf.act + (l & 1) * act_bytes);
    io.in_is_caller = (l == 0);
    io.out_is_caller = (l == L - 1);
    const float* sin = (l == 0) ? nullptr : bf.stats_b;
    float* sout = (l == L - 1) ? nullptr : bf.stats_b;
    cudaError_t e = enqueue_layer(*S->layers[l], p, bf, xm, io, B, T, kc[l], vc[l], max_len, seq, sin, sout,
                                  (l == L - 1 && advance) ? seq : nullptr, (l + 1 < L) ? S->layers[l + 1] : nullptr,
                                  l == 0, st, pdl, es, rec);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Replaces the captured x_in / x_out pointers in the executable graph.
cudaError_t patch_graph(ds_stack* S, const void* x_in, void* x_out) {
  for (PatchNode& pn : S->patch) {
    cudaKernelNodeParams kp{};
    cudaError_t e = cudaGraphKernelNodeGetParams(pn.node, &kp);
    if (e != cudaSuccess) return e;
    std::vector<unsigned char> args = pn.args;
    for (size_t off : pn.in_offsets) std::memcpy(args.data() + off, &x_in, sizeof(void*));
    for (size_t off : pn.out_offsets) std::memcpy(args.data() + off, &x_out, sizeof(void*));
    void* params[3] = {nullptr, nullptr, nullptr};
    for (int i = 0; i <= pn.arg_index; ++i) params[i] = kp.kernelParams[i];
    params[pn.arg_index] = args.data();
    kp.kernelParams = params;
    kp.extra = nullptr;
    e = cudaGraphExecKernelNodeSetParams(S->exec, pn.node, &kp);
    if (e != cudaSuccess) return e;
  }
  S->x_in = x_in;
  S->x_out = x_out;
  return cudaSuccess;
}

}  // namespace

extern "C" {

ds_status ds_stack_destroy(ds_stack* stack) {
  if (stack == nullptr) return DS_OK;
  drop_graph(stack);
  for (cudaEvent_t ev : stack->events) cudaEventDestroy(ev);
  delete stack;
  return DS_OK;
}

size_t ds_stack_workspace_bytes(const ds_stack* stack, int batch) {
  if (stack == nullptr) return 0;
  return ds_layer_workspace_bytes(stack->layers[0], batch, 1);
}

ds_status ds_stack_decode_step(ds_stack* stack, const void* x_in, void* x_out, int batch,
                               void* const* k_caches, void* const* v_caches, int max_len,
                               int32_t* seq_len, void* workspace, size_t ws_bytes, void* stream) {
  if (stack == nullptr) return fail(DS_ERR_INVALID_ARG, "stack is null");
  if (k_caches == nullptr || v_caches == nullptr) return fail(DS_ERR_INVALID_ARG, "cache arrays are null");
  const int L = (int)stack->layers.size();
  const ds_layer& L0 = *stack->layers[0];
  for (int l = 0; l < L; ++l) {
    ds_status s = check_forward_args(L0, x_in, x_out, batch, 1, k_caches[l], v_caches[l], max_len, seq_len, workspace);
    if (s != DS_OK) return s;
  }
  ds_status s = check_device(L0);
  if (s != DS_OK) return s;
  if ((s = check_attn_smem(L0)) != DS_OK) return s;
  Plans p;
  if (!make_plans(L0, batch, &p)) return fail(DS_ERR_UNSUPPORTED, "no GEMM work split for this shape");
  const WsLayout wl = ws_layout(L0, batch, 1, p);
  if (ws_bytes < wl.total) return fail(DS_ERR_WORKSPACE, "workspace smaller than ds_stack_workspace_bytes()");
  const Bufs bf = bufs_of(workspace, wl);
  XMaps xm;
  if (p.tile && !make_xmaps(L0, p, bf, batch, &xm))
    return fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation operand");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int kernels = kernels_per_layer(p) * L;

  if (stack->profiling) {
    const size_t need = (size_t)2 * 5 * L;
    while (stack->events.size() < need) {
      cudaEvent_t ev;
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
      stack->events.push_back(ev);
    }
    EventSink es;
    es.ev = &stack->events;
    cudaError_t e = enqueue_stack(stack, p, bf, &xm, x_in, x_out, batch, k_caches, v_caches, max_len, seq_len, st,
                                  false, &es, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "region kernel launch (profile)");
    g_launches += kernels;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize (profile)");
    for (int k = 0; k < 5 * L; ++k) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, stack->events[2 * k], stack->events[2 * k + 1]);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
      stack->acc_ms[k % 5] += ms;
      stack->acc_n[k % 5] += 1;
    }
    return DS_OK;
  }

  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (st != nullptr) {
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  }
  if (st == nullptr || cs != cudaStreamCaptureStatusNone) {
    cudaError_t e = enqueue_stack(stack, p, bf, &xm, x_in, x_out, batch, k_caches, v_caches, max_len, seq_len, st,
                                  true, nullptr, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "region kernel launch");
    g_launches += kernels;
    return DS_OK;
  }

  GraphKey key;
  key.batch = batch;
  key.kc.assign(k_caches, k_caches + L);
  key.vc.assign(v_caches, v_caches + L);
  key.max_len = max_len;
  key.seq = seq_len;
  key.ws = workspace;
  if (!stack->have_graph || !(stack->key == key)) {
    drop_graph(stack);
    cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
    std::vector<PatchNode> rec;
    cudaError_t el = enqueue_stack(stack, p, bf, &xm, x_in, x_out, batch, k_caches, v_caches, max_len, seq_len, st,
                                   true, nullptr, &rec);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(st, &graph);
    if (el != cudaSuccess) {
      if (graph != nullptr) cudaGraphDestroy(graph);
      return cuda_fail(el, "region kernel launch (capture)");
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(&stack->exec, graph, 0);
    if (e != cudaSuccess) {
      cudaGraphDestroy(graph);
      stack->exec = nullptr;
      return cuda_fail(e, "cudaGraphInstantiate");
    }
    stack->graph = graph;
    stack->patch = std::move(rec);
    stack->key = key;
    stack->x_in = x_in;
    stack->x_out = x_out;
    stack->have_graph = true;
    stack->graph_kernels = kernels;
    stack->captures += 1;
  } else if (x_in != stack->x_in || x_out != stack->x_out) {
    cudaError_t e = patch_graph(stack, x_in, x_out);
    if (e != cudaSuccess) {
      drop_graph(stack);
      return cuda_fail(e, "cudaGraphExecKernelNodeSetParams");
    }
  }
  cudaError_t e = cudaGraphLaunch(stack->exec, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  g_launches += stack->graph_kernels;
  return DS_OK;
}

ds_status ds_stack_forward(ds_stack* stack, const void* x_in, void* x_out, int batch, int new_tokens,
                           void* const* k_caches, void* const* v_caches, int max_len, const int32_t* past_len,
                           void* workspace, size_t ws_bytes, void* stream) {
  if (stack == nullptr) return fail(DS_ERR_INVALID_ARG, "stack is null");
  if (k_caches == nullptr || v_caches == nullptr) return fail(DS_ERR_INVALID_ARG, "cache arrays are null");
  const int L = (int)stack->layers.size();
  const ds_layer& L0 = *stack->layers[0];
  for (int l = 0; l < L; ++l) {
    ds_status s = check_forward_args(L0, x_in, x_out, batch, new_tokens, k_caches[l], v_caches[l], max_len, past_len,
                                     workspace);
    if (s != DS_OK) return s;
  }
  ds_status s = check_device(L0);
  if (s != DS_OK) return s;
  if ((s = check_attn_smem(L0)) != DS_OK) return s;
  const int M = batch * new_tokens;
  Plans p;
  if (!make_plans(L0, M, &p)) return fail(DS_ERR_UNSUPPORTED, "no GEMM work split for this shape");
  const WsLayout wl = ws_layout(L0, batch, new_tokens, p);
  if (ws_bytes < wl.total) return fail(DS_ERR_WORKSPACE, "workspace smaller than ds_layer_workspace_bytes()");
  const Bufs bf = bufs_of(workspace, wl);
  XMaps xm;
  if (p.tile && !make_xmaps(L0, p, bf, M, &xm))
    return fail(DS_ERR_CUDA, "cuTensorMapEncodeTiled failed for an activation operand");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  EventSink es;
  if (stack->profiling) {
    while (stack->events.size() < (size_t)2 * 5 * L) {
      cudaEvent_t ev;
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
      stack->events.push_back(ev);
    }
    es.ev = &stack->events;
  }
  cudaError_t e = enqueue_stack(stack, p, bf, &xm, x_in, x_out, batch, k_caches, v_caches, max_len,
                                const_cast<int32_t*>(past_len), st, !stack->profiling,
                                stack->profiling ? &es : nullptr, nullptr, new_tokens, /*advance=*/false);
  if (e != cudaSuccess) return cuda_fail(e, "region kernel launch");
  g_launches += kernels_per_layer(p) * L;
  if (stack->profiling) {
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize (profile)");
    for (int k = 0; k < 5 * L; ++k) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, stack->events[2 * k], stack->events[2 * k + 1]);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
      stack->acc_ms[k % 5] += ms;
      stack->acc_n[k % 5] += 1;
    }
  }
  return DS_OK;
}

ds_status ds_stack_decode_host(ds_stack* stack, const void* x_host, void* y_host, void* x_dev_in,
                               void* x_dev_out, int batch, void* const* k_caches,
                               void* const* v_caches, int max_len, int32_t* seq_len,
                               void* workspace, size_t ws_bytes, void* stream) {
  if (stack == nullptr) return fail(DS_ERR_INVALID_ARG, "stack is null");
  if (x_host == nullptr || y_host == nullptr) return fail(DS_ERR_INVALID_ARG, "host buffers are null");
  if (batch < 1 || batch > stack->layers[0]->max_rows()) return fail(DS_ERR_UNSUPPORTED, "batch out of range");
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

uint64_t ds_stack_graph_captures(const ds_stack* stack) { return stack == nullptr ? 0 : stack->captures; }

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

ds_status ds_selftest_wait_timeout(void* workspace, uint32_t budget_us, void* stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DS_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (budget_us < 1 || budget_us > 1000000) return fail(DS_ERR_INVALID_ARG, "budget_us must be in 1 .. 1000000");
  cudaError_t e = launch_wait_timeout_selftest(static_cast<unsigned*>(workspace), (unsigned long long)budget_us * 1000ull,
                                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait-timeout self-test launch");
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
