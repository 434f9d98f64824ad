// Internal launch interface between the C-ABI layer (ds_api.cu) and the
// region kernels.  Nothing here is exported from the shared library.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ds_layer.h"

namespace ds {

enum class WKind : int { F16 = 0, BF16 = 1, I8 = 2 };

constexpr int kTensorMapBytes = 128;  // sizeof(CUtensorMap)

// Encodes the tensor map of a row-major weight matrix (rows x row_bytes) whose
// box is one GEMV chunk, 16 rows x chunk_row_bytes, delivered as
// [128-byte segment][row][128 bytes] with the 128-byte swizzle (the layout of
// ring_layout.h); false if the driver entry point or the encoding fails.
bool encode_weight_map(void* map128, const void* base, int rows, size_t row_bytes, int chunk_row_bytes);
// Tensor map of int8 group scales (rows x groups fp16) with box_rows x box_groups boxes.
bool encode_scale_map(void* map128, const void* base, int rows, int groups, int box_groups, int box_rows = 16);
enum class ActKind : int { F16 = 0, BF16 = 1 };

// The four GEMV-based region kernels ([P1] §3.2 regions 1, 3, 3/4 and 4).
enum class Region : int {
  LnQkv = 0,     // R1: LayerNorm1 prologue, QKV GEMV, bias, KV-cache append
  OprojRes = 1,  // R3: O-proj GEMV, bias, residual, LayerNorm2 statistics
  FfnUp = 2,     // R4a: LayerNorm2 prologue, FFN-up GEMV, bias, GeLU
  FfnDown = 3    // R4b: FFN-down GEMV, bias, residual (+ next LayerNorm statistics)
};

// Work split of one skinny GEMM y[M][N] = x[M][K] W[N][K]^T (see gemv_impl.cuh).
// A unit is 16 weight rows x one K slice; a chunk is 8 warp steps of a unit.
// Every CTA owns q whole units (data-parallel part); the leftover units'
// chunks are spread evenly over all CTAs, whose partial sums are combined by
// the last contributor of each row tile.
struct GemvPlan {
  int KS = 1;        // number of K slices
  int K_S = 0;       // slice length
  int tiles = 0;     // N / 16 row tiles
  int units = 0;     // KS * tiles, slice-major (u = s * tiles + t)
  int C = 0;         // chunks per unit
  int chunk_k = 0;   // k per chunk (8 warps x one warp step)
  int q = 0;         // whole units per CTA
  int U_dp = 0;      // q * grid
  long long R = 0;   // leftover chunks spread over the grid
  int maxc = 1;      // most CTAs contributing to one leftover unit
  int whole = 0;     // 1: leftover units go whole to CTAs (no split-K fix-up)
  int interleave = 0;  // 1: CTA c's whole units are c, c + grid, c + 2 grid, ... (else c q .. c q + q - 1)
  int grid = 0;      // CTAs
  int nt = 1;        // n-tiles of 8 batch rows (1, 2, 4, 8)
  int nblk = 4;      // k-blocks per warp step (4, or 2 / 1 for narrow K)
  int stages = 0;    // depth of the shared-memory weight ring (chunks in flight)
  size_t smem = 0;   // dynamic shared memory bytes
};

struct RegionArgs {
  // GEMV operand
  const void* W = nullptr;         // [N][K] weights (fp16/bf16) or int8 codes
  const __half* Wscale = nullptr;  // int8: fp16 scales [N][K/64]
  const void* tmap_w = nullptr;    // device address of W's tensor map (64-byte aligned)
  const void* tmap_s = nullptr;    // int8: device address of the scales' tensor map
  int qgroup = 64;                 // int8: scale group length along K (64 or 128)
  int N = 0, K = 0, M = 0;         // M = B * T rows
  int B = 1, T = 1;
  GemvPlan plan;
  float* partials = nullptr;       // [tiles][KS * maxc][16][M] partial sums
  int* counters = nullptr;         // [tiles] arrival counters (self-resetting)
  const void* bias = nullptr;      // [N] act dtype
  // prologue
  const void* x_act = nullptr;     // R1: layer input [M][K] act dtype
  const float* x_f32 = nullptr;    // R3: attention output; R4a: x1; R4b: GeLU output
  const void* ln_g = nullptr;      // LayerNorm gamma / beta (R1, R4a)
  const void* ln_b = nullptr;
  float eps = 1e-5f;
  const float* stats_in = nullptr; // [K/16][M][2] (sum, M2) partials, or null
  // epilogue
  float* out_f32 = nullptr;        // R1: q [M][H]; R3: x1; R4a: g
  void* out_act = nullptr;         // R4b: layer output [M][N]
  const void* resid_act = nullptr; // R3: layer input (residual)
  const float* resid_f32 = nullptr;// R4b: x1 (residual)
  float* stats_out = nullptr;      // R3 / R4b: [N/16][M][2] partials, or null
  // R1 cache append
  void* k_cache = nullptr;
  void* v_cache = nullptr;
  int heads = 0, head_dim = 0, max_len = 0, H = 0;
  const int32_t* past_len = nullptr;
  unsigned* status = nullptr;
  // R4b of the last layer of a stack step: add 1 to seq_len[0..B) at the end
  int32_t* seq_len_inc = nullptr;
  // The GEMV kernel that runs next on the stream (null map: none).  Once a
  // CTA's own copies are issued it asks L2 to prefetch the first chunks the
  // same CTA index streams there, so HBM keeps working across the kernels'
  // dependency gap.
  const void* next_tmap_w = nullptr;
  const void* next_tmap_s = nullptr;
  GemvPlan next_plan;
  int next_qgroup = 64;  // int8: that matrix's scale group length
};

// Tensor-core tile path (dense_impl.cuh): one output tile is 128 weight rows x
// ntok rows of X; units of the work split are output tiles (u = token tile *
// row_tiles + row tile), chunks are kc-wide K ranges, one K slice.
struct DensePlan {
  GemvPlan ws;         // tiles = units = row_tiles * tok_tiles, KS = 1, chunk_k = kc
  int row_tiles = 0;   // N / 128
  int tok_tiles = 0;   // ceil(M / ntok)
  int ntok = 0;        // X rows per tile = MMA N (multiple of 16, <= 256)
  int kc = 128;        // K per ring stage (64 or 128)
  int stages = 0;
  size_t smem = 0;
  int cluster = 1;     // > 1: the K slices of each tile are one thread-block cluster of this many
                       // CTAs (one slice each) whose partial sums meet in distributed shared memory;
                       // slice s then holds K chunks [s kchunks / cluster, (s + 1) kchunks / cluster)
                       // (ws.C: the longest), else each slice holds ws.C chunks
  int kchunks = 0;     // K / kc
  int i8 = 0;          // 1: int8 weight codes (fp16 activations), dequantised to fp16 in tensor memory
};

struct DenseArgs {
  const void* tmap_w = nullptr;    // device address of W's tile tensor map (box 128 rows x kc)
  const void* tmap_s = nullptr;    // int8: device address of the fp16 scales' [N][K / qgroup] tensor map (box 8 groups x 128 rows)
  int qgroup = 64;                 // int8: scale group length along K (a power of two, >= 64)
  int N = 0, K = 0, M = 0, B = 1, T = 1;
  DensePlan plan;
  float* partials = nullptr;       // [tiles - U_dp][maxc][ntok][128] partial sums of the leftover tiles
  int* counters = nullptr;         // [tiles] arrival counters (self-resetting)
  const void* bias = nullptr;      // [N] act dtype, or null (no bias: a tensor-sliced rank other than 0)
  // epilogue
  float* out_f32 = nullptr;        // R1: q [M][H]; R3: x1; R4b: a tensor-sliced rank's partial sum (else null)
  void* out_act = nullptr;         // R4a: GeLU output (operand hi); R4b: layer output
  void* out_lo = nullptr;          // R4a, bf16: operand lo
  const void* resid_act = nullptr; // R3: layer input, or null (no residual)
  const float* resid_f32 = nullptr;// R4b: x1, or null (no residual)
  float* stats_out = nullptr;      // R3 / R4b: [N/16][M][2] (sum, M2) partials, or null
  void* k_cache = nullptr;         // R1 cache append
  void* v_cache = nullptr;
  int heads = 0, head_dim = 0, max_len = 0, H = 0;
  const int32_t* past_len = nullptr;
  unsigned* status = nullptr;
  int32_t* seq_len_inc = nullptr;  // R4b of a stack step's last layer
  const void* next_tmap_w = nullptr;  // the next tile GEMM (L2 prefetch), or null
  DensePlan next_plan;
  // Expert selection (residual-MoE FFN): when sel_idx is set, W is expert
  // *sel_idx -- its tensor map at tmap_table + 128 * idx, its bias at
  // bias + sel_bias_stride * idx -- read after the dependency wait; when
  // sel_scale is set, the epilogue takes (acc + bias) * *sel_scale.
  const unsigned char* tmap_table = nullptr;
  const int32_t* sel_idx = nullptr;
  const float* sel_scale = nullptr;
  int sel_bias_stride = 0;
};

// Row normalisation ahead of a tile GEMM (regions 1 and 4a): out = LN(x) in
// the MMA operand format (activation dtype; bf16 also writes the lo part).
struct LnPrepArgs {
  int M = 0, K = 0;
  float eps = 1e-5f;
  const void* x_act = nullptr;     // [M][K] act dtype (region 1), or
  const float* x_f32 = nullptr;    // [M][K] fp32 (region 4a)
  const float* stats_in = nullptr; // [K/16][M][2] (sum, M2) partials, or null (two passes over the row)
  const void* ln_g = nullptr;
  const void* ln_b = nullptr;
  void* out_hi = nullptr;          // [M][K]
  void* out_lo = nullptr;          // [M][K], bf16 only
};

struct AttnArgs {
  const float* q = nullptr;         // [B*T][H] fp32
  const void* k_cache = nullptr;    // [B][nh][max_len][d]
  const void* v_cache = nullptr;
  const int32_t* past_len = nullptr;
  int B = 1, T = 1, heads = 0, head_dim = 0, max_len = 0, H = 0;
  int nsplit = 1;                   // CTAs per (b, h), one thread-block cluster (<= 8)
  float scale_log2 = 0.f;           // log2(e) / sqrt(head_dim)
  int stage_keys = 0;               // cached keys per split copied to shared memory up front
  size_t smem = 0;
  float* out = nullptr;             // [B*T][H] fp32, or
  void* out_hi = nullptr;           // [B*T][H] in the MMA operand format (tile path)
  void* out_lo = nullptr;           // (bf16 only)
  unsigned* status = nullptr;       // workspace status word (wait-timeout flag)
};

// Chooses the work split for one GEMV over num_sms CTAs; returns false if no
// valid split exists.
bool gemv_make_plan(WKind wk, ActKind ak, int N, int K, int M, int num_sms, int max_smem, GemvPlan* plan);
cudaError_t launch_region(Region r, WKind wk, ActKind ak, const RegionArgs& a,
                          cudaStream_t st, bool pdl);
// Sets the dynamic shared-memory limit of every region kernel (call once per
// device before the first launch).
cudaError_t prepare_region_kernels(int max_smem);

// Tile path: plan (false if the shape has no tile split), launch, and the
// row normalisation kernel.
bool dense_make_plan(ActKind ak, int N, int K, int M, int num_sms, int max_smem, DensePlan* plan, bool i8 = false);
// Encodes the tile tensor map of a row-major [rows][cols] 16-bit matrix
// (box 128 rows x kc, or ntok rows x kc for activation operands).
bool encode_tile_map(void* map128, const void* base, int rows, int cols, int box_rows, int kc);
cudaError_t launch_dense(Region r, ActKind ak, const DenseArgs& a, const void* xmap_hi, const void* xmap_lo,
                         cudaStream_t st, bool pdl);
cudaError_t launch_ln_prep(ActKind ak, const LnPrepArgs& a, cudaStream_t st, bool pdl);
cudaError_t prepare_dense_kernels(int max_smem);
cudaError_t prepare_moe_kernels(int max_smem);

// Sets a.nsplit, a.stage_keys and a.smem of the decode attention from a.B,
// a.heads, a.max_len and a.head_dim.
void attn_configure(AttnArgs& a, ActKind ak, int num_sms, int max_smem);
// Shared memory of the decode attention kernel staging stage_keys K and V rows.
size_t attn_smem_bytes(int head_dim, int stage_keys);
cudaError_t launch_attention(ActKind ak, const AttnArgs& a, cudaStream_t st, bool pdl);
cudaError_t prepare_attention_kernels(int max_smem);
// Prompt chunks: tiled tensor-core (flash) attention, used from this many new
// tokens per sequence on.
constexpr int kPrefillMinTokens = 16;
size_t attn_prefill_smem_bytes(ActKind ak, int head_dim);
cudaError_t launch_attention_prefill(ActKind ak, const AttnArgs& a, cudaStream_t st, bool pdl);
cudaError_t prepare_attention_prefill_kernels(int max_smem);

}  // namespace ds

struct ds_layer;
namespace ds {
// ds_layer_forward in two steps: validation (nothing enqueued; on success
// *zero_prefix = leading workspace bytes -- status word and arrival counters --
// that must be zero before the call), then the launches.
ds_status layer_forward_check(const ds_layer* layer, const void* x_in, const void* x_out, int batch,
                                int new_tokens, const void* k_cache, const void* v_cache, int max_len,
                                const int32_t* past_len, const void* workspace, size_t ws_bytes,
                                size_t* zero_prefix);
ds_status layer_forward_enqueue(ds_layer* layer, const void* x_in, void* x_out, int batch, int new_tokens,
                                  void* k_cache, void* v_cache, int max_len, const int32_t* past_len,
                                  void* workspace, void* stream);
// Sets the detail string returned by ds_last_error() on this thread.
void set_last_error(const char* msg);
// The device a layer was created on.
int layer_device(const ds_layer* layer);
// Adds n to the count ds_launch_count() reports.
void add_launches(unsigned long long n);

cudaError_t launch_wait_timeout_selftest(unsigned* status, unsigned long long budget_ns, cudaStream_t st);
cudaError_t launch_quantize_int8(const void* w, int n, int k, int group, int8_t* codes, void* scales,
                                 cudaStream_t st);

}  // namespace ds
