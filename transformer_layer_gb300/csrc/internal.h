// Internal launch interface between the C-ABI layer (ds_api.cu) and the
// region kernels.  Nothing here is exported from the shared library.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ds {

enum class WKind : int { F16 = 0, BF16 = 1, I8 = 2 };

constexpr int kTensorMapBytes = 128;  // sizeof(CUtensorMap)

// Encodes the tensor map of a row-major weight matrix (rows x row_bytes) whose
// box is one GEMV chunk, 16 rows x chunk_row_bytes, delivered as
// [128-byte segment][row][128 bytes] with the 128-byte swizzle (the layout of
// ring_layout.h); false if the driver entry point or the encoding fails.
bool encode_weight_map(void* map128, const void* base, int rows, size_t row_bytes, int chunk_row_bytes);
// Tensor map of int8 group scales (rows x groups fp16) with 16 x box_groups boxes.
bool encode_scale_map(void* map128, const void* base, int rows, int groups, int box_groups);
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
  float* out = nullptr;             // [B*T][H] fp32
  unsigned* status = nullptr;       // workspace status word (wait-timeout flag)
};

// ---------------------------------------------------------------- step kernel
// One persistent, cooperative launch runs a whole decode step (T = 1) of a
// stack: per layer the phases LN1+QKV, attention, O-proj, LN2+FFN-up and
// FFN-down, separated by grid-wide barriers, while the copy warps stream the
// weights of the following phases without stopping.
constexpr int kStepMaxLayers = 64;

struct StepLayer {
  const void* w[4];     // w_qkv, w_o, w_fc1, w_fc2
  const __half* sc[4];  // their int8 group scales (int8 weights only)
  const void* bias[4];  // b_qkv, b_o, b_fc1, b_fc2
  const void* tmap_w[4];  // device addresses of the weights' tensor maps
  const void* tmap_s[4];  // and of the int8 scales' tensor maps
  const void* ln1_g;
  const void* ln1_b;
  const void* ln2_g;
  const void* ln2_b;
  void* kc;
  void* vc;
};

struct StepArgs {
  int L = 0, B = 1, H = 0, F = 0, heads = 0, head_dim = 0, max_len = 0;
  int qgroup[4] = {64, 64, 64, 64};  // int8 scale group length of each phase's matrix
  float eps = 1e-5f, scale_log2 = 0.f;
  int nsplit = 1;           // attention key splits per (b, h)
  GemvPlan plan[4];         // QKV, O-proj, FFN-up, FFN-down
  int stages = 0;           // common weight-ring geometry
  size_t SB = 0;            // ring stage stride, bytes
  size_t xs_cap = 0;        // staged-x bytes (largest phase)
  const void* x_in = nullptr;
  void* x_out = nullptr;
  int32_t* seq = nullptr;   // [B] cached positions; +1 at the end of the step
  unsigned* status = nullptr;
  int* counters = nullptr;  // GEMV row-tile arrival counters
  unsigned* grid_bar = nullptr;  // grid barrier counter (returns to 0 at the end)
  int* attn_cnt = nullptr;  // [B][nh] attention split counters
  float *q = nullptr, *o = nullptr, *x1 = nullptr, *g = nullptr;
  float *stats_a = nullptr, *stats_b = nullptr, *partials = nullptr, *attn_part = nullptr;
  char* act = nullptr;      // [2][B][H] ping-pong layer outputs
  StepLayer layer[kStepMaxLayers];
};

int step_attn_nsplit(int B, int heads, int max_len, int grid);
size_t step_smem_bytes(int nt, int stages, size_t SB, size_t xs_cap);
// Fills stages / SB / xs_cap of `s` from its four plans; false if no ring fits.
bool step_geometry(WKind wk, ActKind ak, int M, int max_smem, StepArgs* s);
cudaError_t launch_step(WKind wk, ActKind ak, const StepArgs& s, int grid, cudaStream_t st);
// CTAs of the step kernel that fit on one SM (0 if the launch cannot work).
int step_blocks_per_sm(WKind wk, ActKind ak, int nt, size_t smem);
cudaError_t prepare_step_kernels(int max_smem);

// Chooses the work split for one GEMV; returns false if no valid split exists.
// fixed_grid: exactly num_sms * ctas_per_sm CTAs even for less work (step kernel).
bool gemv_make_plan(WKind wk, ActKind ak, int N, int K, int M, int num_sms, int ctas_per_sm,
                    int max_smem, GemvPlan* plan, bool fixed_grid = false);
cudaError_t launch_region(Region r, WKind wk, ActKind ak, const RegionArgs& a,
                          cudaStream_t st, bool pdl);
// Sets the dynamic shared-memory limit of every region kernel (call once per
// device before the first launch).
cudaError_t prepare_region_kernels(int max_smem);

int attn_nsplit(int B, int heads, int max_len, int num_sms);
// Shared memory of the attention kernel, and the cached keys per split it
// stages there (all of a split's keys when they fit a 48 KB budget).
size_t attn_smem_bytes(int head_dim, int stage_keys);
int attn_stage_keys(int head_dim, int max_len, int nsplit);
cudaError_t launch_attention(ActKind ak, const AttnArgs& a, cudaStream_t st, bool pdl);
cudaError_t prepare_attention_kernels(int max_smem);

}  // namespace ds

struct ds_layer;
namespace ds {
// Leading workspace bytes (status word + arrival counters) that must be zero
// before a ds_layer_forward call with this batch shape; 0 if invalid.
size_t layer_workspace_zero_prefix(const ds_layer* layer, int batch, int new_tokens);
// Sets the detail string returned by ds_last_error() on this thread.
void set_last_error(const char* msg);

cudaError_t launch_quantize_int8(const void* w, int n, int k, int group, int8_t* codes, void* scales,
                                 cudaStream_t st);

}  // namespace ds
