/*
 * ds_layer.h -- C ABI of libdslayer.so: fused decode steps of a pre-LN
 * GPT-style transformer layer, or a stack of such layers, on one GB300 GPU.
 *
 * Source pages (cited by title and section):
 *   [P1] "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核
 *        与 MoQ 量化支持" -- §3 intro (vector-matrix / skinny matrix-matrix GEMM
 *        with ops fused at its reduction boundary), §3.1 (fusion principles),
 *        §3.2 (the four fusion regions of a layer), §3.3 (shared memory and
 *        warp-level reductions), §5.2 (int8 inference kernels, quantisation
 *        groups).
 *   [P3] "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、PR-MoE 优化与
 *        init_inference 全解析" -- table "推理配置参数详解" (dtype choices,
 *        triangular_masking).
 *
 * What one layer computes (regions of [P1] §3.2; T new tokens per sequence):
 *   R1  h1 = LayerNorm1(x);  [q|k|v] = h1 W_qkv^T + b_qkv;  k, v are appended
 *       to the caller's KV cache at positions past_len[b] .. past_len[b]+T-1.
 *   R2  o = softmax(q K^T / sqrt(d), causal) V per head, over the cache.
 *   R3  x1 = x + o W_o^T + b_o, and the statistics of LayerNorm2(x1).
 *   R4  g = GeLU_tanh(LN2(x1) W_1^T + b_1);  y = x1 + g W_2^T + b_2.
 * LayerNorm: biased variance, eps from the config (1e-5 by default), affine
 * after the normalisation.  GeLU: 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))).
 *
 * Conventions shared by every entry point
 *   - All tensors are caller-owned DEVICE memory unless a parameter says HOST.
 *     The library copies no weights: create() stores the pointers, so the
 *     caller keeps them alive and unchanged until destroy().
 *   - Weights are [out][in] row-major (the input axis K is contiguous).
 *     Fused QKV rows: q block (rows 0..H-1), k block, v block; inside a block
 *     head i owns rows i*d .. (i+1)*d-1.
 *   - Hidden states are [B][T][H] (batch rows, new tokens, features) in the
 *     activation dtype.  The K and V caches of a layer are two separate
 *     arrays [B][nh][max_len][d] in the activation dtype.
 *   - Every pointer must be 16-byte aligned (the workspace 256-byte aligned);
 *     d must be 64 or 128; H and F must be multiples of 256 for fp16/bf16
 *     weights and of 512 for int8 weights, and of 1024 where a matrix with
 *     that input width uses groups of 128 (H with quant_group 128; F with
 *     quant_group 128 and no extra MLP grouping).
 *   - Rows R = B*T (batch rows x new tokens) per call: 1..4096 with fp16 /
 *     bf16 weights and with int8 weights under fp16 activations; 1..64 with
 *     int8 weights under bf16 activations.  Up to 7 rows (and always for
 *     int8 under bf16) the GEMMs run as streaming skinny-GEMM kernels with
 *     the LayerNorm fused into their prologue; from 8 rows as tensor-core
 *     tile kernels (tcgen05, accumulators in tensor memory), each LayerNorm
 *     then running as a small row kernel ahead of its GEMM (seven kernels
 *     per layer instead of five).  The int8 tile kernels dequantise each
 *     stage of codes to fp16 in tensor memory, the MMAs' A operand (q * s
 *     rounded once to fp16, the MMA operand type); the int8 streaming kernels apply each group's
 *     scale to its fp32 partial sum.  With int8 weights under bf16
 *     activations the activations staged per GEMV slice (80 KB of shared
 *     memory) bound R further: up to 39 rows for groups of 64, 19 once a
 *     matrix uses groups of 128.  Beyond the limits ds_layer_workspace_bytes
 *     and ds_stack_workspace_bytes return 0 and the forward calls return
 *     DS_ERR_UNSUPPORTED before any launch.
 *   - The forward calls run on the device the layer was created on, which
 *     must be the current device (else DS_ERR_INVALID_ARG, nothing launched).
 *   - Calls are asynchronous on the given stream (never synchronising, except
 *     ds_stack_region_times, ds_workspace_status and ds_stack_decode_host,
 *     which say so).  A stream of 0 means the legacy default stream.
 *   - Errors: arguments are validated before any launch; a bad argument
 *     returns DS_ERR_INVALID_ARG or DS_ERR_UNSUPPORTED and launches nothing.
 *     A launch failure returns DS_ERR_CUDA.  Faults that happen later on the
 *     device surface on a later call.  No C++ exception crosses this ABI.
 *     ds_last_error() gives a human-readable detail of the last failure on
 *     the calling thread.  There is no CPU fallback.
 *   - A handle may be used from one stream at a time.
 */
#ifndef DS_LAYER_H
#define DS_LAYER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DS_API __attribute__((visibility("default")))
#else
#define DS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size or shape      */
  DS_ERR_UNSUPPORTED = 2,   /* a valid request the library does not implement    */
  DS_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed        */
  DS_ERR_WORKSPACE = 4,     /* workspace smaller than ds_*_workspace_bytes()      */
  DS_ERR_DEVICE = 5         /* a device-side check failed (see ds_workspace_status) */
} ds_status;

typedef enum { DS_F16 = 0, DS_BF16 = 1, DS_I8 = 2 } ds_dtype;

/* Shape and numeric format of one layer ([P1] §3.2; dtypes as in the [P3]
 * configuration table; int8 weights as in [P1] §5.2). */
typedef struct {
  int hidden;          /* H                                                   */
  int heads;           /* nh; head_dim d = H / nh                             */
  int ffn;             /* F, width of the FFN up-projection                   */
  float ln_eps;        /* LayerNorm epsilon (1e-5 in every shipped workload)  */
  ds_dtype act_dtype;  /* DS_F16 or DS_BF16: hidden states, caches, biases, LN */
  ds_dtype weight_dtype; /* DS_F16 / DS_BF16 (must equal act_dtype) or DS_I8    */
  int quant_group;     /* DS_I8 only: group length along K, 64 or 128          */
  int mlp_extra_grouping; /* DS_I8 only: 0, or 1 = the FFN matrices w_fc1 and
                           * w_fc2 use groups of quant_group / 2 (twice as many
                           * groups as w_qkv and w_o; quant_group must then be 128) */
} ds_layer_config;

/* Device pointers to one layer's parameters.  Vectors are in act_dtype.
 * Matrices are [out][in]: w_qkv [3H][H], w_o [H][H], w_fc1 [F][H], w_fc2 [H][F],
 * in weight_dtype (int8 codes for DS_I8).  For DS_I8, s_* hold the float16
 * group scales [out][in / g]: g = quant_group for s_qkv and s_o, and for s_fc1
 * and s_fc2 quant_group / 2 with mlp_extra_grouping, else quant_group.  They
 * are ignored for other weight dtypes. */
typedef struct {
  const void *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o;
  const void *ln2_g, *ln2_b, *w_fc1, *b_fc1, *w_fc2, *b_fc2;
  const void *s_qkv, *s_o, *s_fc1, *s_fc2;
} ds_layer_weights;

typedef struct ds_layer ds_layer;
typedef struct ds_stack ds_stack;

/* Validates the config and stores the weight pointers (no copy, no launch).
 * *out receives a handle owned by the caller; free it with ds_layer_destroy. */
DS_API ds_status ds_layer_create(const ds_layer_config* cfg, const ds_layer_weights* w,
                          ds_layer** out);
DS_API ds_status ds_layer_destroy(ds_layer* layer);

/* Bytes of device workspace that ds_layer_forward needs for `batch` sequences
 * of `new_tokens` tokens each.  Returns 0 for invalid arguments. */
DS_API size_t ds_layer_workspace_bytes(const ds_layer* layer, int batch, int new_tokens);

/* Zero-fills a workspace (the counters inside it must start at zero).  Call it
 * once after allocating a workspace; every successful call leaves the
 * counters at zero again, so one workspace serves any number of calls. */
DS_API ds_status ds_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* One layer forward over T = new_tokens new tokens per sequence (regions
 * R1..R4 of [P1] §3.2); T > 1 is a prompt chunk (query t of sequence b sees
 * keys 0 .. past_len[b] + t, [P3] triangular_masking).
 *   x_in     [B][T][H] act_dtype, read only
 *   x_out    [B][T][H] act_dtype, written (must not alias x_in)
 *   k_cache, v_cache  [B][nh][max_len][d]; positions past_len[b]+t are written
 *   past_len [B] int32 DEVICE array, read only; past_len[b] + T <= max_len is
 *            required.  A violating row is not written: its outputs are left
 *            unspecified and the workspace status word records
 *            DS_DEVFLAG_CACHE_OVERFLOW (read it with ds_workspace_status).
 *   workspace  device scratch of at least ds_layer_workspace_bytes() bytes,
 *            zero-filled once (ds_workspace_init) before first use.
 * Five kernels (seven on the tile path) are enqueued on `stream` (a
 * cudaStream_t). */
DS_API ds_status ds_layer_forward(ds_layer* layer, const void* x_in, void* x_out, int batch,
                           int new_tokens, void* k_cache, void* v_cache, int max_len,
                           const int32_t* past_len, void* workspace, size_t ws_bytes,
                           void* stream);

/* ds_layer_forward for callers that cannot allocate device memory (plugins in
 * frameworks that own and pre-reserve all GPU memory, latency-critical loops
 * that must not risk the device-wide synchronisation of an allocation,
 * real-time hosts that forbid allocation after start-up).  The pages have no
 * counterpart: this is a property of the library, not of the method.
 * Runs the same kernels, with the workspace taken from a 16 MiB static
 * device array inside the library (every GPU that loads the library holds
 * it until the process exits); nothing is allocated or freed.
 *   - Returns DS_ERR_UNSUPPORTED when ds_layer_workspace_bytes(layer, batch,
 *     new_tokens) exceeds 16 MiB, and the argument errors of ds_layer_forward
 *     (a rejected call enqueues nothing and leaves the array untouched).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make it before any
 *     stream capture.  The cached address is not valid across
 *     cudaDeviceReset: do not use this entry point after a device reset.
 *   - All calls share the array: calls that overlap on the GPU race.  Each
 *     accepted call clears the array's status word and counters first;
 *     ds_noalloc_status reads the flags the last call left. */
DS_API ds_status ds_layer_forward_noalloc(ds_layer* layer, const void* x_in, void* x_out, int batch,
                                          int new_tokens, void* k_cache, void* v_cache, int max_len,
                                          const int32_t* past_len, void* stream);

/* Device status flags (DS_DEVFLAG_*) of the last ds_layer_forward_noalloc
 * call on the current device: copies the static array's status word to
 * *flags_out, clears it and synchronises `stream` (order it after that call).
 * Returns DS_ERR_DEVICE when a flag was set, DS_OK otherwise. */
DS_API ds_status ds_noalloc_status(uint32_t* flags_out, void* stream);

/* A stack of layers that share one config.  The layer handles stay owned by
 * the caller and must outlive the stack. */
DS_API ds_status ds_stack_create(ds_layer* const* layers, int n_layers, ds_stack** out);
DS_API ds_status ds_stack_destroy(ds_stack* stack);
DS_API size_t ds_stack_workspace_bytes(const ds_stack* stack, int batch);

/* One decode step (T = 1) through every layer of the stack.
 *   x_in, x_out  [B][H] act_dtype (must not alias)
 *   k_caches, v_caches  HOST arrays of n_layers DEVICE pointers, one cache
 *            pair per layer, each [B][nh][max_len][d]
 *   seq_len  [B] int32 DEVICE array: positions already cached; the new token
 *            is written at seq_len[b], and the step adds 1 to every entry on
 *            the device after the last layer has read it.
 * The launch sequence (5 kernels per layer, 7 on the tile path, chained with
 * programmatic dependent launch; the first kernel waits for all earlier work
 * on `stream`) is captured into a CUDA graph on the first call with a given
 * (batch, caches, max_len, seq_len, workspace) and replayed afterwards.  A
 * call with other x_in / x_out buffers updates the captured graph in place
 * (the kernel nodes that hold them) instead of capturing again, so a decode
 * loop may alternate or rotate its hidden-state buffers freely.  When
 * `stream` is the legacy default stream or is already capturing, the kernels
 * are launched directly. */
DS_API ds_status ds_stack_decode_step(ds_stack* stack, const void* x_in, void* x_out, int batch,
                               void* const* k_caches, void* const* v_caches, int max_len,
                               int32_t* seq_len, void* workspace, size_t ws_bytes,
                               void* stream);

/* A prompt chunk through every layer of the stack: T = new_tokens new tokens
 * per sequence, query t of sequence b attending keys 0 .. past_len[b] + t
 * ([P3] triangular_masking); each layer appends its keys and values at
 * positions past_len[b] .. past_len[b] + T - 1 of its own caches.
 *   x_in, x_out  [B][T][H] act_dtype (must not alias)
 *   past_len [B] int32 DEVICE array, read only (not advanced)
 *   workspace    at least ds_layer_workspace_bytes(layer 0, batch, new_tokens)
 * Launched directly (no graph capture), 5 or 7 kernels per layer.  In
 * profile mode (ds_stack_set_profiling) the region kernels are timed as for
 * ds_stack_decode_step and the call synchronises the stream. */
DS_API ds_status ds_stack_forward(ds_stack* stack, const void* x_in, void* x_out, int batch, int new_tokens,
                                  void* const* k_caches, void* const* v_caches, int max_len,
                                  const int32_t* past_len, void* workspace, size_t ws_bytes, void* stream);

/* The same decode step with the step's input and output in HOST memory:
 * copies x_host -> x_dev_in, runs ds_stack_decode_step, copies x_dev_out ->
 * y_host and synchronises `stream` before returning (end-to-end timing).
 * x_dev_in / x_dev_out are caller-owned device staging buffers [B][H]. */
DS_API ds_status ds_stack_decode_host(ds_stack* stack, const void* x_host, void* y_host,
                               void* x_dev_in, void* x_dev_out, int batch,
                               void* const* k_caches, void* const* v_caches, int max_len,
                               int32_t* seq_len, void* workspace, size_t ws_bytes,
                               void* stream);

/* Profile mode: when on, ds_stack_decode_step launches without the graph and
 * without programmatic dependent launch, records a CUDA event pair around
 * every region kernel, synchronises the stream at the end of the step and
 * accumulates the per-region kernel times. */
DS_API ds_status ds_stack_set_profiling(ds_stack* stack, int enabled);
/* Average microseconds per launch of each region kernel since the last reset:
 * us_out[0] R1 LN1+QKV, [1] R2 attention, [2] R3 O-proj+residual+LN2 stats,
 * [3] R4a FFN-up+GeLU, [4] R4b FFN-down+residual; launches_out[i] = launches
 * averaged.  Resets the accumulators. */
DS_API ds_status ds_stack_region_times(ds_stack* stack, float us_out[5], int launches_out[5]);

/* Number of CUDA-graph captures ds_stack_decode_step has made for this
 * stack since it was created (a new argument set captures again; new x_in /
 * x_out buffers do not). */
DS_API uint64_t ds_stack_graph_captures(const ds_stack* stack);

/* MoQ-style quantisation of a float16 weight matrix w_f16 [n][k] ([P1] §5.2):
 * per group of `group` (32, 64 or 128) consecutive weights along k, scale
 * s = fp16_rne(float32(max|w|) / 127) and code q = clamp(rne(w / s), -127, 127)
 * (IEEE float32 division); s = 0 and q = 0 for an all-zero group.
 * codes [n][k] int8 and scales_f16 [n][k/group] are written on `stream`. */
DS_API ds_status ds_quantize_int8(const void* w_f16, int n, int k, int group, int8_t* codes,
                           void* scales_f16, void* stream);

/* ---------------------------------------------------------------------------
 * Residual-MoE (PR-MoE) FFN block ([P3] section "用 PR-MoE 结构进一步提速并降低推理
 * 成本": mlp_type 'residual', per-layer expert counts; configuration table:
 * moe.type standard / residual, moe_experts).  The page gives no formula; the
 * reading implemented, for R rows of hidden states x:
 *   h = LayerNorm2(x);  p = softmax(h W_g^T) over E experts;
 *   e = argmax p (ties: the lowest index);
 *   y = x + MLP(h) + p_e * Expert_e(h),
 * MLP and every expert being GeLU FFNs of the layer's shape (W1 [F][H] + b1,
 * GeLU, W2 [H][F] + b2) and W_g [E][H] having no bias.  The expert of each
 * row is chosen on the device (no host synchronisation). */
typedef struct ds_moe_ffn ds_moe_ffn;
typedef struct {
  int hidden;          /* H, a multiple of 256                          */
  int ffn;             /* F, a multiple of 256 (MLP and experts)        */
  int experts;         /* E, 1 .. 1024                                  */
  float ln_eps;        /* LayerNorm epsilon                             */
  ds_dtype act_dtype;  /* DS_F16 or DS_BF16: activations and weights    */
} ds_moe_config;
/* Device pointers (act_dtype): ln2_g/ln2_b [H]; w_gate [E][H]; the dense MLP
 * w_fc1 [F][H], b_fc1 [F], w_fc2 [H][F], b_fc2 [H]; the experts stacked:
 * we_fc1 [E][F][H], be_fc1 [E][F], we_fc2 [E][H][F], be_fc2 [E][H].  Stored,
 * not copied: keep them alive and unchanged until ds_moe_ffn_destroy. */
typedef struct {
  const void *ln2_g, *ln2_b, *w_gate, *w_fc1, *b_fc1, *w_fc2, *b_fc2;
  const void *we_fc1, *be_fc1, *we_fc2, *be_fc2;
} ds_moe_weights;

DS_API ds_status ds_moe_ffn_create(const ds_moe_config* cfg, const ds_moe_weights* w, ds_moe_ffn** out);
DS_API ds_status ds_moe_ffn_destroy(ds_moe_ffn* moe);
/* Workspace bytes for `rows` rows (1 .. 4096); 0 for invalid arguments.  The
 * workspace is zero-filled once (ds_workspace_init) before first use. */
DS_API size_t ds_moe_ffn_workspace_bytes(const ds_moe_ffn* moe, int rows);
/* y = x + MLP(h) + p_e Expert_e(h) for x_in [rows][H] -> x_out [rows][H]
 * (act_dtype, not aliasing).  expert_out: optional DEVICE int32 [rows]
 * receiving each row's expert.  Asynchronous on `stream`: 4 + 2 rows kernels
 * (row LayerNorm, gate, dense MLP up / down, per row the chosen expert's
 * up / down), the device status flags in the workspace as for a layer. */
DS_API ds_status ds_moe_ffn_forward(ds_moe_ffn* moe, const void* x_in, void* x_out, int rows,
                                    int32_t* expert_out, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Tensor-sliced (Megatron-style) layer.  [P1] §3.2: the Attn and FF blocks
 * of a layer are split across GPUs in the Megatron-LM manner, so each block
 * ends in one cross-GPU all-reduce; §3.1, second fusion principle: every
 * all-reduce is a fusion boundary; the page's injection-policy passage: the
 * attention output GEMM and the layer output GEMM are the two linear layers
 * whose partial results are reduced across ranks.  The page gives no
 * formula; the split implemented, for W ranks (Hl = H/W, Fl = F/W, rank r):
 *   - rank r owns heads r*nh/W .. (r+1)*nh/W-1: their q, k and v rows of
 *     W_qkv / b_qkv, their KV caches, and columns r*Hl .. (r+1)*Hl-1 of W_o;
 *   - rank r owns FFN features r*Fl .. (r+1)*Fl-1: those rows of W_1 / b_1
 *     and those columns of W_2;
 *   - LayerNorm parameters are replicated; b_o, b_fc2 and the residuals are
 *     added by rank 0 only, inside its partial sums.
 * One layer step, on every rank, around two all-reduces (sum, fp32) that
 * the caller performs with its collective library (NCCL, torch.distributed):
 *   ds_tp_attention_partial   x1_r = [r==0](x + b_o) + o_r W_o[:, cols_r]^T
 *                             (LayerNorm1 + QKV of the rank's heads + KV
 *                             append + attention + O-proj, 4 kernels)
 *   all-reduce                x1 = sum over ranks of x1_r
 *   ds_tp_ffn_partial         y_r = [r==0](x1 + b_fc2)
 *                                   + GeLU(LN2(x1) W_1[rows_r]^T + b_1[rows_r]) W_2[:, rows_r]^T
 *                             (LayerNorm2 + FFN-up + GeLU + FFN-down, 3 kernels)
 *   all-reduce                y = sum over ranks of y_r
 *   ds_tp_finish              x_out = y in the activation dtype (1 kernel)
 * The partial sums are written by the epilogues of the two reduced GEMMs
 * (the reduction boundary), in fp32, so the all-reduce is the only step
 * between the fused regions.  fp16 / bf16 weights only (the tensor-core tile
 * kernels run every GEMM, at any row count 1..4096).  No device-to-device
 * traffic happens inside the library. */
typedef struct ds_tp_layer ds_tp_layer;
typedef struct {
  ds_layer_config layer; /* the FULL layer: hidden H, heads nh, ffn F, ln_eps,
                          * act_dtype; weight_dtype == act_dtype (fp16 / bf16) */
  int tp_size;           /* W, 1 .. 64, dividing nh; H/W and F/W multiples of 128 */
  int tp_rank;           /* r, 0 .. W-1 */
} ds_tp_config;

/* Where a rank's weights come from in the full layer: block i copies rows
 * src_row .. src_row+rows-1, columns src_col .. src_col+cols-1 of the full
 * matrix (row pitch src_cols elements) to rows dst_row .. dst_row+rows-1 of
 * the rank's matrix (row pitch cols elements).  Vectors are one-column
 * matrices.  Matrices not listed (LayerNorm parameters, b_o, b_fc2) are
 * replicated. */
typedef enum { DS_TP_W_QKV = 0, DS_TP_B_QKV = 1, DS_TP_W_O = 2, DS_TP_W_FC1 = 3,
               DS_TP_B_FC1 = 4, DS_TP_W_FC2 = 5 } ds_tp_matrix;
typedef struct {
  int matrix;    /* ds_tp_matrix */
  int src_row, src_col, rows, cols, src_cols, dst_row;
} ds_tp_block;

/* HOST only, no device needed: writes the rank's blocks (10: three each for
 * w_qkv and b_qkv, one for each other sliced matrix) to out[0 .. cap-1] and
 * returns their number, or -1 for an invalid config (ds_last_error says why)
 * or cap < 10. */
DS_API int ds_tp_shard_blocks(const ds_tp_config* cfg, ds_tp_block* out, int cap);
/* Copies the rank's slices of the FULL layer weights `full` (host or device
 * memory, [out][in] as for ds_layer_create) into the caller's buffers
 * `shard` (device memory, shapes: w_qkv [3Hl][H], b_qkv [3Hl], w_o [H][Hl],
 * w_fc1 [Fl][H], b_fc1 [Fl], w_fc2 [H][Fl]; only these six fields are
 * written, the others are ignored).  Asynchronous on `stream`
 * (cudaMemcpy2DAsync per block); the full weights must stay valid until the
 * stream reaches this point. */
DS_API ds_status ds_tp_shard_weights(const ds_tp_config* cfg, const ds_layer_weights* full,
                                     const ds_layer_weights* shard, void* stream);
/* The rank's layer over its shard: `w` holds the rank's device matrices in
 * the shapes above, and the replicated ln1_g, ln1_b, b_o, ln2_g, ln2_b,
 * b_fc2 [H] (b_o and b_fc2 are read on rank 0 only); s_* are ignored.
 * Stored, not copied. */
DS_API ds_status ds_tp_layer_create(const ds_tp_config* cfg, const ds_layer_weights* w, ds_tp_layer** out);
DS_API ds_status ds_tp_layer_destroy(ds_tp_layer* layer);
/* Workspace bytes for batch x new_tokens rows (1 .. 4096 rows); 0 for
 * invalid arguments.  Zero-filled once (ds_workspace_init) before first use;
 * one workspace serves the three calls of a step. */
DS_API size_t ds_tp_layer_workspace_bytes(const ds_tp_layer* layer, int batch, int new_tokens);
/* x_in [B][T][H] act dtype -> x1_part [B*T][H] fp32 (this rank's share of
 * x1).  k_cache / v_cache: the rank's caches [B][nh/W][max_len][d]; the new
 * keys and values are written at past_len[b] .. past_len[b]+T-1 as for
 * ds_layer_forward (past_len is not advanced). */
DS_API ds_status ds_tp_attention_partial(ds_tp_layer* layer, const void* x_in, float* x1_part, int batch,
                                         int new_tokens, void* k_cache, void* v_cache, int max_len,
                                         const int32_t* past_len, void* workspace, size_t ws_bytes,
                                         void* stream);
/* x1 [rows][H] fp32 (the all-reduced x1) -> y_part [rows][H] fp32 (this
 * rank's share of the layer output).  x1 and y_part must not alias. */
DS_API ds_status ds_tp_ffn_partial(ds_tp_layer* layer, const float* x1, float* y_part, int rows,
                                   void* workspace, size_t ws_bytes, void* stream);
/* y [rows][H] fp32 (the all-reduced layer output) -> x_out [rows][H] in the
 * activation dtype (round to nearest even). */
DS_API ds_status ds_tp_finish(ds_tp_layer* layer, const float* y, void* x_out, int rows, void* stream);

/* Device-side status flags recorded in the workspace. */
#define DS_DEVFLAG_CACHE_OVERFLOW 0x1  /* past_len[b] + T > max_len for some row */
#define DS_DEVFLAG_WAIT_TIMEOUT 0x2    /* an in-kernel pipeline wait gave up (outputs invalid) */
#define DS_DEVFLAG_BOUNDS 0x4          /* diagnostic build only (DS_DEBUG_BOUNDS defined, i.e.
                                        * libdslayer_debug_bounds.so): a kernel found an index
                                        * outside its buffer and skipped the access (outputs
                                        * invalid); normal builds compile the checks away */

/* Copies the workspace status word to *flags_out, clears it, and synchronises
 * `stream`.  Returns DS_ERR_DEVICE when a flag was set, DS_OK otherwise. */
DS_API ds_status ds_workspace_status(void* workspace, uint32_t* flags_out, void* stream);

/* Self-test of the device-side failure detection (the pages describe no such
 * mechanism; it is a property of this library).  Every wait inside the
 * kernels is bounded: when it runs out, the kernel records
 * DS_DEVFLAG_WAIT_TIMEOUT in the workspace status word and returns instead of
 * hanging.  This call launches one thread that waits, with the same routine,
 * on a barrier nothing arrives on, for budget_us microseconds (1 .. 10^6);
 * the wait runs out and sets the flag in `workspace` (any workspace, 256-byte
 * aligned), which ds_workspace_status then reports.  Asynchronous on
 * `stream`; the context stays usable. */
DS_API ds_status ds_selftest_wait_timeout(void* workspace, uint32_t budget_us, void* stream);

/* Number of kernels this library has launched (a graph replay counts every
 * kernel node in the graph) since the process started. */
DS_API uint64_t ds_launch_count(void);

DS_API const char* ds_status_string(ds_status s);
/* Detail of the last failure on the calling thread ("" if none). */
DS_API const char* ds_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DS_LAYER_H */
