// Region 2: decode attention over the KV cache with scale, causal mask and
// softmax fused; the key splits of one head are merged on chip.
//
// Pages cited:
//   [P1] "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、算子融合推理内核
//        与 MoQ 量化支持", §3.2 region 2: transform and attention merged, the
//        head-split layout read through index arithmetic ("implicit matrix
//        transformation") instead of being materialised; §3.3: shared memory
//        between reductions, warp-level reductions of partial results.
//   [P3] "DeepSpeed MoE 大规模稀疏模型推理实战指南：并行切分、PR-MoE 优化与
//        init_inference 全解析", table "推理配置参数详解": triangular_masking,
//        the causal mask.
//
// What it computes, per sequence b, new token t and head h:
//   s_j = q . k_j / sqrt(d) for j <= past_len[b] + t;  p = softmax(s);  o = sum_j p_j v_j.
//
// GB300 design (not the pages'): a layer has only nh (20-40) heads at batch
// 1, far fewer than 152 SMs, so each (b, h) is split along the keys over a
// thread-block cluster of `nsplit` (<= 8) CTAs, as many as keep the grid
// within one CTA per SM; such a grid asks for more than half of an SM's
// shared memory, so that no two CTAs share an SM (the block scheduler would
// otherwise pack them onto a fraction of the SMs).  With more (b, h) pairs
// than one wave of resident CTAs holds, the keys are split to pack the waves
// (attn_configure).  Before griddepcontrol.wait a
// CTA copies the cached K and V rows of its keys that the previous kernel
// does not write (positions < past_len) into shared memory with two TMA bulk
// copies, so that once the QKV kernel completes only q and the new rows come
// from global memory.  A key's d values are spread over d/8 lanes (16-byte
// loads) and reduced with warp shuffles; each lane group keeps a running
// max / sum / p.V (online softmax, log2 domain): one pass over the keys, no
// score buffer.  The groups of a CTA merge in shared memory; every CTA of the
// cluster then stores its (O, M, L) into rank 0's shared memory (distributed
// shared memory), and rank 0 merges them locally: no global partials, no
// atomics, no remote loads.
#include <math.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kAttnThreads = 256;
constexpr int kAttnMaxSplit = 8;  // portable cluster size

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                   : "memory");
}

// Stores a float into the shared memory of CTA `rank` of this cluster, at the
// same offset as `local` in this CTA.
__device__ __forceinline__ void st_cluster(float* local, uint32_t rank, float v) {
  uint32_t addr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(addr) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(addr), "f"(v) : "memory");
}

// Shared-memory carve-up (floats, then the staged K and V rows, then one
// mbarrier): og [KPI][D] per-group p.V, mg / lg [KPI] per-group max and sum,
// part [D + 2] this CTA's (O, M, L), mrg [8][D + 2] the cluster's partials
// (used in rank 0), Ks / Vs [stage_keys][D].
__host__ __device__ inline size_t attn_floats(int D) {
  const int kpi = kAttnThreads / (D / 8);
  return (size_t)kpi * D + 2 * kpi + (size_t)(1 + kAttnMaxSplit) * (D + 2);
}
__host__ __device__ inline size_t attn_stage_offset(int D) { return (attn_floats(D) * 4 + 127) & ~(size_t)127; }

// Keys [j0, j1) of this CTA (relative to its first key), NBX per key group
// and pass, folded into the group's running max m, sum l and p.V o8 (log2
// domain).  Rows j < n_sm come from shared memory (Ks, Vs), the others from
// global memory (Kg, Vg).
template <typename ACT, int D, int NBX>
__device__ __forceinline__ void attn_keys(int j0, int j1, int kr, int kq, int n_sm, const ACT* Ks, const ACT* Vs,
                                          const ACT* Kg, const ACT* Vg, const float (&qv)[8], float& m, float& l,
                                          float (&o8)[8]) {
  constexpr int LPK = D / 8;
  constexpr int KPI = kAttnThreads / LPK;
  for (int base = j0; base < j1; base += NBX * KPI) {
    uint4 kk[NBX], vv[NBX];
#pragma unroll
    for (int i = 0; i < NBX; ++i) {
      const int j = base + i * KPI + kr;
      if (j < j1) {
        if (j < n_sm) {
          kk[i] = lds_u128(smem_u32(Ks + (size_t)j * D + kq * 8));
          vv[i] = lds_u128(smem_u32(Vs + (size_t)j * D + kq * 8));
        } else {
          kk[i] = *reinterpret_cast<const uint4*>(Kg + (size_t)j * D + kq * 8);
          vv[i] = *reinterpret_cast<const uint4*>(Vg + (size_t)j * D + kq * 8);
        }
      } else {
        kk[i] = make_uint4(0u, 0u, 0u, 0u);
        vv[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float s[NBX];
    float bm = -INFINITY;
#pragma unroll
    for (int i = 0; i < NBX; ++i) {
      const uint32_t kw[4] = {kk[i].x, kk[i].y, kk[i].z, kk[i].w};
      float d = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 f = Act<ACT>::unpack2(kw[w]);
        d += f.x * qv[2 * w] + f.y * qv[2 * w + 1];
      }
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      s[i] = (base + i * KPI + kr < j1) ? d : -INFINITY;
      bm = fmaxf(bm, s[i]);
    }
    const float m_new = fmaxf(m, bm);
    const float scale = (m_new == -INFINITY) ? 1.f : exp2f(m - m_new);
    l *= scale;
#pragma unroll
    for (int i = 0; i < 8; ++i) o8[i] *= scale;
#pragma unroll
    for (int i = 0; i < NBX; ++i) {
      const float p = (s[i] == -INFINITY) ? 0.f : exp2f(s[i] - m_new);
      l += p;
      const uint32_t vw[4] = {vv[i].x, vv[i].y, vv[i].z, vv[i].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 f = Act<ACT>::unpack2(vw[w]);
        o8[2 * w] += p * f.x;
        o8[2 * w + 1] += p * f.y;
      }
    }
    m = m_new;
  }
}

template <typename ACT, int D>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
  constexpr int LPK = D / 8;               // lanes per key (16 B each)
  constexpr int KPI = kAttnThreads / LPK;  // key groups per CTA (keys per pass)
  constexpr int NB = 8;                    // passes whose K and V loads are in flight together
  extern __shared__ __align__(128) float sm[];
  float* og = sm;
  float* mg = og + KPI * D;
  float* lg = mg + KPI;
  float* part = lg + KPI;
  float* mrg = part + (D + 2);
  ACT* Ks = reinterpret_cast<ACT*>(reinterpret_cast<unsigned char*>(sm) + attn_stage_offset(D));
  ACT* Vs = Ks + (size_t)a.stage_keys * D;
  uint64_t* bar = reinterpret_cast<uint64_t*>(Vs + (size_t)a.stage_keys * D);

  const int sp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;  // sp = rank in the cluster
  const int nsplit = gridDim.x;
  const int tid = threadIdx.x;
  const int kq = tid % LPK, kr = tid / LPK;

  // past_len is only changed by the last kernel of a stack step, which has
  // completed before this step's first kernel starts (that one is launched
  // without programmatic overlap), so it may be read before the wait.
  const int past = a.past_len[b];
  int S_all = past + a.T;
  if (S_all > a.max_len) S_all = a.max_len;
  if (S_all < 1) S_all = 1;
  const int chunk = (S_all + nsplit - 1) / nsplit;
  const int lo = sp * chunk;
  const int hi = min(S_all, lo + chunk);
  const size_t head_row0 = ((size_t)b * a.heads + h) * a.max_len;
  const ACT* Kc = static_cast<const ACT*>(a.k_cache) + head_row0 * D;
  const ACT* Vc = static_cast<const ACT*>(a.v_cache) + head_row0 * D;
  // Keys [lo, lo + n_st) are cached rows nobody writes during this step.
  const int n_st = max(0, min(min(hi, past) - lo, a.stage_keys));

  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0 && n_st > 0) {
    const uint32_t bytes = (uint32_t)(n_st * D * sizeof(ACT));
    const uint64_t pol = l2_evict_first_policy();
    mbar_arrive_expect_tx(smem_u32(bar), 2 * bytes);
    bulk_g2s(smem_u32(Ks), Kc + (size_t)lo * D, bytes, smem_u32(bar), pol);
    bulk_g2s(smem_u32(Vs), Vc + (size_t)lo * D, bytes, smem_u32(bar), pol);
    // rows past the staging budget: into L2
    const int pe = min(hi, past);
    if (pe > lo + n_st) {
      prefetch_l2_bulk(Kc + (size_t)(lo + n_st) * D, (uint32_t)((pe - lo - n_st) * D * sizeof(ACT)));
      prefetch_l2_bulk(Vc + (size_t)(lo + n_st) * D, (uint32_t)((pe - lo - n_st) * D * sizeof(ACT)));
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  // If the staging copy does not complete within the wait budget (the flag is
  // then set), this thread reads those rows from global memory instead of
  // shared memory, and the CTA waits again for the copy before it exits.
  const bool staged = (n_st == 0) || mbar_wait(smem_u32(bar), 0, a.status);
  const int n_sm = staged ? n_st : 0;  // rows read from shared memory

  for (int t = 0; t < a.T; ++t) {
    const int St = min(past + t + 1, S_all);
    int n_keys = max(0, min(hi, St) - lo);
    if (!ds_in_bounds(lo + n_keys <= a.max_len && b < a.B && h < a.heads, a.status)) n_keys = 0;
    float qv[8];
    {
      const float* qp = a.q + (size_t)(b * a.T + t) * a.H + h * D + kq * 8;
      const float4 q0 = *reinterpret_cast<const float4*>(qp);
      const float4 q1 = *reinterpret_cast<const float4*>(qp + 4);
      qv[0] = q0.x; qv[1] = q0.y; qv[2] = q0.z; qv[3] = q0.w;
      qv[4] = q1.x; qv[5] = q1.y; qv[6] = q1.z; qv[7] = q1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] *= a.scale_log2;
    }
    float m = -INFINITY, l = 0.f;
    float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // whole passes of NB keys per group, then the remainder two at a time
    const int n_full = n_keys - n_keys % (NB * KPI);
    attn_keys<ACT, D, NB>(0, n_full, kr, kq, n_sm, Ks, Vs, Kc + (size_t)lo * D, Vc + (size_t)lo * D, qv, m, l, o8);
    attn_keys<ACT, D, 2>(n_full, n_keys, kr, kq, n_sm, Ks, Vs, Kc + (size_t)lo * D, Vc + (size_t)lo * D, qv, m, l, o8);
    // Merge the key groups of this CTA, then push (O, M, L) to rank 0.
#pragma unroll
    for (int i = 0; i < 8; ++i) og[kr * D + kq * 8 + i] = o8[i];
    if (kq == 0) {
      mg[kr] = m;
      lg[kr] = l;
    }
    __syncthreads();
    if (tid < D) {
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < KPI; ++r) M = fmaxf(M, mg[r]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < KPI; ++r) {
          const float w = exp2f(mg[r] - M);
          L += w * lg[r];
          O += w * og[r * D + tid];
        }
      }
      float* slot = mrg + sp * (D + 2);
      st_cluster(slot + tid, 0, O);
      if (tid == 0) {
        st_cluster(slot + D, 0, M);
        st_cluster(slot + D + 1, 0, L);
      }
    }
    cluster_sync_all();  // every CTA's partial is in rank 0; og/mg/lg free again
    if (sp == 0 && tid < D) {
      float M = -INFINITY;
      for (int r = 0; r < nsplit; ++r) M = fmaxf(M, mrg[r * (D + 2) + D]);
      float L = 0.f, O = 0.f;
      for (int r = 0; r < nsplit; ++r) {
        const float mr = mrg[r * (D + 2) + D];
        const float w = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
        L += w * mrg[r * (D + 2) + D + 1];
        O += w * mrg[r * (D + 2) + tid];
      }
      const float o = O / L;
      const size_t oi = (size_t)(b * a.T + t) * a.H + h * D + tid;
      if (!ds_in_bounds(oi < (size_t)a.B * a.T * a.H, a.status)) {
        // (debug builds: an output index outside the buffer; skipped)
      } else if (a.out_hi != nullptr) {  // tensor-core operand: hi (and lo for bf16)
        const ACT hv = Act<ACT>::from_f(o);
        static_cast<ACT*>(a.out_hi)[oi] = hv;
        if (a.out_lo != nullptr) static_cast<ACT*>(a.out_lo)[oi] = Act<ACT>::from_f(o - Act<ACT>::to_f(hv));
      } else {
        a.out[oi] = o;
      }
    }
    if (t + 1 < a.T) cluster_sync_all();  // rank 0 has read the partials before they are overwritten
  }
  if (!staged) mbar_wait(smem_u32(bar), 0, a.status);  // no copy may land after the CTA exits
}

size_t attn_smem_bytes(int head_dim, int stage_keys) {
  return attn_stage_offset(head_dim) + (size_t)2 * stage_keys * head_dim * 2 + 16;
}

// CTAs of the decode attention (activation ak, head size D) with `smem`
// bytes of dynamic shared memory that one SM holds at once; 0 if unknown.
// Cached: the launch shape is worked out per call.
static int attn_ctas_per_sm(ActKind ak, int D, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_tuple(dev, (int)ak, D, smem);
  std::lock_guard<std::mutex> lk(mu);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const void* k = nullptr;
  if (ak == ActKind::F16) k = D == 64 ? (const void*)attn_decode_kernel<__half, 64> : (const void*)attn_decode_kernel<__half, 128>;
  else k = D == 64 ? (const void*)attn_decode_kernel<__nv_bfloat16, 64> : (const void*)attn_decode_kernel<__nv_bfloat16, 128>;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kAttnThreads, smem) != cudaSuccess) {
    n = 0;
    (void)cudaGetLastError();
  }
  cache[key] = n;
  return n;
}

// Launch shape of the decode attention for a.B, a.heads, a.max_len and
// a.head_dim: nsplit CTAs (one cluster) per (b, h), as many as keep the
// grid within one CTA per SM (at most 8, at least ~32 keys each); such a
// grid stages up to all of a split's keys and asks for more than half of an
// SM's shared memory so that the CTAs spread over the SMs.  Larger grids
// (many sequences) take a 48 KB staging budget, several CTAs sharing an SM,
// and, past one wave of resident CTAs, as many splits per (b, h) as pack
// the CTAs into whole waves: with 640 (b, h) pairs and 296 CTAs resident at
// once, one CTA per pair leaves the third wave three-quarters empty (72 % of
// the slots used), three splits use 93 % of them.
void attn_configure(AttnArgs& a, ActKind ak, int num_sms, int max_smem) {
  const int bh = a.B * a.heads, D = a.head_dim;
  int ns = num_sms / (bh > 0 ? bh : 1);
  if (ns > kAttnMaxSplit) ns = kAttnMaxSplit;
  const int cap = a.max_len / 32;
  if (ns > cap) ns = cap;
  if (ns < 1) ns = 1;
  const bool spread = (long long)bh * ns <= num_sms;
  const size_t fixed = attn_smem_bytes(D, 0);
  const size_t budget = spread ? ((size_t)max_smem > fixed + 1024 ? (size_t)max_smem - fixed - 1024 : 0) : 48 * 1024;
  auto stage_keys = [&](int n) {
    int sk = (int)(budget / ((size_t)4 * D));  // K and V rows of 16-bit values
    const int per_split = (a.max_len + n - 1) / n;
    return sk > per_split ? per_split : sk;
  };
  if (!spread) {
    const int per_sm = attn_ctas_per_sm(ak, D, attn_smem_bytes(D, stage_keys(ns)));
    const long long slots = (long long)per_sm * num_sms;
    // only past one wave, and only into splits of 256 keys or more (shorter
    // ones, or splitting a grid that fits at once, measured slower)
    if (per_sm > 0 && bh > slots) {
      auto packing = [&](int n) {
        const long long c = (long long)bh * n, waves = (c + slots - 1) / slots;
        return (double)c / (double)(waves * slots);
      };
      const int cap_w = a.max_len / 256;
      const int nmax = cap_w < kAttnMaxSplit ? cap_w : kAttnMaxSplit;
      int best = ns;
      for (int n = ns + 1; n <= nmax && packing(best) < 0.9; ++n)
        if (packing(n) > packing(best) + 0.05) best = n;
      ns = best;
    }
  }
  const int sk = stage_keys(ns);
  size_t smem = attn_smem_bytes(D, sk);
  if (spread) {
    const size_t half = (size_t)max_smem / 2 + 1024;
    if (smem < half && half <= (size_t)max_smem) smem = half;
  }
  a.nsplit = ns;
  a.stage_keys = sk;
  a.smem = smem;
}

cudaError_t launch_attention(ActKind ak, const AttnArgs& a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.heads, a.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = a.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (ak == ActKind::F16) {
    if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__half, 64>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__half, 128>, a);
  } else {
    if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__nv_bfloat16, 64>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_decode_kernel<__nv_bfloat16, 128>, a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t prepare_attention_kernels(int max_smem) {
  cudaError_t e = cudaSuccess;
#define DS_PREP_ATTN(T, D)                                                                            \
  if (e == cudaSuccess)                                                                               \
    e = cudaFuncSetAttribute(attn_decode_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             max_smem)
  DS_PREP_ATTN(__half, 64);
  DS_PREP_ATTN(__half, 128);
  DS_PREP_ATTN(__nv_bfloat16, 64);
  DS_PREP_ATTN(__nv_bfloat16, 128);
#undef DS_PREP_ATTN
  return e;
}

}  // namespace ds
