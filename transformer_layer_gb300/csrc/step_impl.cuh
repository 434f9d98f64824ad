// Persistent decode-step kernel: every layer of a stack, all five phases,
// in one cooperative launch with one CTA per SM.
//
// Page cited as [P1]: "DeepSpeed Inference 内核优化深度解析：多 GPU 自适应并行、
// 算子融合推理内核与 MoQ 量化支持", §3.2 (the four fusion regions, each phase
// below is one of them or half of region 3), §3.1 (fuse at the reduction
// boundaries; CTAs meet only through memory, with block-level syncs), §3.3.
// The generation loop calls every layer once per token; this kernel is one
// such call for all layers of the stack.
//
// GB300 design (not the pages'): separate kernels each pay a ramp-up (first
// weights still in flight) and a drain; at batch 1 those bubbles cost about a
// third of the step.  Here the same CTA roles as the region kernels (copy
// warps, MMA warps, epilogue warp) run all phases in sequence.  Between
// phases the MMA warps wait at a grid-wide barrier for the previous phase's
// results, but the copy warps never wait for activations: they stream the
// next phases' weights into the ring straight through the barriers and
// through attention, so HBM does not idle at phase boundaries.  Attention runs
// on the MMA warps (two groups of four warps) while the ring fills with the
// O-proj weights.  Every wait is bounded in wall-clock time.
#pragma once

#include "gemv_impl.cuh"

namespace ds {

constexpr int kStepThreads = kGemvThreads;
// Per-group attention scratch (floats): og [KPI][d], mg, lg [KPI], flag; two groups.
constexpr int kAttnGroupFloats = 16 * 64 + 2 * 16 + 32;  // the larger of d = 64 / 128 (1024 + 32 + pad)
constexpr int kAttnScratchFloats = 2 * kAttnGroupFloats;
constexpr int kBarAttn = 10;  // 10, 11: the two attention groups (128 threads each)
// Chunks of the next phase each CTA asks L2 to prefetch at the end of a phase
// (x 152 CTAs x 16 KB ~ 39 MB, well inside the 129 MB L2).
constexpr int kStepL2Lookahead = 16;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// MMA warps wait until `target` arrivals have reached the grid barrier (all
// CTAs finished the previous phase); one thread polls, bounded in time.
__device__ __forceinline__ void step_wait(const unsigned* bar, unsigned target, unsigned* status, bool& dead) {
  if (threadIdx.x == 0 && !dead) {
    if (ld_acquire_u32(bar) < target) {
      const unsigned long long t0 = global_ns();
      for (unsigned i = 1;; ++i) {
        if (ld_acquire_u32(bar) >= target) break;
        if ((i & 15u) == 0 && global_ns() - t0 > kWaitBudgetNs) {
          atomicOr(status, kFlagWaitTimeout);
          dead = true;
          break;
        }
        __nanosleep(64);
      }
    }
  }
  bar_sync(kBarStage, kProducers * 32);
}

// The epilogue warp's wait for the same barrier (lane 0 polls).
__device__ __forceinline__ void step_wait_warp(const unsigned* bar, unsigned target, unsigned* status,
                                               bool& dead) {
  if ((threadIdx.x & 31) == 0 && !dead) {
    if (ld_acquire_u32(bar) < target) {
      const unsigned long long t0 = global_ns();
      for (unsigned i = 1;; ++i) {
        if (ld_acquire_u32(bar) >= target) break;
        if ((i & 15u) == 0 && global_ns() - t0 > kWaitBudgetNs) {
          atomicOr(status, kFlagWaitTimeout);
          dead = true;
          break;
        }
        __nanosleep(64);
      }
    }
  }
  __syncwarp();
}

// One arrival at the grid barrier (the caller has fenced its stores).  The
// last arrival of the whole step returns the counter to zero for the next
// launch.
__device__ __forceinline__ void step_arrive(unsigned* bar, unsigned total) {
  const unsigned old = atomicAdd(bar, 1u);
  if (old == total - 1) atomicExch(bar, 0u);
}

// Region arguments of phase `r` (0 QKV, 1 O-proj, 2 FFN-up, 3 FFN-down) of layer l.
__device__ __forceinline__ RegionArgs step_region_args(const StepArgs& s, int l, int r) {
  RegionArgs a;
  const StepLayer& ly = s.layer[l];
  const size_t act_bytes = (size_t)s.B * s.H * 2;
  const void* x_l = (l == 0) ? s.x_in : static_cast<const void*>(s.act + ((l - 1) & 1) * act_bytes);
  a.M = s.B;
  a.B = s.B;
  a.T = 1;
  a.partials = s.partials;
  a.counters = s.counters;
  a.eps = s.eps;
  a.status = s.status;
  a.H = s.H;
  a.W = ly.w[r];
  a.Wscale = ly.sc[r];
  a.qgroup = s.qgroup[r];
  a.tmap_w = ly.tmap_w[r];
  a.tmap_s = ly.tmap_s[r];
  a.bias = ly.bias[r];
  if (r == 0) {
    a.N = 3 * s.H;
    a.K = s.H;
    a.x_act = x_l;
    a.ln_g = ly.ln1_g;
    a.ln_b = ly.ln1_b;
    a.stats_in = (l == 0) ? nullptr : s.stats_b;
    a.out_f32 = s.q;
    a.k_cache = ly.kc;
    a.v_cache = ly.vc;
    a.heads = s.heads;
    a.head_dim = s.head_dim;
    a.max_len = s.max_len;
    a.past_len = s.seq;
  } else if (r == 1) {
    a.N = s.H;
    a.K = s.H;
    a.x_f32 = s.o;
    a.out_f32 = s.x1;
    a.resid_act = x_l;
    a.stats_out = s.stats_a;
  } else if (r == 2) {
    a.N = s.F;
    a.K = s.H;
    a.x_f32 = s.x1;
    a.ln_g = ly.ln2_g;
    a.ln_b = ly.ln2_b;
    a.stats_in = s.stats_a;
    a.out_f32 = s.g;
  } else {
    a.N = s.H;
    a.K = s.F;
    a.x_f32 = s.g;
    a.resid_f32 = s.x1;
    a.out_act = (l == s.L - 1) ? s.x_out : static_cast<void*>(s.act + (l & 1) * act_bytes);
    a.stats_out = (l == s.L - 1) ? nullptr : s.stats_b;
  }
  return a;
}

// L2 prefetch of the cached K/V rows of this group's attention items (they
// are not written during the step), issued before the barrier wait.
template <typename ACT>
__device__ void step_attn_prefetch(const StepArgs& s, int l, int group, int gt) {
  if (gt != 0) return;
  const int D = s.head_dim, ns = s.nsplit;
  const int items = s.B * s.heads * ns;
  for (int it = blockIdx.x * 2 + group; it < items; it += 2 * gridDim.x) {
    const int b = it / (s.heads * ns), rem = it - b * s.heads * ns, h = rem / ns, sp = rem - h * ns;
    const int past = s.seq[b];
    int S_all = min(past + 1, s.max_len);
    if (S_all < 1) S_all = 1;
    const int chunk = (S_all + ns - 1) / ns, lo = sp * chunk, pe = min(lo + chunk, past);
    if (pe > lo) {
      const size_t row0 = ((size_t)b * s.heads + h) * s.max_len;
      const ACT* Kc = static_cast<const ACT*>(s.layer[l].kc) + row0 * D;
      const ACT* Vc = static_cast<const ACT*>(s.layer[l].vc) + row0 * D;
      prefetch_l2_bulk(Kc + (size_t)lo * D, (uint32_t)((pe - lo) * D * sizeof(ACT)));
      prefetch_l2_bulk(Vc + (size_t)lo * D, (uint32_t)((pe - lo) * D * sizeof(ACT)));
    }
  }
}

// Attention phase of layer l on one group of 4 MMA warps (128 threads).
// Items are (b, h, key split); each writes its (O, M, L) partial, and the
// last split of a head to finish (arrival counter, no waiting) merges them.
template <typename ACT, int D>
__device__ void step_attention(const StepArgs& s, int l, int group, int gt, float* scratch) {
  constexpr int LPK = D / 8;     // lanes per key
  constexpr int KPI = 128 / LPK; // key groups per 128 threads
  constexpr int NB = 8;          // passes with K and V loads in flight together
  float* og = scratch;           // [KPI][D]
  float* mg = og + KPI * D;      // [KPI]
  float* lg = mg + KPI;          // [KPI]
  int* flag = reinterpret_cast<int*>(lg + KPI);
  const int bar_id = kBarAttn + group;
  const int kq = gt % LPK, kr = gt / LPK;
  const int ns = s.nsplit, H = s.H;
  const int items = s.B * s.heads * ns;
  const StepLayer& ly = s.layer[l];
  for (int it = blockIdx.x * 2 + group; it < items; it += 2 * gridDim.x) {
    const int b = it / (s.heads * ns), rem = it - b * s.heads * ns, h = rem / ns, sp = rem - h * ns;
    const int past = s.seq[b];
    int S_all = min(past + 1, s.max_len);
    if (S_all < 1) S_all = 1;
    const int chunk = (S_all + ns - 1) / ns;
    const int lo = sp * chunk;
    const int n_keys = max(0, min(S_all, lo + chunk) - lo);
    const size_t row0 = ((size_t)b * s.heads + h) * s.max_len;
    const ACT* Kc = static_cast<const ACT*>(ly.kc) + row0 * D;
    const ACT* Vc = static_cast<const ACT*>(ly.vc) + row0 * D;
    float qv[8];
    {
      const float* qp = s.q + (size_t)b * H + h * D + kq * 8;
      const float4 q0 = *reinterpret_cast<const float4*>(qp);
      const float4 q1 = *reinterpret_cast<const float4*>(qp + 4);
      qv[0] = q0.x; qv[1] = q0.y; qv[2] = q0.z; qv[3] = q0.w;
      qv[4] = q1.x; qv[5] = q1.y; qv[6] = q1.z; qv[7] = q1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) qv[i] *= s.scale_log2;
    }
    float m = -INFINITY, lsum = 0.f;
    float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int base = 0; base < n_keys; base += NB * KPI) {
      uint4 kk[NB], vv[NB];
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const int j = base + i * KPI + kr;
        if (j < n_keys) {
          kk[i] = *reinterpret_cast<const uint4*>(Kc + (size_t)(lo + j) * D + kq * 8);
          vv[i] = *reinterpret_cast<const uint4*>(Vc + (size_t)(lo + j) * D + kq * 8);
        } else {
          kk[i] = make_uint4(0u, 0u, 0u, 0u);
          vv[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float sc[NB];
      float bm = -INFINITY;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const uint32_t kw[4] = {kk[i].x, kk[i].y, kk[i].z, kk[i].w};
        float d = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 f = Act<ACT>::unpack2(kw[w]);
          d += f.x * qv[2 * w] + f.y * qv[2 * w + 1];
        }
#pragma unroll
        for (int o = LPK / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        sc[i] = (base + i * KPI + kr < n_keys) ? d : -INFINITY;
        bm = fmaxf(bm, sc[i]);
      }
      const float m_new = fmaxf(m, bm);
      const float scale = (m_new == -INFINITY) ? 1.f : exp2f(m - m_new);
      lsum *= scale;
#pragma unroll
      for (int i = 0; i < 8; ++i) o8[i] *= scale;
#pragma unroll
      for (int i = 0; i < NB; ++i) {
        const float p = (sc[i] == -INFINITY) ? 0.f : exp2f(sc[i] - m_new);
        lsum += p;
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
    // merge this group's key groups, write the split's partial
#pragma unroll
    for (int i = 0; i < 8; ++i) og[kr * D + kq * 8 + i] = o8[i];
    if (kq == 0) {
      mg[kr] = m;
      lg[kr] = lsum;
    }
    bar_sync(bar_id, 128);
    float* part = s.attn_part + ((size_t)(b * s.heads + h) * ns) * (D + 2);
    if (gt < D) {
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < KPI; ++r) M = fmaxf(M, mg[r]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < KPI; ++r) {
          const float w = exp2f(mg[r] - M);
          L += w * lg[r];
          O += w * og[r * D + gt];
        }
      }
      part[sp * (D + 2) + gt] = O;
      if (gt == 0) {
        part[sp * (D + 2) + D] = M;
        part[sp * (D + 2) + D + 1] = L;
      }
    }
    __threadfence();
    bar_sync(bar_id, 128);
    if (gt == 0) *flag = (atomicAdd(&s.attn_cnt[b * s.heads + h], 1) == ns - 1);
    bar_sync(bar_id, 128);
    if (*flag) {
      __threadfence();
      if (gt < D) {
        float M = -INFINITY;
        for (int r = 0; r < ns; ++r) M = fmaxf(M, ld_cg(part + r * (D + 2) + D));
        float L = 0.f, O = 0.f;
        for (int r = 0; r < ns; ++r) {
          const float mr = ld_cg(part + r * (D + 2) + D);
          const float w = (mr == -INFINITY) ? 0.f : exp2f(mr - M);
          L += w * ld_cg(part + r * (D + 2) + D + 1);
          O += w * ld_cg(part + r * (D + 2) + gt);
        }
        s.o[(size_t)b * H + h * D + gt] = O / L;
      }
      if (gt == 0) s.attn_cnt[b * s.heads + h] = 0;
    }
    bar_sync(bar_id, 128);  // scratch and flag reused by the next item
  }
}

template <WKind WK, typename ACT, int NT>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(const __grid_constant__ StepArgs s) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const GemvSmem sm = gemv_carve<NT>(smem_raw, s.stages, s.SB, s.xs_cap, kAttnScratchFloats);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) gemv_init_ring(sm);
  __syncthreads();
  const unsigned G = gridDim.x;
  const unsigned total = 5u * (unsigned)s.L * G;  // arrivals in one step

  if (warp < kProducers) {
    // ---------------- MMA warps: GEMV phases and attention ----------------
    RingPos rp;
    int seg = 0;
    bool dead = false;
    unsigned p = 0;  // phase index
    const int group = warp >> 2, gt = tid & 127;
    for (int l = 0; l < s.L; ++l) {
      for (int r = 0; r < 5; ++r, ++p) {
        if (r == 1) step_attn_prefetch<ACT>(s, l, group, gt);
        if (p > 0) step_wait(s.grid_bar, p * G, s.status, dead);
        if (r == 1) {
          if (s.head_dim == 64)
            step_attention<ACT, 64>(s, l, group, gt, sm.attn + group * kAttnGroupFloats);
          else
            step_attention<ACT, 128>(s, l, group, gt, sm.attn + group * kAttnGroupFloats);
          __threadfence();
          bar_sync(kBarStage, kProducers * 32);
          if (tid == 0) step_arrive(s.grid_bar, total);
          continue;
        }
        const int reg = r == 0 ? 0 : r - 1;
        const RegionArgs a = step_region_args(s, l, reg);
        if (reg == 0) gemv_mma_phase<Region::LnQkv, WK, ACT, NT, 1>(a, s.plan[0], sm, rp, seg);
        else if (reg == 1) gemv_mma_phase<Region::OprojRes, WK, ACT, NT, 1>(a, s.plan[1], sm, rp, seg);
        else if (reg == 2) gemv_mma_phase<Region::FfnUp, WK, ACT, NT, 1>(a, s.plan[2], sm, rp, seg);
        else gemv_mma_phase<Region::FfnDown, WK, ACT, NT, 1>(a, s.plan[3], sm, rp, seg);
      }
    }
    gemv_mma_drain<NT>(seg);
  } else if (warp >= kTmaWarp0) {
    // ---------------- copy warps: every phase's weights, never waiting on activations ----------------
    RingPos rp;
    const uint64_t pol = l2_evict_first_policy();
    const int tw = warp - kTmaWarp0;
    for (int l = 0; l < s.L; ++l) {
      for (int reg = 0; reg < 4; ++reg) {
        const RegionArgs a = step_region_args(s, l, reg);
        if (reg == 0) gemv_tma_phase<Region::LnQkv, WK, ACT, NT>(a, s.plan[0], sm, rp, tw, pol);
        else if (reg == 1) gemv_tma_phase<Region::OprojRes, WK, ACT, NT>(a, s.plan[1], sm, rp, tw, pol);
        else if (reg == 2) gemv_tma_phase<Region::FfnUp, WK, ACT, NT>(a, s.plan[2], sm, rp, tw, pol);
        else gemv_tma_phase<Region::FfnDown, WK, ACT, NT>(a, s.plan[3], sm, rp, tw, pol);
        // The ring now holds this phase's tail; while the MMA warps finish it
        // and cross the phase barrier (and attention), HBM keeps streaming the
        // next phase's first chunks into L2, where its copies will find them.
        const int nl = reg == 3 ? l + 1 : l, nreg = reg == 3 ? 0 : reg + 1;
        if (nl < s.L)
          gemv_l2_prefetch_phase<WK>(s.layer[nl].tmap_w[nreg], s.layer[nl].tmap_s[nreg], s.plan[nreg],
                                     kStepL2Lookahead, s.qgroup[nreg]);
      }
    }
  } else if (warp == kEpiWarp) {
    // ---------------- epilogue warp: GEMV epilogues, then the phase arrival ----------------
    // (one epilogue warp here: the grid arrival is per CTA; warp kEpiWarp + 1 idles)
    int seg = 0;
    bool dead = false;
    unsigned p = 0;  // phase index
    for (int l = 0; l < s.L; ++l) {
      for (int r = 0; r < 5; ++r, ++p) {
        if (r == 1) continue;  // attention: the MMA warps arrive
        // Never run ahead of the grid: a phase where this CTA has no work
        // must not be arrived at before the previous phase completed.
        if (p > 0) step_wait_warp(s.grid_bar, p * G, s.status, dead);
        const int reg = r == 0 ? 0 : r - 1;
        const RegionArgs a = step_region_args(s, l, reg);
        if (reg == 0) gemv_epi_phase<Region::LnQkv, WK, ACT, NT>(a, s.plan[0], sm, seg);
        else if (reg == 1) gemv_epi_phase<Region::OprojRes, WK, ACT, NT>(a, s.plan[1], sm, seg);
        else if (reg == 2) gemv_epi_phase<Region::FfnUp, WK, ACT, NT>(a, s.plan[2], sm, seg);
        else gemv_epi_phase<Region::FfnDown, WK, ACT, NT>(a, s.plan[3], sm, seg);
        __threadfence();
        __syncwarp();
        if (lane == 0) step_arrive(s.grid_bar, total);
      }
    }
    // Every phase that reads seq[] has completed in every CTA once this CTA's
    // last phase began (the FFN-down phase follows the last attention barrier).
    if (blockIdx.x == 0)
      for (int b = lane; b < s.B; b += 32) s.seq[b] += 1;
  }
}

}  // namespace ds
