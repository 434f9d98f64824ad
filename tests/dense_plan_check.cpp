// CPU replay of the tile GEMMs' work plan (transformer_layer_gb300/csrc/dense_plan.h)
// over many shapes, checking the invariants the kernels rely on:
//  * token tiles of 16..256 rows (int8: 64), covering the M rows;
//  * 2..8 ring stages within the shared memory, and more than half an SM's
//    shared memory per CTA (no two tile CTAs share an SM, nor its 512 tensor-
//    memory columns);
//  * the tensor-memory columns of the accumulators (two per MMA issuer) and
//    int8 W tiles within 512, and an even ring depth when fp16 / bf16 run two
//    issuers (each owns the stages of one parity), which decode-size tiles
//    (up to 64 token rows) always do;
//  * a grid within the SMs; a cluster plan with one K slice per CTA, at most 8
//    CTAs per cluster, slices that cover the K chunks exactly once (each at
//    least one chunk), and -- for slices of unequal length, a size chosen by
//    the capacity query -- all its clusters on the GPU at once; uniform slices
//    otherwise.
// The GPU's cluster capacity comes from a model of 8 GPCs of 18-19 SMs.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "dense_plan.h"

using namespace ds;

namespace {

int g_fail = 0;
long g_uneven = 0, g_pow2 = 0, g_two_issuers = 0, g_int8 = 0;  // coverage of the sweep

#define CHECK(cond)                                                                                        \
  do {                                                                                                     \
    if (!(cond)) {                                                                                         \
      if (g_fail++ < 20)                                                                                   \
        std::printf("FAIL %s: N=%d K=%d M=%d ak=%d i8=%d sms=%d\n", #cond, N, K, M, (int)ak, (int)i8, sms); \
    }                                                                                                      \
  } while (0)

// Clusters of `size` CTAs (one per SM) that fit at once: a cluster lives in one GPC.
int capacity(int size, int sms) {
  std::vector<int> gpc(8, sms / 8);
  for (int i = 0; i < sms % 8; ++i) gpc[i] += 1;
  int n = 0;
  for (int g : gpc) n += g / size;
  return n;
}

void check_plan(ActKind ak, bool i8, int N, int K, int M, int sms, int max_smem) {
  DensePlan p;
  const bool ok = dense_make_plan_t(ak, N, K, M, sms, max_smem, &p, i8, [&](int s) { return capacity(s, sms); });
  if (!ok) return;  // (a shape without a plan is refused before any launch)
  const bool split = ak == ActKind::BF16;
  const GemvPlan& w = p.ws;
  // token tiles
  CHECK(p.ntok % 16 == 0 && p.ntok >= 16 && p.ntok <= (i8 ? 64 : 256));
  CHECK(p.ntok * p.tok_tiles >= M && p.ntok * (p.tok_tiles - 1) < M);
  CHECK(p.kc == 64 || p.kc == 128);
  CHECK(!i8 || p.kc == 128);
  CHECK(p.kchunks * p.kc == K);
  CHECK(w.tiles == p.row_tiles * p.tok_tiles && p.row_tiles * 128 == N);
  // ring and shared memory
  const size_t SB = (dense_stage_bytes(p.ntok, p.kc, split, i8) + 1023) & ~(size_t)1023;
  CHECK(p.stages >= 2 && p.stages <= kDenseMaxStages);
  CHECK(p.smem <= (size_t)max_smem && (size_t)p.stages * SB < p.smem);
  CHECK(2 * p.smem > (size_t)max_smem + 1024);  // one tile CTA per SM
  // tensor memory and MMA issuers
  const int nis = dense_issuers(p.ntok, p.stages, i8);
  CHECK(nis == 1 || nis == kDenseMaxIssuers);
  CHECK(dense_tmem_cols(p.ntok, nis, i8) <= 512);
  CHECK(i8 || nis == 1 || p.stages % 2 == 0);
  CHECK(i8 || p.ntok > 64 || nis == kDenseMaxIssuers);  // decode-size tiles get their second issuer
  CHECK(!i8 || nis == kDenseMaxIssuers);
  if (nis > 1 && !i8) ++g_two_issuers;
  if (i8) ++g_int8;
  // work split
  CHECK(w.grid >= 1 && w.grid <= sms);
  CHECK(w.units == w.tiles * w.KS);
  if (p.cluster > 1) {
    CHECK(p.cluster == w.KS && p.cluster <= 8);
    CHECK(w.grid == w.units && w.q == 1 && w.R == 0 && w.grid % p.cluster == 0);
    CHECK(capacity(p.cluster, sms) >= w.tiles || (p.kchunks % p.cluster == 0 && (p.cluster & (p.cluster - 1)) == 0));
    CHECK((size_t)p.stages * SB >= (size_t)p.ntok * 128 * 4);  // a partial tile fits the idle ring
    int covered = 0, longest = 0;
    for (int s = 0; s < p.cluster; ++s) {
      const int c0 = s * p.kchunks / p.cluster, c1 = (s + 1) * p.kchunks / p.cluster;
      CHECK(c0 == covered && c1 - c0 >= 1);
      covered = c1;
      if (c1 - c0 > longest) longest = c1 - c0;
    }
    CHECK(covered == p.kchunks && longest == w.C);
    if (p.kchunks % p.cluster != 0) ++g_uneven;
    else ++g_pow2;
  } else {
    CHECK(p.kchunks % w.KS == 0 && w.C * w.KS == p.kchunks);
  }
}

}  // namespace

int main() {
  const int Ns[] = {128, 256, 512, 1024, 2048, 2560, 3072, 4096, 5120, 7680, 10240, 12288, 15360, 16384, 20480};
  const int Ks[] = {256, 512, 1024, 2560, 4096, 5120, 10240, 16384, 20480};
  const int Ms[] = {8, 9, 16, 17, 31, 32, 48, 63, 64, 65, 100, 128, 129, 150, 192, 255, 256, 300, 512, 1000, 2048, 4096};
  const int smss[] = {148, 152, 132};
  const int max_smem = 232448;
  long checked = 0;
  for (int sms : smss)
    for (int N : Ns)
      for (int K : Ks)
        for (int M : Ms)
          for (int v = 0; v < 3; ++v) {
            const ActKind ak = v == 1 ? ActKind::BF16 : ActKind::F16;
            const bool i8 = v == 2;
            if (i8 && (K % 1024 != 0 || M > 4096)) continue;  // int8 layers: K a multiple of 8 groups of 128
            check_plan(ak, i8, N, K, M, sms, max_smem);
            ++checked;
          }
  if (g_uneven == 0 || g_pow2 == 0 || g_two_issuers == 0 || g_int8 == 0) {
    std::printf("coverage: uneven clusters %ld, even clusters %ld, two-issuer plans %ld, int8 plans %ld\n", g_uneven,
                g_pow2, g_two_issuers, g_int8);
    return 1;
  }
  if (g_fail) {
    std::printf("%d failures in %ld plans\n", g_fail, checked);
    return 1;
  }
  std::printf("ok\n");
  return 0;
}
