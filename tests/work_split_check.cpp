// CPU replay of the skinny-GEMM work split (the same functions the kernels
// call, from transformer_layer_gb300/csrc/work_split.h).  For each plan it
// walks every CTA's chunk sequence as the streaming warps do and its segment
// list as the epilogue warp does, and checks that:
//   - every (slice, tile, chunk) is processed exactly once;
//   - both sides see the same segments, each inside one unit;
//   - a segment is finished directly only if it covers a whole unit alone;
//   - the partial contributions of each row tile equal its arrival target,
//     with distinct slots below maxc.
// Prints "ok" and exits 0, or prints the first violation and exits 1.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <tuple>
#include <vector>

#include "work_split.h"

using namespace ds;

static int fail(const char* what, int N, int K, int M, int G, int a, int b) {
  std::printf("FAIL %s N=%d K=%d M=%d G=%d (%d, %d)\n", what, N, K, M, G, a, b);
  return 1;
}

static int verify(const GemvPlan& P, int N, int K, int M) {
  const int G = P.grid, C = P.C, tiles = P.tiles;
  if (!P.whole && P.R > 0 && P.R < G) return fail("fewer leftover chunks than CTAs", N, K, M, G, (int)P.R, G);
  std::map<std::tuple<int, int, int>, int> cover;
  std::map<int, std::vector<std::pair<int, int>>> parts;  // tile -> (slice, slot)
  for (int cta = 0; cta < G; ++cta) {
    long long ra, rb;
    ws_left_range(P, cta, G, &ra, &rb);
    const int dp_b = ws_dp_first(P, cta);
    const int nch = (int)(rb - ra) + P.q * C;
    // streaming warps
    Cursor q;
    ws_cursor_init(q, P, ra, rb, dp_b);
    std::vector<std::vector<std::tuple<int, int, int>>> segs(1);
    for (int j = 0; j < nch; ++j) {
      if (q.s < 0 || q.s >= P.KS || q.t < 0 || q.t >= tiles || q.kc < 0 || q.kc >= C)
        return fail("cursor out of range", N, K, M, G, cta, j);
      cover[std::make_tuple(q.s, q.t, q.kc)] += 1;
      segs.back().push_back(std::make_tuple(q.s, q.t, q.kc));
      if (ws_segment_ends(q, P, j, nch)) segs.emplace_back();
      ws_cursor_next(q, P, dp_b);
    }
    segs.pop_back();
    // epilogue warp
    std::vector<std::pair<int, int>> esegs;
    for (long long i = ra; i < rb;) {
      int u, js;
      long long end;
      ws_leftover_segment(P, i, rb, cta, G, &u, &end, &js);
      esegs.push_back(std::make_pair(u, js));
      if (end <= i) return fail("leftover segment does not advance", N, K, M, G, cta, (int)i);
      i = end;
    }
    for (int i = 0; i < P.q; ++i) esegs.push_back(std::make_pair(ws_dp_unit(P, cta, i), 0));
    if (esegs.size() != segs.size())
      return fail("segment count differs", N, K, M, G, (int)esegs.size(), (int)segs.size());
    for (size_t i = 0; i < segs.size(); ++i) {
      const int u = esegs[i].first, js = esegs[i].second, s = u / tiles, t = u % tiles;
      for (auto& ch : segs[i])
        if (std::get<0>(ch) != s || std::get<1>(ch) != t) return fail("segment crosses units", N, K, M, G, cta, u);
      if (js < 0 || js >= P.maxc) return fail("slot out of range", N, K, M, G, cta, js);
      const bool direct = (P.KS == 1 && ws_unit_contrib(u, P, G) == 1);
      if (direct && (int)segs[i].size() != C) return fail("direct segment not whole", N, K, M, G, cta, u);
      if (!direct) parts[t].push_back(std::make_pair(s, js));
    }
  }
  for (int s = 0; s < P.KS; ++s)
    for (int t = 0; t < tiles; ++t)
      for (int kc = 0; kc < C; ++kc)
        if (cover[std::make_tuple(s, t, kc)] != 1) return fail("chunk not covered once", N, K, M, G, t, kc);
  for (auto& kv : parts) {
    const int t = kv.first;
    if ((int)kv.second.size() != ws_tile_target(t, P, G))
      return fail("contributions differ from target", N, K, M, G, t, (int)kv.second.size());
    std::set<std::pair<int, int>> uniq(kv.second.begin(), kv.second.end());
    if (uniq.size() != kv.second.size()) return fail("duplicate partial slot", N, K, M, G, t, 0);
    for (auto& sj : kv.second) {
      const int n = ws_unit_contrib(sj.first * tiles + t, P, G);
      if (sj.second >= n) return fail("slot beyond contributors", N, K, M, G, t, sj.second);
    }
  }
  return 0;
}

static int check(int N, int K, int M, int G0, bool i8, bool split) {
  const int blk_k = i8 ? 64 : 32, pad = i8 ? 8 : 32;
  auto xs = [&](int K_S) { return (size_t)(split ? 2 : 1) * M * (K_S + pad) * 2; };
  GemvPlan P;
  if (!ws_make_plan(N, K, M, G0, blk_k, 8, 80 * 1024, xs, &P)) return 0;  // shape not supported
  return verify(P, N, K, M);
}

// The tensor-core tile path: units are output tiles (128 weight rows x one
// token tile), one K slice, chunks of 128 along K.
static int check_tiles(int tiles, int K, int G0) {
  GemvPlan P;
  P.tiles = tiles;
  P.KS = 1;
  P.K_S = K;
  P.chunk_k = 128;
  P.C = K / 128;
  P.units = tiles;
  ws_distribute(P, G0);
  return verify(P, 128 * tiles, K, 0);
}

// The tile path's plan with one whole unit per CTA: each tile cut into KS
// slices along K when there are few tiles.
static int check_tiles_sliced(int tiles, int K, int G0) {
  GemvPlan P;
  P.tiles = tiles;
  P.chunk_k = 128;
  int KS = 1;
  if (tiles * 5 < G0 * 3)
    while (KS < 8 && tiles * KS * 2 <= G0 && (K / 128) % (KS * 2) == 0) KS *= 2;
  P.KS = KS;
  P.K_S = K / KS;
  P.C = P.K_S / 128;
  P.units = tiles * KS;
  // as the tile planner with several token tiles: more tiles than CTAs ->
  // whole tiles, round-robin (the planner splits leftovers with one token tile)
  const bool many = tiles > G0 && (tiles % 3) != 0;
  ws_distribute(P, G0, true, many);
  P.interleave = many ? 1 : 0;
  if (P.units <= G0 && (P.grid != P.units || P.q != 1 || P.R != 0))
    return fail("one unit per CTA not kept", 128 * tiles, K, 0, P.grid, P.units, P.q);
  if (many && P.R > 0 && !P.whole) return fail("leftover tiles split", 128 * tiles, K, 0, P.grid, P.units, P.q);
  return verify(P, 128 * tiles, K, 0);
}

int main() {
  int bad = 0;
  // Shapes of the shipped workloads (QKV, O-proj, FFN-up, FFN-down), batch rows 1..64.
  const int HF[][2] = {{256, 1024}, {512, 2048}, {2560, 10240}, {4096, 16384}, {5120, 20480}};
  const int Ms[] = {1, 2, 3, 4, 8, 16, 24, 32, 40, 64};
  for (auto& hf : HF)
    for (int M : Ms)
      for (int i8 = 0; i8 < 2; ++i8)
        for (int split = 0; split < 2; ++split)
          for (int G : {152, 304}) {
            const int H = hf[0], F = hf[1];
            bad |= check(3 * H, H, M, G, i8, split);
            bad |= check(H, H, M, G, i8, split);
            bad |= check(F, H, M, G, i8, split);
            bad |= check(H, F, M, G, i8, split);
          }
  // Pseudo-random shapes and grid sizes.
  unsigned x = 12345u;
  auto rnd = [&](int n) { x = x * 1103515245u + 12345u; return (int)((x >> 8) % (unsigned)n); };
  for (int it = 0; it < 3000 && !bad; ++it) {
    const bool i8 = rnd(2);
    const int K = (i8 ? 512 : 256) * (1 + rnd(40));
    const int N = 16 * (1 + rnd(600));
    const int M = 1 + rnd(64);
    const int G = 1 + rnd(400);
    bad |= check(N, K, M, G, i8, rnd(2));
    if (it % 4 == 0) bad |= check_tiles(1 + rnd(400), 256 * (1 + rnd(40)), G);
  }
  for (auto& hf : HF)
    for (int tt = 1; tt <= 8; tt *= 2) {      // token tiles of a long prompt
      const int H = hf[0], F = hf[1];
      bad |= check_tiles(tt * 3 * H / 128, H, 152);
      bad |= check_tiles(tt * H / 128, H, 152);
      bad |= check_tiles(tt * F / 128, H, 152);
      bad |= check_tiles(tt * H / 128, F, 152);
      bad |= check_tiles_sliced(tt * 3 * H / 128, H, 152);
      bad |= check_tiles_sliced(tt * H / 128, H, 152);
      bad |= check_tiles_sliced(tt * F / 128, H, 152);
      bad |= check_tiles_sliced(tt * H / 128, F, 152);
    }
  for (int it = 0; it < 400 && !bad; ++it)
    bad |= check_tiles_sliced(1 + rnd(300), 256 * (1 + rnd(64)), 1 + rnd(300));
  if (!bad) std::printf("ok\n");
  return bad;
}
