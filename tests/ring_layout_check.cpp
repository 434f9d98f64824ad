// CPU replay of the GEMV weight-ring layout (transformer_layer_gb300/csrc/
// ring_layout.h).  For each chunk width it places every byte where a 3-D TMA
// tensor copy with the 128-byte swizzle puts it (16-byte unit index XOR the
// 1024-byte-window row bits of the shared-memory address), then replays the
// fragment loads of all 8 MMA warps and checks that:
//   - each lane reads exactly the (row, byte) its MMA fragment needs;
//   - the fragment rows of a tile cover rows 0..15 once;
//   - every 128-bit load is free of shared-memory bank conflicts (the 8
//     lanes of each quarter-warp hit 8 distinct 16-byte bank groups).
// Prints "ok" and exits 0, or prints the first violation and exits 1.
#include <cstdio>
#include <set>
#include <vector>

#include "ring_layout.h"

using namespace ds;

static int fail(const char* what, int cb, int a, int b) {
  std::printf("FAIL %s chunk_row_bytes=%d (%d, %d)\n", what, cb, a, b);
  return 1;
}

static int check(int cb /* chunk row bytes */, int nblk) {
  const int chunk = 16 * cb;
  // Where the swizzled tensor copy stores (row r, byte o): logical offset in
  // the [s][r][128] box, then bits 4..6 ^= bits 7..9.
  std::vector<int> owner(chunk, -1);
  for (int r = 0; r < 16; ++r)
    for (int o = 0; o < cb; o += 16) {
      const int logical = ((o / 128) * 16 + r) * 128 + (o % 128);
      const int phys = logical ^ (((logical >> 7) & 7) << 4);
      if (phys < 0 || phys + 16 > chunk) return fail("copy out of chunk", cb, r, o);
      for (int k = 0; k < 16; ++k) {
        if (owner[phys + k] != -1) return fail("copy overlap", cb, r, o);
        owner[phys + k] = r * 65536 + o + k;
      }
    }
  std::set<int> rows;
  for (int g = 0; g < 8; ++g) {
    rows.insert(rl_row(g));
    rows.insert(rl_row(g) + 8);
  }
  if ((int)rows.size() != 16 || *rows.begin() != 0 || *rows.rbegin() != 15) return fail("row cover", cb, 0, 0);
  // A warp step is nblk blocks of 64 bytes per row; 8 warps cover the chunk row.
  const int step = nblk * 64;
  if (8 * step != cb) return fail("step width", cb, step, 0);
  for (int w = 0; w < 8; ++w)
    for (int b = 0; b < nblk; ++b)
      for (int half = 0; half < 2; ++half) {
        int addr[32];
        for (int lane = 0; lane < 32; ++lane) {
          const int g = lane >> 2, c = lane & 3;
          const int r = rl_row(g) + 8 * half;
          const int o = w * step + b * 64 + 16 * c;
          const int a = (int)rl_offset(r, o);
          if (a < 0 || a + 16 > chunk || (a & 15)) return fail("load out of chunk", cb, w, lane);
          for (int k = 0; k < 16; ++k)
            if (owner[a + k] != r * 65536 + o + k) return fail("wrong bytes", cb, w * 100 + b, lane);
          addr[lane] = a;
        }
        for (int q = 0; q < 4; ++q) {
          std::set<int> groups;
          for (int l = 8 * q; l < 8 * q + 8; ++l) groups.insert((addr[l] / 16) % 8);
          if (groups.size() != 8) return fail("bank conflict", cb, w * 100 + b, q);
        }
      }
  return 0;
}

int main() {
  int bad = 0;
  // chunk rows of 8 warps x nblk blocks of 64 bytes (fp16: 32 elements, int8: 64 codes)
  for (int nblk : {1, 2, 4}) bad |= check(8 * nblk * 64, nblk);
  if (!bad) std::printf("ok\n");
  return bad;
}
