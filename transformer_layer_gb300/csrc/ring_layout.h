// Shared-memory layout of one weight chunk of the GEMV ring, as the TMA
// tensor copy writes it, and the addressing the MMA warps read it with.
// Shared by the kernels and the CPU replay test (tests/ring_layout_check.cpp).
//
// A chunk is 16 weight rows x CB bytes (CB = chunk_k x weight bytes, a
// multiple of 128).  One 3-D TMA copy with the 128-byte swizzle writes it as
// [segment s = byte / 128][row r][128 bytes]; the swizzle stores 16-byte unit
// j of (s, r) at unit j ^ (r % 8) of its 128 bytes (the stage starts on a
// 1024-byte boundary, so the XOR term is exactly r % 8).
//
// Fragment row g (0..7) of the 16x16 A operand of mma.m16n8k16 reads weight
// rows rl_row(g) and rl_row(g) + 8, with rl_row = 0, 4, 1, 5, 2, 6, 3, 7: the
// two rows a quarter-warp reads then have XOR terms that differ by 4, i.e.
// they sit in opposite 64-byte halves of the 128-byte bank window, and every
// 128-bit fragment load is free of bank conflicts.  The epilogue undoes the
// permutation when it stores the partial tiles.
#pragma once

#if defined(__CUDACC__)
#define DS_RL __host__ __device__ __forceinline__
#else
#define DS_RL inline
#endif

namespace ds {

constexpr int kSwizzleBytes = 128;  // TMA swizzle span = bytes of a chunk row per segment

// Weight row (within the 16-row tile) that fragment row g (0..7) reads.
DS_RL int rl_row(int g) { return (g >> 1) | ((g & 1) << 2); }

// Byte offset within a chunk of byte o (a multiple of 16) of weight row r.
DS_RL unsigned rl_offset(int r, int o) {
  return (unsigned)(((o >> 7) * 16 + r) * 128 + ((((o >> 4) & 7) ^ (r & 7)) << 4));
}

}  // namespace ds
