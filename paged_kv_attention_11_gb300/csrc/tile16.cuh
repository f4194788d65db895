// 16-key K/V tiles staged by TMA for the mma.sync decode kernels (the
// split-KV decode and the shared-prefix pass): layout in shared memory and
// the fragment address of a key row.
#pragma once

#include <stdint.h>

namespace pkv {

constexpr int kTile = 16;  // keys per pipeline stage
constexpr int kGP = 8;     // query rows per mma N tile (the GQA group, padded)

// Shared-memory address of 16-byte chunk c (0..D/8-1) of key row `key` in a
// staged K or V tile.  A tile is one TMA box of the pool's 5-D view
// {64 columns, 8 rows, D/64 column chunks, P/8 row groups, pages*H_kv}: it
// lands as [row group (2)][column chunk (D/64)][8 rows][128 bytes], every
// [8 rows][128 bytes] block one 1024-byte swizzle atom (16-byte unit u of
// row r at unit u ^ r).  The 8 rows an ldmatrix reads (8 consecutive keys,
// one column chunk) sit in 8 distinct bank groups.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int key, int c) {
  return base + (key >> 3) * (D / 64) * 1024 + (c >> 3) * 1024 + (key & 7) * 128 +
         (((c & 7) ^ (key & 7)) << 4);
}

}  // namespace pkv

namespace pkv {

// Shared-prefix (cascade) decode: the number of leading keys that group j's
// sequences share, as the prefix pass and the decode kernel both read it.
// A length that is negative, not a whole number of pages, or longer than a
// block-table row gives 0 (no sharing; the prefix pass flags it).
__device__ __forceinline__ int shared_prefix_len(const int32_t* prefix_lens, int j, int P,
                                                 int cap) {
  const int pl = __ldg(prefix_lens + j);
  return (pl > 0 && pl % P == 0 && pl <= cap) ? pl : 0;
}

}  // namespace pkv
