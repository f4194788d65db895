// 16-key K/V tiles staged by TMA for the mma.sync decode kernels (the
// split-KV decode and the shared-prefix pass): layout in shared memory and
// the fragment address of a key row.
#pragma once

#include <stdint.h>

namespace pkv {

constexpr int kTile = 16;  // keys per pipeline stage
constexpr int kGP = 8;     // query rows per mma N tile (the GQA group, padded)

// Shared-memory address of 16-byte chunk c (0..D/8-1) of key row `key` in a
// staged tile.  Default staging: D/64 boxes of [16 rows x 128 B] (one box
// per 64-column slice).  ONEBOX (head_dim 128): one box of 32 rows x 128 B,
// row = 2*key + c/8.  Both are 128-byte swizzled: 16-byte unit u of a row r
// sits at unit u ^ (r % 8).
template <int D, bool ONEBOX>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int key, int c) {
  if (ONEBOX) {
    const int rp = 2 * key + (c >> 3);
    return base + rp * 128 + (((c & 7) ^ (rp & 7)) << 4);
  } else {
    return base + (c >> 3) * (kTile * 128) + key * 128 + (((c & 7) ^ (key & 7)) << 4);
  }
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
