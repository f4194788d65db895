// paged_kv_append: scatter new K/V rows into the page pools through a slot
// mapping (scripts/benchmarks commit log, flex paged-KV engine "Files"
// paragraph: the in-kernel k_cache[addr] = k_val write of each new row).
//
// Pure data movement, HBM-bound.  The new rows are a flat array of 16-byte
// vectors (token, kv head, 8 dims); vector i of the K rows goes to the same
// place in the K pool as vector i of the V rows in the V pool.  A token row
// of one kv head is head_dim*2 contiguous bytes on both sides, so
// consecutive threads read and write consecutive 16-byte words.
//
// Each thread moves kVecs vectors of K and of V per pass, strided by the
// grid so that a warp's accesses stay coalesced, and issues all of their
// loads (and the slot loads) before its first store: 2*kVecs 16-byte loads
// in flight per thread instead of one round trip per vector.  Index math is
// 32-bit (the host caps the vector count below 2^31).
#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr int kAppendThreads = 256;
constexpr int kAppendVecs = 4;          // vectors of K (and of V) per thread per pass
constexpr int kAppendBlocksPerSM = 4;   // 1024 threads x 64 registers per SM

__global__ void __launch_bounds__(kAppendThreads, kAppendBlocksPerSM) kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, uint32_t total_vecs,
    uint32_t vecs_per_tok, uint32_t vecs_per_row, int32_t H_kv, int32_t P, int64_t num_slots,
    int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < total_vecs;
       base += kAppendVecs * stride) {
    uint4 kv[kAppendVecs], vv[kAppendVecs];
    int64_t slot[kAppendVecs];
    uint32_t r[kAppendVecs];
#pragma unroll
    for (int j = 0; j < kAppendVecs; ++j) {
      const uint32_t i = base + j * stride;
      slot[j] = -1;
      if (i < total_vecs) {
        const uint32_t t = i / vecs_per_tok;
        r[j] = i - t * vecs_per_tok;
        slot[j] = __ldg(slot_mapping + t);
        kv[j] = __ldg(k_new + i);
        vv[j] = __ldg(v_new + i);
      }
    }
#pragma unroll
    for (int j = 0; j < kAppendVecs; ++j) {
      const int64_t s = slot[j];
      if (s < 0) continue;  // padding row (or past the end): skip
      if (s >= num_slots) {
        if (r[j] == 0) raise_err(err, PKV_DEVERR_SLOT);
        continue;
      }
      const uint32_t h = r[j] / vecs_per_row;
      const uint32_t v = r[j] - h * vecs_per_row;
      const int64_t page = s / P;
      const int64_t row = s - page * P;
      const int64_t dst = ((page * H_kv + h) * P + row) * vecs_per_row + v;
      k_cache[dst] = kv[j];
      v_cache[dst] = vv[j];
    }
  }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t H_kv,
                             int32_t D, int32_t P, int64_t num_pages, int32_t* err,
                             cudaStream_t stream, int num_sms) {
  const int32_t vecs_per_row = D / 8;
  const int64_t vecs_per_tok = (int64_t)H_kv * vecs_per_row;
  const int64_t total = (int64_t)num_tokens * vecs_per_tok;
  if (total == 0) return cudaSuccess;
  if (total >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  const int64_t per_block = (int64_t)kAppendThreads * kAppendVecs;
  int64_t blocks = (total + per_block - 1) / per_block;
  const int64_t cap = (int64_t)num_sms * kAppendBlocksPerSM;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kAppendThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<const uint4*>(k_new),
                            static_cast<const uint4*>(v_new), static_cast<uint4*>(k_cache),
                            static_cast<uint4*>(v_cache), slot_mapping, (uint32_t)total,
                            (uint32_t)vecs_per_tok, (uint32_t)vecs_per_row, H_kv, P,
                            num_pages * P, err);
}

}  // namespace pkv
