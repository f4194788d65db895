// paged_kv_append: scatter new K/V rows into the page pools through a slot
// mapping (scripts/benchmarks commit log, flex paged-KV engine "Files"
// paragraph: the in-kernel k_cache[addr] = k_val write of each new row).
//
// Pure data movement, HBM-bound: every thread moves one 16-byte vector of K
// and the matching vector of V.  A token row of one kv head is head_dim*2
// contiguous bytes on both sides, so consecutive threads read and write
// consecutive 16-byte words (coalesced 512-byte warp transactions).
#include "common.cuh"
#include "kernels.h"

namespace pkv {

__global__ void __launch_bounds__(256) kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int64_t total_vecs,
    int32_t vecs_per_tok, int32_t vecs_per_row, int32_t H_kv, int32_t P, int64_t num_slots,
    int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_vecs; i += stride) {
    const int64_t t = i / vecs_per_tok;
    const int32_t r = (int32_t)(i - t * vecs_per_tok);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding row: skip
    if (slot >= num_slots) {
      if (r == 0) raise_err(err, PKV_DEVERR_SLOT);
      continue;
    }
    const int32_t h = r / vecs_per_row;
    const int32_t v = r - h * vecs_per_row;
    const int64_t page = slot / P;
    const int64_t row = slot - page * P;
    const int64_t dst = ((page * H_kv + h) * P + row) * vecs_per_row + v;
    const uint4 kv = __ldg(k_new + i);
    const uint4 vv = __ldg(v_new + i);
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t H_kv,
                             int32_t D, int32_t P, int64_t num_pages, int32_t* err,
                             cudaStream_t stream, int num_sms) {
  const int32_t vecs_per_row = D / 8;
  const int32_t vecs_per_tok = H_kv * vecs_per_row;
  const int64_t total = (int64_t)num_tokens * vecs_per_tok;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<const uint4*>(k_new),
                            static_cast<const uint4*>(v_new), static_cast<uint4*>(k_cache),
                            static_cast<uint4*>(v_cache), slot_mapping, total, vecs_per_tok,
                            vecs_per_row, H_kv, P, num_pages * P, err);
}

}  // namespace pkv
