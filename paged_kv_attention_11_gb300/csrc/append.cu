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
// One warp per token: lane l moves vectors l, l+32, ... of the token's K
// and V rows (H_kv*head_dim*2 contiguous bytes on the source side, one
// head_dim*2-byte run per kv head on the pool side), so a warp's accesses
// are coalesced on both sides.  All of a lane's loads (and the token's slot)
// are issued before its first store; the grid holds every token of a
// prefill-sized step at once (5645 tokens = 5645 warps), so the whole
// batch of reads is in flight together.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr int kAppendThreads = 256;   // 8 tokens per block
constexpr int kAppendBlocksPerSM = 5;  // 40 warps (tokens) per SM: 6080 in one wave

// J: vectors of K (and of V) per lane per pass
template <int J>
__global__ void __launch_bounds__(kAppendThreads, 5) kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, const int64_t* __restrict__ slot_mapping, int32_t num_tokens,
    int32_t vecs_per_tok, int32_t vecs_per_row, int32_t H_kv, int32_t P, int64_t num_slots,
    int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int wpb = kAppendThreads / 32;
  const int nw = gridDim.x * wpb;
  for (int tok = blockIdx.x * wpb + (threadIdx.x >> 5); tok < num_tokens; tok += nw) {
    const int64_t slot = __ldg(slot_mapping + tok);
    const int64_t src0 = (int64_t)tok * vecs_per_tok;
    for (int v0 = 0; v0 < vecs_per_tok; v0 += 32 * J) {
      uint4 kv[J], vv[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int v = v0 + lane + 32 * j;
        if (v < vecs_per_tok) {
          kv[j] = __ldg(k_new + src0 + v);
          vv[j] = __ldg(v_new + src0 + v);
        }
      }
      if (slot < 0) continue;  // padding row: skip
      if (slot >= num_slots) {
        if (lane == 0 && v0 == 0) raise_err(err, PKV_DEVERR_SLOT);
        continue;
      }
      const int64_t page = slot / P;
      const int row = (int)(slot - page * P);
      // head 0 of the row; a head's row sits P * vecs_per_row vectors further
      uint4* kd = k_cache + (page * H_kv * P + row) * vecs_per_row;
      uint4* vd = v_cache + (kd - k_cache);
      const int hstride = P * vecs_per_row;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int v = v0 + lane + 32 * j;
        if (v < vecs_per_tok) {
          const int h = v / vecs_per_row;
          const int off = h * hstride + (v - h * vecs_per_row);
          kd[off] = kv[j];
          vd[off] = vv[j];
        }
      }
    }
  }
}

template <int J>
static cudaError_t launch_append_t(const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, const int64_t* slot_mapping, int32_t num_tokens,
                                   int32_t vpt, int32_t vpr, int32_t H_kv, int32_t P,
                                   int64_t num_slots, int32_t* err, cudaStream_t stream,
                                   int num_sms) {
  int64_t blocks = ((int64_t)num_tokens + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
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
  return cudaLaunchKernelEx(&cfg, kv_append_kernel<J>, static_cast<const uint4*>(k_new),
                            static_cast<const uint4*>(v_new), static_cast<uint4*>(k_cache),
                            static_cast<uint4*>(v_cache), slot_mapping, num_tokens, vpt, vpr,
                            H_kv, P, num_slots, err);
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t H_kv,
                             int32_t D, int32_t P, int64_t num_pages, int32_t* err,
                             cudaStream_t stream, int num_sms) {
  const int32_t vecs_per_row = D / 8;
  const int64_t vecs_per_tok = (int64_t)H_kv * vecs_per_row;
  const int64_t total = (int64_t)num_tokens * vecs_per_tok;
  if (total == 0) return cudaSuccess;
  if (total >= (int64_t(1) << 31) || vecs_per_tok >= (int64_t(1) << 24))
    return cudaErrorNotSupported;
  const int32_t vpt = (int32_t)vecs_per_tok;
  const int64_t num_slots = num_pages * P;
  if (vpt <= 32)
    return launch_append_t<1>(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens, vpt,
                              vecs_per_row, H_kv, P, num_slots, err, stream, num_sms);
  // 2 vectors of K and of V per lane per pass: 46 registers, 5 blocks per SM
  // (4 would spill at that occupancy); a 2 KB token row takes two passes
  return launch_append_t<2>(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens, vpt,
                            vecs_per_row, H_kv, P, num_slots, err, stream, num_sms);
}

}  // namespace pkv
