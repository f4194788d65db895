// pkv_copy: a byte copy done by the SMs instead of a copy engine, for the
// small per-step transfers between pinned host memory and the GPU (a decode
// step's queries, new K/V rows and tables in; its output rows out).
//
// On a GB300 the copy engines take 11-14 us for a transfer of 0.5-0.8 MB
// (their fixed cost dominates at that size), while the SMs reach pinned
// host memory directly over the chip-to-chip link (unified addressing maps
// pinned memory at the same address on the device).  Each thread moves
// 16-byte words; a grid of up to 8 blocks per SM puts a whole
// step-sized transfer in flight at once, and larger copies loop with four
// words per thread in flight.
//
// Launched with programmatic dependent launch like the attention kernels:
// griddepcontrol.wait precedes the first load, so the copy may directly
// follow the kernel whose output it reads, and the kernel that follows the
// copy may run its prologue while the copy drains.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kCopyBlocksPerSM = 8;

__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(uint4* __restrict__ dst,
                                                               const uint4* __restrict__ src,
                                                               int64_t n) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
  for (int64_t base = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; base < n;
       base += stride * kCopyUnroll) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j) {
      const int64_t i = base + j * stride;
      if (i < n) v[j] = src[i];
    }
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j) {
      const int64_t i = base + j * stride;
      if (i < n) dst[i] = v[j];
    }
  }
}

cudaError_t launch_copy16(void* dst, const void* src, int64_t n16, cudaStream_t stream,
                          int num_sms) {
  if (n16 <= 0) return cudaSuccess;
  int64_t blocks = (n16 + kCopyThreads - 1) / kCopyThreads;
  const int64_t cap = (int64_t)num_sms * kCopyBlocksPerSM;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy16_kernel, static_cast<uint4*>(dst),
                            static_cast<const uint4*>(src), n16);
}

}  // namespace pkv
