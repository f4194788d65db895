// paged_attn_varlen: tcgen05 prefill kernel (in progress).
#include "common.cuh"
#include "kernels.h"

namespace pkv {

cudaError_t launch_varlen(void*, const VarlenMaps&, const int32_t*, const int32_t*,
                          const int32_t*, int32_t, int32_t, int32_t, int32_t, int32_t, int32_t,
                          int32_t, int32_t, int64_t, float, int32_t, int32_t, int32_t*,
                          cudaStream_t, int) {
  return cudaErrorNotSupported;
}

}  // namespace pkv
