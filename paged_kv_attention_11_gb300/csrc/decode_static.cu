// paged_attn_decode_static: the decode entry point for callers that cannot
// allocate device memory.
//
// Some callers of this library may not allocate on the path that runs the
// attention step: an engine that has carved all free HBM into its KV page
// pool ahead of time, a plugin host that hands a kernel only its input and
// output buffers, or code running where a cudaMalloc would stall or be
// refused.  For them this entry point runs the same split-KV decode as
// paged_attn_decode, but its scratch (per-segment arrival counters and the
// partial outputs of split sequences) lives in one fixed array of device
// memory that belongs to the library itself.
//
// That array is a file-scope __device__ object of kDecodeStaticScratchBytes
// bytes: every GPU that loads the library holds it until the process exits.
// Host code only ever sees a host-side stand-in for its name, so the device
// address is looked up with cudaGetSymbolAddress once per device (with that
// device current) the first time the entry point runs there; make that first
// call before any stream capture.  All calls share the array: the arrival
// counters are cleared on the call's stream before every launch, and calls
// whose work overlaps on the GPU (other streams, other threads) race on it.
#include <mutex>
#include <string>

#include "../../include/pkv.h"
#include "kernels.h"

namespace {

constexpr size_t kDecodeStaticScratchBytes = size_t(8) << 20;  // 8 MiB

__device__ __align__(256) unsigned char g_decode_scratch[kDecodeStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up once).
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

pkv_status paged_attn_decode_static(void* out, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_table,
                                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                    int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t page_size, int64_t num_pages,
                                    int32_t max_seq_len, float scale, int32_t window,
                                    int32_t* err_flag, void* stream) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      num_pages <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
      num_q_heads % num_kv_heads != 0 || !(scale == scale))
    return PKV_ERR_INVALID;
  if (batch == 0) return PKV_OK;
  const size_t need =
      paged_attn_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim);
  if (need == 0) return PKV_ERR_UNSUPPORTED;  // shape outside the supported set
  if (need > kDecodeStaticScratchBytes) {
    pkv::set_last_error("paged_attn_decode_static: this batch needs " + std::to_string(need) +
                        " bytes of scratch, more than the library's fixed " +
                        std::to_string(kDecodeStaticScratchBytes) +
                        "-byte buffer; use paged_attn_decode with a caller workspace");
    return PKV_ERR_UNSUPPORTED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
  void* scratch = nullptr;
  if (e == cudaSuccess) e = scratch_address(dev, &scratch);
  if (e == cudaSuccess) {
    // the arrival and queue counters (the first batch*num_kv_heads + 2
    // int32) must start at zero
    e = cudaMemsetAsync(scratch, 0, ((size_t)batch * num_kv_heads + 2) * sizeof(int32_t),
                        static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) {
    pkv::set_last_error(cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  return paged_attn_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                           batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                           max_seq_len, scale, window, scratch, kDecodeStaticScratchBytes,
                           err_flag, stream);
}

}  // extern "C"
