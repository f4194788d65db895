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
// bytes.  CUDA places it on a device when this file's module is loaded
// there, which under the default lazy module loading is the first call of
// this entry point on that device (the address lookup below); from then on
// the device holds it until the process exits.  So the first call on each
// device must come before the caller hands the remaining free HBM to its
// page pool, and before any stream capture.  Host code only ever sees a
// host-side stand-in for the array's name, so the device address is looked
// up with cudaGetSymbolAddress with the device current, once per device and
// CUDA context (a new primary context after cudaDeviceReset, or another
// context on the same device, gets its own lookup).  All calls share the
// array: the arrival counters are cleared on the call's stream before every
// launch, and calls whose work overlaps on the GPU (other streams, other
// threads) race on it.
#include <cuda.h>

#include <mutex>
#include <string>

#include "../../include/pkv.h"
#include "kernels.h"

namespace {

constexpr size_t kDecodeStaticScratchBytes = size_t(8) << 20;  // 8 MiB

__device__ __align__(256) unsigned char g_decode_scratch[kDecodeStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};
void* g_scratch_ptr[kMaxDevices] = {nullptr};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (the
// library does not link libcuda directly).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of the scratch array in the current device's current
// context, looked up once per (device, context).
cudaError_t scratch_address(int dev, void** out) {
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr) return cudaErrorNotSupported;
  // no context is current before the runtime's first use of the device;
  // the lookup below binds the primary one
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (ctx == nullptr || g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
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
  // every check of paged_attn_decode runs before anything touches the
  // shared array, so a rejected call enqueues nothing
  const pkv_status chk = pkv::decode_check_args(out, q, k_cache, v_cache, block_table,
                                                max_blocks_per_seq, seq_lens, batch, num_q_heads,
                                                num_kv_heads, head_dim, page_size, num_pages,
                                                max_seq_len, scale);
  if (chk != PKV_OK || batch == 0) return chk;
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
