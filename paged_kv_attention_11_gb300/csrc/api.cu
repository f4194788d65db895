// C ABI layer: argument validation, TMA descriptor encoding, dispatch.
// Declarations and the contract of every entry point are in include/pkv.h.
#include <mutex>
#include <string>

#include "../../include/pkv.h"
#include "kernels.h"

namespace {

thread_local std::string g_last_cuda_error;

pkv_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = cudaGetErrorString(e);
  return PKV_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;

int num_sms_current(int* out) {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  if (cache[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    cache[dev] = n;
  }
  *out = cache[dev];
  return 0;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// K or V pool [num_pages, H_kv, P, D] bf16 viewed as {D, P, num_pages*H_kv};
// box = 64 columns x 16 rows, 128-byte swizzle.
bool encode_pool_map(CUtensorMap* m, const void* base, int D, int P, int64_t num_pages,
                     int H_kv) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)P, (cuuint64_t)(num_pages * H_kv)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)P * D * 2};
  cuuint32_t box[3] = {64, 16, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K or V pool for the varlen kernel: same view, box = 64 columns x `rows` rows.
bool encode_pool_map_rows(CUtensorMap* m, const void* base, int D, int P, int64_t num_pages,
                          int H_kv, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)P, (cuuint64_t)(num_pages * H_kv)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)P * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [total_q, H_q, D] viewed as {D, G, H_kv, total_q}; box = 64 x G x 1 x (128/G)
// so one box holds 128 (position, head) rows of one kv group.
bool encode_q_map(CUtensorMap* m, const void* base, int D, int G, int H_kv, int total_q) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)G, (cuuint64_t)H_kv, (cuuint64_t)total_q};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)G * D * 2,
                           (cuuint64_t)H_kv * G * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(128 / G)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool supported_head_dim(int D) { return D == 64 || D == 128 || D == 256; }

}  // namespace

extern "C" {

const char* pkv_status_string(int32_t s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID: return "PKV_ERR_INVALID";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    default: return "PKV_UNKNOWN_STATUS";
  }
}

const char* pkv_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

pkv_status paged_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int32_t page_size, int64_t num_pages,
                           int32_t* err_flag, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0)
    return PKV_ERR_INVALID;
  if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  cudaError_t e = pkv::launch_kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                                        num_kv_heads, head_dim, page_size, num_pages, err_flag,
                                        static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

size_t paged_attn_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
      !supported_head_dim(head_dim))
    return 0;
  int sms = 0;
  if (num_sms_current(&sms) != 0) return 0;
  return pkv::decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, sms);
}

pkv_status paged_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             int64_t num_pages, int32_t max_seq_len, float scale, int32_t window,
                             void* workspace, size_t workspace_bytes, int32_t* err_flag,
                             void* stream) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      num_pages <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0)
    return PKV_ERR_INVALID;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID;
  if (!(scale == scale)) return PKV_ERR_INVALID;  // NaN
  if (!supported_head_dim(head_dim) || page_size % 16 != 0 || num_q_heads / num_kv_heads > 8 ||
      num_pages * (int64_t)num_kv_heads > 0x7fffffffLL || batch > 16384)
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens || !workspace)
    return PKV_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  if (workspace_bytes <
      pkv::decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, sms))
    return PKV_ERR_INVALID;
  CUtensorMap tmK, tmV;
  if (!encode_pool_map(&tmK, k_cache, head_dim, page_size, num_pages, num_kv_heads) ||
      !encode_pool_map(&tmV, v_cache, head_dim, page_size, num_pages, num_kv_heads))
    return cuda_fail(cudaErrorInvalidValue);
  cudaError_t e = pkv::launch_decode(
      out, q, tmK, tmV, block_table, max_blocks_per_seq, seq_lens, batch, num_q_heads,
      num_kv_heads, head_dim, page_size, num_pages, max_seq_len, scale, window, workspace,
      err_flag, static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

pkv_status paged_attn_varlen(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* cu_seq_lens_q, const int32_t* cu_seq_lens_k,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             int32_t batch, int32_t max_seqlen_q, int32_t max_seqlen_k,
                             int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t page_size, int64_t num_pages, float scale,
                             int32_t causal, int32_t window, int32_t* err_flag, void* stream) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      num_pages <= 0 || max_blocks_per_seq <= 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
      total_q < 0)
    return PKV_ERR_INVALID;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID;
  if (!(scale == scale)) return PKV_ERR_INVALID;
  if (causal != 0 && causal != 1) return PKV_ERR_INVALID;
  if (!causal && window > 0) return PKV_ERR_INVALID;
  const int G = num_q_heads / num_kv_heads;
  if (!supported_head_dim(head_dim) || page_size % 16 != 0 || (128 % G) != 0 ||
      num_pages * (int64_t)num_kv_heads > 0x7fffffffLL)
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !cu_seq_lens_q || !cu_seq_lens_k || !block_table)
    return PKV_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  pkv::VarlenMaps maps;
  const int kv_rows = head_dim == 256 ? 64 : 128;  // keys per KV tile
  const int box_rows = page_size < kv_rows ? page_size : kv_rows;
  // a KV tile must be whole page slices: page_size divides it or is a
  // multiple of it
  if (kv_rows % page_size != 0 && page_size % kv_rows != 0) return PKV_ERR_UNSUPPORTED;
  if (!encode_q_map(&maps.q, q, head_dim, G, num_kv_heads, total_q) ||
      !encode_pool_map_rows(&maps.k, k_cache, head_dim, page_size, num_pages, num_kv_heads,
                            box_rows) ||
      !encode_pool_map_rows(&maps.v, v_cache, head_dim, page_size, num_pages, num_kv_heads,
                            box_rows))
    return cuda_fail(cudaErrorInvalidValue);
  cudaError_t e = pkv::launch_varlen(out, maps, cu_seq_lens_q, cu_seq_lens_k, block_table,
                                     max_blocks_per_seq, batch, max_seqlen_q, total_q,
                                     num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                                     scale, causal, window, err_flag,
                                     static_cast<cudaStream_t>(stream), sms);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

}  // extern "C"
