// C ABI layer: argument validation, TMA descriptor encoding, dispatch.
// Declarations and the contract of every entry point are in include/pkv.h.
#include <string.h>

#include <mutex>
#include <string>

#include "../../include/pkv.h"
#include "kernels.h"
#include "tmap.h"

using pkv::encode_pool_map_groups;
using pkv::encode_q_map;

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

bool supported_head_dim(int D) { return D == 64 || D == 128 || D == 256; }
// decode also runs the 512-wide heads of full-attention layers
bool decode_head_dim(int D) { return supported_head_dim(D) || D == 512; }

}  // namespace

namespace pkv {
void set_last_error(const std::string& msg) { g_last_cuda_error = msg; }

pkv_status decode_check_args(const void* out, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* block_table,
                             int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t page_size, int64_t num_pages, int32_t max_seq_len,
                             float scale) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      num_pages <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0)
    return PKV_ERR_INVALID;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID;
  if (!(scale == scale)) return PKV_ERR_INVALID;  // NaN
  if (!decode_head_dim(head_dim) || page_size % 16 != 0 || num_q_heads / num_kv_heads > 8 ||
      num_pages * (int64_t)num_kv_heads > 0x7fffffffLL || batch > 4096)
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens) return PKV_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID;
  return PKV_OK;
}
}  // namespace pkv

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

pkv_status pkv_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return PKV_OK;
  if (!dst || !src || bytes % 16 != 0 || !aligned16(dst) || !aligned16(src))
    return PKV_ERR_INVALID;
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
  if (d < s + bytes && s < d + bytes) return PKV_ERR_INVALID;  // overlapping ranges
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  // both ends must be memory this device reaches at the same address:
  // its own device memory, or host memory pinned through CUDA (mapped at
  // the same address under unified addressing)
  for (const void* p : {static_cast<const void*>(dst), src}) {
    cudaPointerAttributes at;
    e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) return cuda_fail(e);
    const bool ok = (at.type == cudaMemoryTypeDevice && at.device == dev) ||
                    (at.type == cudaMemoryTypeManaged) ||
                    (at.type == cudaMemoryTypeHost && at.devicePointer == p);
    if (!ok) {
      g_last_cuda_error =
          "pkv_copy: each pointer must be device memory of the current device or pinned host "
          "memory mapped at the same address";
      return PKV_ERR_UNSUPPORTED;
    }
  }
  int sms = 0;
  if (int err = num_sms_current(&sms)) return cuda_fail((cudaError_t)err);
  e = pkv::launch_copy16(dst, src, (int64_t)(bytes / 16), static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

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
  if ((int64_t)num_tokens * num_kv_heads * (head_dim / 8) >= (int64_t(1) << 31))
    return PKV_ERR_UNSUPPORTED;
  cudaError_t e = pkv::launch_kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, num_tokens,
                                        num_kv_heads, head_dim, page_size, num_pages, err_flag,
                                        static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

size_t paged_attn_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
      !decode_head_dim(head_dim))
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
  const pkv_status chk =
      pkv::decode_check_args(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                             batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                             max_seq_len, scale);
  if (chk != PKV_OK || batch == 0) return chk;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  if (workspace_bytes <
      pkv::decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, sms))
    return PKV_ERR_INVALID;
  cudaError_t e = pkv::launch_decode(
      out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, batch, num_q_heads,
      num_kv_heads, head_dim, page_size, num_pages, max_seq_len, scale, window, workspace,
      workspace_bytes, err_flag, static_cast<cudaStream_t>(stream), sms);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

pkv_status paged_attn_decode_append(void* out, const void* q, const void* k_new,
                                    const void* v_new, void* k_cache, void* v_cache,
                                    const int32_t* block_table, int32_t max_blocks_per_seq,
                                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                    int64_t num_pages, int32_t max_seq_len, float scale,
                                    int32_t window, void* workspace, size_t workspace_bytes,
                                    int32_t* err_flag, void* stream) {
  const pkv_status chk =
      pkv::decode_check_args(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                             batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                             max_seq_len, scale);
  if (chk != PKV_OK || batch == 0) return chk;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  if (workspace_bytes <
      pkv::decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, sms))
    return PKV_ERR_INVALID;
  const pkv::DecodeAppend app = {k_new, v_new};
  cudaError_t e = pkv::launch_decode(
      out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, batch, num_q_heads,
      num_kv_heads, head_dim, page_size, num_pages, max_seq_len, scale, window, workspace,
      workspace_bytes, err_flag, static_cast<cudaStream_t>(stream), sms, nullptr, &app);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

size_t paged_attn_decode_shared_prefix_workspace_size(int32_t batch, int32_t num_q_heads,
                                                      int32_t num_kv_heads, int32_t head_dim) {
  if (!supported_head_dim(head_dim)) return 0;
  const size_t dec =
      paged_attn_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim);
  if (dec == 0) return 0;
  const size_t rows = (size_t)batch * num_q_heads;
  return align256(dec) + align256(rows * 4) + align256(rows * head_dim * 4);
}

pkv_status paged_attn_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t batch, int32_t group_size, const int32_t* prefix_lens, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t page_size, int64_t num_pages,
    int32_t max_seq_len, float scale, void* workspace, size_t workspace_bytes,
    int32_t* err_flag, void* stream) {
  const pkv_status chk =
      pkv::decode_check_args(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                             batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                             max_seq_len, scale);
  if (chk != PKV_OK) return chk;
  if (group_size < 1) return PKV_ERR_INVALID;
  if (!supported_head_dim(head_dim) ||
      group_size * (num_q_heads / num_kv_heads) > pkv::prefix_max_rows(head_dim))
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!prefix_lens || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  const size_t dec = align256(
      pkv::decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, sms));
  const size_t rows = (size_t)batch * num_q_heads;
  if (workspace_bytes < dec + align256(rows * 4) + align256(rows * head_dim * 4))
    return PKV_ERR_INVALID;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* pre_lse = reinterpret_cast<float*>(ws + dec);
  float* pre_o = reinterpret_cast<float*>(ws + dec + align256(rows * 4));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = pkv::launch_prefix_pass(q, k_cache, v_cache, block_table, max_blocks_per_seq,
                                          seq_lens, prefix_lens, batch, group_size, num_q_heads,
                                          num_kv_heads, head_dim, page_size, num_pages, scale,
                                          pre_o, pre_lse, err_flag, st, sms);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return cuda_fail(e);
  pkv::DecodeCascade cas = {prefix_lens, group_size, pre_o, pre_lse};
  e = pkv::launch_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                         batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                         max_seq_len, scale, 0, workspace, dec, err_flag, st, sms, &cas);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
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
  if (!(scale >= 0.f)) return PKV_ERR_INVALID;  // NaN or negative
  if (causal != 0 && causal != 1) return PKV_ERR_INVALID;
  if (!causal && window > 0) return PKV_ERR_INVALID;
  const int G = num_q_heads / num_kv_heads;
  if (!decode_head_dim(head_dim) || page_size % 16 != 0 || (128 % G) != 0 ||
      num_pages * (int64_t)num_kv_heads > 0x7fffffffLL || batch > 1024)
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !cu_seq_lens_q || !cu_seq_lens_k || !block_table)
    return PKV_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  pkv::VarlenMaps maps;
  const int kv_rows = pkv::varlen_kv_tile(head_dim);  // keys per KV tile
  const int box_rows = page_size < kv_rows ? page_size : kv_rows;
  // a KV tile must be whole page slices: page_size divides it or is a
  // multiple of it
  if (kv_rows % page_size != 0 && page_size % kv_rows != 0) return PKV_ERR_UNSUPPORTED;
  if (!encode_q_map(&maps.q, q, head_dim, G, num_kv_heads, total_q) ||
      !encode_pool_map_groups(&maps.k, k_cache, head_dim, page_size, num_pages, num_kv_heads,
                              box_rows) ||
      !encode_pool_map_groups(&maps.v, v_cache, head_dim, page_size, num_pages, num_kv_heads,
                              box_rows, pkv::varlen_v_cols(head_dim)))
    return cuda_fail(cudaErrorInvalidValue);
  cudaError_t e = pkv::launch_varlen(out, maps, cu_seq_lens_q, cu_seq_lens_k, block_table,
                                     max_blocks_per_seq, batch, max_seqlen_q, total_q,
                                     num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                                     scale, causal, window, err_flag,
                                     static_cast<cudaStream_t>(stream), sms);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

static pkv_status mixed_impl(void* dec_out, const void* dec_q, const int32_t* dec_block_table,
                            int32_t dec_max_blocks_per_seq, const int32_t* dec_seq_lens,
                            int32_t dec_batch, int32_t dec_max_seq_len, void* pre_out,
                            const void* pre_q, const int32_t* cu_seq_lens_q,
                            const int32_t* cu_seq_lens_k, const int32_t* pre_block_table,
                            int32_t pre_max_blocks_per_seq, int32_t pre_batch,
                            int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t total_q,
                            const void* k_cache, const void* v_cache, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                            int64_t num_pages, float scale, int32_t window, int32_t decode_ctas,
                            void* workspace, size_t workspace_bytes, int32_t* err_flag,
                            void* stream, const void* k_new, const void* v_new,
                            const int64_t* slot_mapping, int32_t num_new) {
  if (dec_batch < 0 || pre_batch < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return PKV_ERR_INVALID;
  if (!(scale >= 0.f)) return PKV_ERR_INVALID;  // NaN or negative
  // the decode half: every check of paged_attn_decode
  const pkv_status chk =
      pkv::decode_check_args(dec_out, dec_q, k_cache, v_cache, dec_block_table,
                             dec_batch > 0 ? dec_max_blocks_per_seq : 1, dec_seq_lens, dec_batch,
                             num_q_heads, num_kv_heads, head_dim, page_size, num_pages,
                             dec_max_seq_len, scale);
  if (chk != PKV_OK) return chk;
  // the prefill half: the checks of paged_attn_varlen (causal)
  const int G = num_q_heads / num_kv_heads;
  const bool has_var = pre_batch > 0 && total_q > 0;
  if (has_var) {
    if (pre_max_blocks_per_seq <= 0) return PKV_ERR_INVALID;
    if (!pre_out || !pre_q || !cu_seq_lens_q || !cu_seq_lens_k || !pre_block_table)
      return PKV_ERR_INVALID;
    if (!aligned16(pre_out) || !aligned16(pre_q)) return PKV_ERR_INVALID;
    if ((128 % G) != 0 || pre_batch > 1024) return PKV_ERR_UNSUPPORTED;
  }
  if (head_dim != 128 || (128 % page_size != 0 && page_size % 128 != 0))
    return PKV_ERR_UNSUPPORTED;
  if (num_new < 0) return PKV_ERR_INVALID;
  if (num_new > 0) {
    // the new rows and their slots; the grid barrier's counters live in the
    // workspace, which every appending call needs
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new))
      return PKV_ERR_INVALID;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PKV_ERR_INVALID;
  }
  if (dec_batch == 0 && !has_var && num_new == 0) return PKV_OK;
  if (dec_batch > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  if ((dec_batch > 0 || num_new > 0) &&
      workspace_bytes <
          pkv::decode_workspace_bytes(dec_batch, num_q_heads, num_kv_heads, head_dim, sms))
    return PKV_ERR_INVALID;
  pkv::VarlenMaps maps;
  if (has_var) {
    const int box_rows = page_size < 128 ? page_size : 128;
    if (!encode_q_map(&maps.q, pre_q, head_dim, G, num_kv_heads, total_q) ||
        !encode_pool_map_groups(&maps.k, k_cache, head_dim, page_size, num_pages, num_kv_heads,
                                box_rows) ||
        !encode_pool_map_groups(&maps.v, v_cache, head_dim, page_size, num_pages, num_kv_heads,
                                box_rows))
      return cuda_fail(cudaErrorInvalidValue);
  } else {
    memset(&maps, 0, sizeof(maps));
  }
  pkv::MixedLaunch L;
  L.dec_out = dec_out;
  L.dec_q = dec_q;
  L.dec_block_table = dec_block_table;
  L.dec_seq_lens = dec_seq_lens;
  L.dec_max_blocks = dec_max_blocks_per_seq;
  L.dec_batch = dec_batch;
  L.dec_max_seq_len = dec_max_seq_len;
  L.pre_out = pre_out;
  L.pre_q = pre_q;
  L.cu_q = cu_seq_lens_q;
  L.cu_k = cu_seq_lens_k;
  L.pre_block_table = pre_block_table;
  L.pre_max_blocks = pre_max_blocks_per_seq;
  L.pre_batch = has_var ? pre_batch : 0;
  L.max_seqlen_q = max_seqlen_q;
  L.max_seqlen_k = max_seqlen_k;
  L.total_q = total_q;
  L.k_cache = k_cache;
  L.v_cache = v_cache;
  L.H_q = num_q_heads;
  L.H_kv = num_kv_heads;
  L.D = head_dim;
  L.P = page_size;
  L.num_pages = num_pages;
  L.scale = scale;
  L.window = window;
  L.decode_ctas = decode_ctas;
  L.workspace = workspace;
  L.workspace_bytes = workspace_bytes;
  L.err = err_flag;
  L.k_new = k_new;
  L.v_new = v_new;
  L.slot_mapping = slot_mapping;
  L.num_new = num_new;
  cudaError_t e = pkv::launch_mixed(L, maps, static_cast<cudaStream_t>(stream), sms);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

pkv_status paged_attn_mixed(void* dec_out, const void* dec_q, const int32_t* dec_block_table,
                            int32_t dec_max_blocks_per_seq, const int32_t* dec_seq_lens,
                            int32_t dec_batch, int32_t dec_max_seq_len, void* pre_out,
                            const void* pre_q, const int32_t* cu_seq_lens_q,
                            const int32_t* cu_seq_lens_k, const int32_t* pre_block_table,
                            int32_t pre_max_blocks_per_seq, int32_t pre_batch,
                            int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t total_q,
                            const void* k_cache, const void* v_cache, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                            int64_t num_pages, float scale, int32_t window, int32_t decode_ctas,
                            void* workspace, size_t workspace_bytes, int32_t* err_flag,
                            void* stream) {
  return mixed_impl(dec_out, dec_q, dec_block_table, dec_max_blocks_per_seq, dec_seq_lens,
                    dec_batch, dec_max_seq_len, pre_out, pre_q, cu_seq_lens_q, cu_seq_lens_k,
                    pre_block_table, pre_max_blocks_per_seq, pre_batch, max_seqlen_q,
                    max_seqlen_k, total_q, k_cache, v_cache, num_q_heads, num_kv_heads,
                    head_dim, page_size, num_pages, scale, window, decode_ctas, workspace,
                    workspace_bytes, err_flag, stream, nullptr, nullptr, nullptr, 0);
}

pkv_status paged_attn_mixed_append(
    void* dec_out, const void* dec_q, const int32_t* dec_block_table,
    int32_t dec_max_blocks_per_seq, const int32_t* dec_seq_lens, int32_t dec_batch,
    int32_t dec_max_seq_len, void* pre_out, const void* pre_q, const int32_t* cu_seq_lens_q,
    const int32_t* cu_seq_lens_k, const int32_t* pre_block_table, int32_t pre_max_blocks_per_seq,
    int32_t pre_batch, int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t total_q,
    const void* k_new, const void* v_new, const int64_t* slot_mapping, int32_t num_new_tokens,
    void* k_cache, void* v_cache, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t page_size, int64_t num_pages, float scale, int32_t window, int32_t decode_ctas,
    void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream) {
  return mixed_impl(dec_out, dec_q, dec_block_table, dec_max_blocks_per_seq, dec_seq_lens,
                    dec_batch, dec_max_seq_len, pre_out, pre_q, cu_seq_lens_q, cu_seq_lens_k,
                    pre_block_table, pre_max_blocks_per_seq, pre_batch, max_seqlen_q,
                    max_seqlen_k, total_q, k_cache, v_cache, num_q_heads, num_kv_heads,
                    head_dim, page_size, num_pages, scale, window, decode_ctas, workspace,
                    workspace_bytes, err_flag, stream, k_new, v_new, slot_mapping,
                    num_new_tokens);
}

pkv_status pkv_rope_table(float* cos_sin, int32_t max_position, int32_t head_dim,
                          double theta, void* stream) {
  if (max_position < 0 || head_dim <= 0 || head_dim % 2 != 0) return PKV_ERR_INVALID;
  if (!(theta > 0.0) || theta > 1e300) return PKV_ERR_INVALID;  // NaN, <= 0 or infinite
  if (max_position == 0) return PKV_OK;
  if (!cos_sin || !aligned16(cos_sin)) return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  cudaError_t e = pkv::launch_rope_table(cos_sin, max_position, head_dim, theta,
                                         static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

pkv_status paged_kv_append_rope(void* q, const void* k_new, const void* v_new, void* k_cache,
                                void* v_cache, const int64_t* slot_mapping,
                                const int32_t* positions, const float* cos_sin,
                                int32_t max_position, const void* q_norm_weight,
                                const void* k_norm_weight, float norm_eps, int32_t num_tokens,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t page_size, int64_t num_pages, int32_t* err_flag,
                                void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
      num_pages <= 0 || max_position <= 0 || (q && num_q_heads <= 0))
    return PKV_ERR_INVALID;
  if (!(norm_eps >= 0.f) || norm_eps > 3e38f) return PKV_ERR_INVALID;  // NaN, < 0, inf
  if (!supported_head_dim(head_dim)) return PKV_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)num_tokens * ((q ? num_q_heads : 0) + (int64_t)num_kv_heads);
  if (rows * (head_dim / 8) >= (int64_t(1) << 30)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping || !positions || !cos_sin)
    return PKV_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(cos_sin) || (q && !aligned16(q)) || (q_norm_weight && !aligned16(q_norm_weight)) ||
      (k_norm_weight && !aligned16(k_norm_weight)))
    return PKV_ERR_INVALID;
  int sms = 0;
  if (int e = num_sms_current(&sms)) return cuda_fail((cudaError_t)e);
  pkv::RopeAppendArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.slot_mapping = slot_mapping;
  a.positions = positions;
  a.cos_sin = cos_sin;
  a.q_w = q ? q_norm_weight : nullptr;
  a.k_w = k_norm_weight;
  a.eps = norm_eps;
  a.max_pos = max_position;
  a.T = num_tokens;
  a.H_q = q ? num_q_heads : 0;
  a.H_kv = num_kv_heads;
  a.P = page_size;
  a.P_shift = -1;
  for (int sh = 0; sh < 31; ++sh)
    if ((1 << sh) == page_size) a.P_shift = sh;
  a.num_slots = num_pages * (int64_t)page_size;
  a.err = err_flag;
  cudaError_t e =
      pkv::launch_kv_append_rope(a, head_dim, static_cast<cudaStream_t>(stream), sms);
  if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

}  // extern "C"
