// Internal launch interface between the C ABI layer (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/pkv.h"

namespace pkv {

// Message returned by pkv_last_cuda_error() on this host thread.
void set_last_error(const std::string& msg);

// Host-side argument checks of paged_attn_decode, everything but the
// workspace (PKV_OK, PKV_ERR_INVALID or PKV_ERR_UNSUPPORTED; nothing is
// enqueued).
pkv_status decode_check_args(const void* out, const void* q, const void* k_cache,
                             const void* v_cache,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             int64_t num_pages, int32_t max_seq_len, float scale);

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t num_tokens, int32_t H_kv,
                             int32_t D, int32_t P, int64_t num_pages, int32_t* err,
                             cudaStream_t stream, int num_sms);

// n16 16-byte words from src to dst by the SMs (copy.cu)
cudaError_t launch_copy16(void* dst, const void* src, int64_t n16, cudaStream_t stream,
                          int num_sms);

// Arguments of the fused norm + rotary + append kernel (rope_append.cu).
struct RopeAppendArgs {
  void* q;                      // [T, H_q, D] bf16, transformed in place; null: no q
  const void* k_new;            // [T, H_kv, D] bf16
  const void* v_new;            // [T, H_kv, D] bf16
  void* k_cache;                // [num_pages, H_kv, P, D] bf16
  void* v_cache;
  const int64_t* slot_mapping;  // [T]
  const int32_t* positions;     // [T]
  const float* cos_sin;         // [max_pos, D] f32: cos in [0, D/2), sin in [D/2, D)
  const void* q_w;              // [D] bf16 RMSNorm weight of q, or null (no norm)
  const void* k_w;              // [D] bf16 RMSNorm weight of k, or null
  float eps;
  int32_t max_pos, T, H_q, H_kv, P;
  int32_t P_shift;              // log2(P) when P is a power of two, else -1
  int64_t num_slots;
  int32_t* err;
};

cudaError_t launch_rope_table(float* cos_sin, int32_t max_pos, int32_t D, double theta,
                              cudaStream_t stream, int num_sms);

cudaError_t launch_kv_append_rope(const RopeAppendArgs& a, int32_t D, cudaStream_t stream,
                                  int num_sms);

// kv heads per decode work item: two for head_dim 128 with an even number
// of kv heads and a GQA group of at most 4 (one TMA box then carries both
// heads' slice of a page: half the boxes per byte, +20-27 % per-SM decode
// rate), else one.
#ifndef PKV_DEC_HP2
#define PKV_DEC_HP2 1
#endif
inline int decode_heads_per_item(int32_t D, int32_t H_kv, int32_t G) {
  return (PKV_DEC_HP2 && D == 128 && H_kv % 2 == 0 && G >= 1 && G <= 4) ? 2 : 1;
}

size_t decode_workspace_bytes(int32_t batch, int32_t H_q, int32_t H_kv, int32_t D, int num_sms);

// Shared-prefix (cascade) inputs of the decode kernel: the groups' prefix
// lengths and the prefix pass's partials ([batch * H_q, D] and [batch * H_q]).
struct DecodeCascade {
  const int32_t* prefix_lens;
  int32_t group_size;
  const float* pre_o;
  const float* pre_lse;
};

// Fused append of the decode step: each sequence's newest K/V row, written
// by the decode kernel to position seq_lens[b] - 1 ([batch, H_kv, D] bf16;
// the pools as written by paged_kv_append).
struct DecodeAppend {
  const void* k_new;
  const void* v_new;
};

cudaError_t launch_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, int32_t max_blocks,
                          const int32_t* seq_lens, int32_t batch, int32_t H_q, int32_t H_kv,
                          int32_t D, int32_t P, int64_t num_pages, int32_t max_seq_len,
                          float scale, int32_t window, void* workspace, size_t workspace_bytes,
                          int32_t* err, cudaStream_t stream, int num_sms,
                          const DecodeCascade* cascade = nullptr,
                          const DecodeAppend* append = nullptr);

// Prefix pass of the cascade: partial (o, log2-sum-exp) of every member row
// over its group's shared prefix.  Query rows per (group, kv head) are
// group_size * H_q / H_kv, at most prefix_max_rows(D).
int prefix_max_rows(int D);
cudaError_t launch_prefix_pass(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* seq_lens, const int32_t* prefix_lens,
                               int32_t batch, int32_t group_size, int32_t H_q, int32_t H_kv,
                               int32_t D, int32_t P, int64_t num_pages, float scale,
                               float* pre_o, float* pre_lse, int32_t* err, cudaStream_t stream,
                               int num_sms);

struct VarlenMaps {
  CUtensorMap q;  // 4-D view of q: {D, G, H_kv, total_q}
  CUtensorMap k;  // 3-D view of the K pool: {D, P, num_pages*H_kv}
  CUtensorMap v;  // same for V
};

// Arguments of the single-launch mixed step (mixed.cu): decode rows and
// causal prefill chunks over one pool.
struct MixedLaunch {
  void* dec_out;
  const void* dec_q;
  const int32_t* dec_block_table;
  const int32_t* dec_seq_lens;
  int32_t dec_max_blocks, dec_batch, dec_max_seq_len;
  void* pre_out;
  const void* pre_q;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* pre_block_table;
  int32_t pre_max_blocks, pre_batch, max_seqlen_q, max_seqlen_k, total_q;
  const void* k_cache;
  const void* v_cache;
  int32_t H_q, H_kv, D, P;
  int64_t num_pages;
  float scale;
  int32_t window;
  int32_t decode_ctas;  // CTAs that start with decode; <= 0: chosen here
  void* workspace;
  size_t workspace_bytes;
  int32_t* err;
  // the fused append (paged_attn_mixed_append): num_new tokens' K/V rows
  // ([num_new, H_kv, D]) to the pools at slot_mapping; num_new = 0: none
  const void* k_new;
  const void* v_new;
  const int64_t* slot_mapping;
  int32_t num_new;
};

// keys per KV tile of the varlen kernel for a head_dim (page_size must
// divide it or be a multiple of it)
int varlen_kv_tile(int head_dim);
// columns of V (and of O) one varlen work item covers (head_dim, or half of
// it at 512)
int varlen_v_cols(int head_dim);

cudaError_t launch_mixed(const MixedLaunch& L, const VarlenMaps& vmaps, cudaStream_t stream,
                         int num_sms);

cudaError_t launch_varlen(void* out, const VarlenMaps& maps, const int32_t* cu_q,
                          const int32_t* cu_k, const int32_t* block_table, int32_t max_blocks,
                          int32_t batch, int32_t max_seqlen_q, int32_t total_q, int32_t H_q,
                          int32_t H_kv, int32_t D, int32_t P, int64_t num_pages, float scale,
                          int32_t causal, int32_t window, int32_t* err, cudaStream_t stream,
                          int num_sms);

}  // namespace pkv
