// paged_attn_decode: the split-KV decode kernel (its body, decode_cta, is in
// decode_body.cuh) and its host-side launch.
#include "decode_body.cuh"
#include "tmap.h"

namespace pkv {

template <int D, int NW, int NSTAGE, bool APPEND, int HP>
__global__ void __launch_bounds__((NW + 2) * 32, 1)
    decode_split_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  decode_cta<D, NW, NSTAGE, false, APPEND, HP>(a, tmK, tmV, smem, blockIdx.x);
}

// --------------------------------------------------------------- host side
// Launch shape per head_dim: consumer warps, pipeline stages (16-key K+V
// tiles) per CTA, resident CTAs per SM.  Overridable at build time for
// tuning sweeps.
#ifndef PKV_DEC_NW
#define PKV_DEC_NW 4
#endif
#ifndef PKV_DEC_NSTAGE
#define PKV_DEC_NSTAGE 24  // 192 KB of K/V in flight per SM; 16 when the batch's plan needs room
#endif
#ifndef PKV_DEC_CTAS
#define PKV_DEC_CTAS 1
#endif
template <int D>
struct DecodeCfg;
template <> struct DecodeCfg<64> { static constexpr int NW = 4, NSTAGE = 16, CTAS_PER_SM = 1; };
template <> struct DecodeCfg<128> {
  static constexpr int NW = PKV_DEC_NW, NSTAGE = PKV_DEC_NSTAGE, CTAS_PER_SM = PKV_DEC_CTAS;
};
template <> struct DecodeCfg<256> { static constexpr int NW = 4, NSTAGE = 8, CTAS_PER_SM = 1; };
template <> struct DecodeCfg<512> { static constexpr int NW = 2, NSTAGE = 4, CTAS_PER_SM = 1; };

static int decode_ctas_per_sm(int D) {
  switch (D) {
    case 64: return DecodeCfg<64>::CTAS_PER_SM;
    case 128: return DecodeCfg<128>::CTAS_PER_SM;
    case 256: return DecodeCfg<256>::CTAS_PER_SM;
    default: return DecodeCfg<512>::CTAS_PER_SM;
  }
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Work items (and so partial slots) are at most one per segment plus 2 per
// CTA: a segment is cut into chunks of >= W/(2N) tiles.  A slot holds the
// item's HP * G query rows.
static int64_t decode_max_rows(int32_t batch, int32_t H_kv, int32_t G, int32_t D, int num_sms) {
  const int HP = decode_heads_per_item(D, H_kv, G);
  const int64_t pieces = (int64_t)batch * (H_kv / HP) + 2 * (int64_t)num_sms * decode_ctas_per_sm(D);
  return pieces * G * HP;
}

// Workspace: [seg_count: batch*H_kv int32][merge_jobs: batch*H_kv int32]
//            [queue: 8 int32] ... [part_lse: pieces*G f32][part_o: pieces*G*D f32]
// (partials aligned to the end of the caller's buffer)
size_t decode_workspace_bytes(int32_t batch, int32_t H_q, int32_t H_kv, int32_t D, int num_sms) {
  const int64_t rows = decode_max_rows(batch, H_kv, H_q / H_kv, D, num_sms);
  return align256(((size_t)batch * H_kv * 2 + 8) * 4) + align256((size_t)rows * 4) +
         align256((size_t)rows * D * 4);
}

// Counters sit at the front and the partial results at the back of the
// workspace, so calls with different batch sizes that share one workspace
// never see each other's partials in their counter slots.
void decode_workspace_split(DecodeArgs& a, void* workspace, size_t workspace_bytes,
                            int32_t batch, int32_t H_kv, int32_t D, int num_sms) {
  const int64_t rows = decode_max_rows(batch, H_kv, a.G, D, num_sms);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.seg_count = reinterpret_cast<int32_t*>(ws);
  a.merge_jobs = a.seg_count + (int64_t)batch * H_kv;
  a.queue = a.merge_jobs + (int64_t)batch * H_kv;
  uint8_t* end = ws + (workspace_bytes & ~size_t(255));
  end -= align256((size_t)rows * D * 4);
  a.part_o = reinterpret_cast<float*>(end);
  end -= align256((size_t)rows * 4);
  a.part_lse = reinterpret_cast<float*>(end);
}

template <int D, int NW, int NSTAGE, bool APPEND, int HP = 1>
static cudaError_t launch_decode_s(DecodeArgs a, const void* k_cache, const void* v_cache,
                                   int max_seq_len, cudaStream_t stream, int num_sms) {
  using C = DecodeCfg<D>;
  using P_ = DecodePlan<D, NW, NSTAGE, HP>;
  auto kern = decode_split_kernel<D, NW, NSTAGE, APPEND, HP>;
  (void)max_seq_len;
  // one TMA box per 16-key K or V tile (all D columns of one page and the
  // item's HP heads)
  CUtensorMap tmK, tmV;
  const bool enc_ok =
      encode_pool_map_groups(&tmK, k_cache, D, a.P, a.num_pages, a.H_kv, kTile, 0, HP) &&
      encode_pool_map_groups(&tmV, v_cache, D, a.P, a.num_pages, a.H_kv, kTile, 0, HP);
  if (!enc_ok) return cudaErrorInvalidValue;
  const size_t smem = P_(a.G, a.batch).total;
  if (smem > 227 * 1024) return cudaErrorNotSupported;
  // Raise the dynamic shared-memory limit once per device (and again only
  // if a larger batch needs more); cache the resident CTAs per SM for it.
  static int configured[64] = {0};
  static int occupancy[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] != (int)smem) {
    if (configured[dev] < (int)smem) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, (NW + 2) * 32, smem);
    if (e != cudaSuccess) return e;
    if (configured[dev] < (int)smem) configured[dev] = (int)smem;
    occupancy[dev] = occ;
  }
  int per_sm = occupancy[dev] < C::CTAS_PER_SM ? occupancy[dev] : C::CTAS_PER_SM;
  if (per_sm < 1) per_sm = 1;
  // persistent grid: every resident CTA takes items until the queue is empty
  const int64_t n = (int64_t)num_sms * per_sm;
  a.cta_count = (int32_t)n;
  // the cut rule's share: with two-head items on every SM, a segment is cut
  // above half of a CTA's share of keys x heads (items of one head would be
  // cut there too); the mixed-step kernel, whose decode starts on part of
  // the SMs, keeps the finer cut of half a share of items
  a.share_ctas = (int32_t)(HP == 2 ? (n + 1) / 2 : n);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n);
  cfg.blockDim = dim3((NW + 2) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tmK, tmV);
}

// The configured shape when the batch's shared-memory plan leaves room for
// it, else smaller rings (then fewer consumer warps): large batches need
// room for the per-sequence schedule arrays.
template <int D, int NW, int NSTAGE, int HP = 1>
static bool decode_fits(const DecodeArgs& a) {
  return DecodePlan<D, NW, NSTAGE, HP>(a.G, a.batch).total <= 227 * 1024;
}

template <int D, bool APPEND>
static cudaError_t launch_decode_t(DecodeArgs a, const void* k_cache, const void* v_cache,
                                   int max_seq_len, cudaStream_t stream, int num_sms) {
  using C = DecodeCfg<D>;
  if constexpr (D == 256) {
    // A small call (at most ~1 MB of K/V per SM: a few windows or short
    // rows) runs at the per-SM streaming rate, not HBM's: 2 consumer warps
    // and 10 stages of 16 KB (160 KB in flight) beat 4 warps and 8 stages
    // there (sliding-window decode, 32 rows of a 512-key window: 20.5 vs
    // 22.5 us).  Larger calls keep 4 consumer warps.
    const int64_t keys = (a.window > 0 && a.window < max_seq_len) ? a.window : max_seq_len;
    const int64_t bytes = (int64_t)a.batch * a.H_kv * keys * D * 4;
    if (bytes <= ((int64_t)num_sms << 20) && decode_fits<D, 2, 10>(a))
      return launch_decode_s<D, 2, 10, APPEND>(a, k_cache, v_cache, max_seq_len, stream,
                                                num_sms);
  }
  if constexpr (D == 128) {
    // two kv heads per item (one 8 KB box per tile: half the boxes per
    // byte): 12 stages of 16 KB, or 8.  On the qwen3 batch 59.4 against
    // 61.4 us for one-head items (the cut rule counts keys, so two-head
    // items are cut no more often)
    if (decode_heads_per_item(D, a.H_kv, a.G) == 2) {
      if (decode_fits<D, 4, 12, 2>(a))
        return launch_decode_s<D, 4, 12, APPEND, 2>(a, k_cache, v_cache, max_seq_len, stream,
                                                     num_sms);
      if (decode_fits<D, 4, 8, 2>(a))
        return launch_decode_s<D, 4, 8, APPEND, 2>(a, k_cache, v_cache, max_seq_len, stream,
                                                    num_sms);
    }
  }
  if (decode_fits<D, C::NW, C::NSTAGE>(a))
    return launch_decode_s<D, C::NW, C::NSTAGE, APPEND>(a, k_cache, v_cache, max_seq_len,
                                                         stream, num_sms);
  if constexpr (D <= 128) {
    if (decode_fits<D, 4, 16>(a))
      return launch_decode_s<D, 4, 16, APPEND>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
    if (decode_fits<D, 4, 8>(a))
      return launch_decode_s<D, 4, 8, APPEND>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
  } else if constexpr (D == 256) {
    if (decode_fits<D, 2, 8>(a))
      return launch_decode_s<D, 2, 8, APPEND>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
    if (decode_fits<D, 2, 4>(a))
      return launch_decode_s<D, 2, 4, APPEND>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, int32_t max_blocks,
                          const int32_t* seq_lens, int32_t batch, int32_t H_q, int32_t H_kv,
                          int32_t D, int32_t P, int64_t num_pages, int32_t max_seq_len,
                          float scale, int32_t window, void* workspace, size_t workspace_bytes,
                          int32_t* err, cudaStream_t stream, int num_sms,
                          const DecodeCascade* cascade, const DecodeAppend* append) {
  DecodeArgs a;
  // the pools are written only by the fused append (append != null)
  a.k_new = append ? static_cast<const uint4*>(append->k_new) : nullptr;
  a.v_new = append ? static_cast<const uint4*>(append->v_new) : nullptr;
  a.k_pool = append ? static_cast<uint4*>(const_cast<void*>(k_cache)) : nullptr;
  a.v_pool = append ? static_cast<uint4*>(const_cast<void*>(v_cache)) : nullptr;
  a.prefix_lens = cascade ? cascade->prefix_lens : nullptr;
  a.group_size = cascade ? cascade->group_size : 1;
  a.pre_o = cascade ? cascade->pre_o : nullptr;
  a.pre_lse = cascade ? cascade->pre_lse : nullptr;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.max_blocks = max_blocks;
  a.batch = batch;
  a.H_q = H_q;
  a.H_kv = H_kv;
  a.G = H_q / H_kv;
  a.P = P;
  a.num_pages = num_pages;
  a.window = window;
  a.scale_log2 = scale * 1.4426950408889634f;
  decode_workspace_split(a, workspace, workspace_bytes, batch, H_kv, D, num_sms);
  a.err = err;
  // the fused append is a separate build of the kernel, so that the plain
  // decode carries none of its code
  const bool app = a.k_new != nullptr;
  switch (D) {
    case 64:
      return app ? launch_decode_t<64, true>(a, k_cache, v_cache, max_seq_len, stream, num_sms)
                 : launch_decode_t<64, false>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
    case 128:
      return app ? launch_decode_t<128, true>(a, k_cache, v_cache, max_seq_len, stream, num_sms)
                 : launch_decode_t<128, false>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
    case 256:
      return app ? launch_decode_t<256, true>(a, k_cache, v_cache, max_seq_len, stream, num_sms)
                 : launch_decode_t<256, false>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
    case 512:
      return app ? launch_decode_t<512, true>(a, k_cache, v_cache, max_seq_len, stream, num_sms)
                 : launch_decode_t<512, false>(a, k_cache, v_cache, max_seq_len, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
