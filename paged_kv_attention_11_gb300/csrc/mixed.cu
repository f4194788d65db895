// paged_attn_mixed: the attention of one continuous-batching step -- decode
// rows and prefill chunks -- in a single persistent launch.
//
// Source: scripts/benchmarks commit log, batch-sweep commit (vLLM runs
// chunked prefill and decode of one step packed into the same kernels) and
// README "Why continuous batching is still slower than vLLM on this
// workload" (separate prefill and decode passes per step).
//
// Decode is bound by HBM bandwidth, prefill by the tensor cores and its own
// latency chain; run back to back, each leaves the other's resource idle.
// Here one grid of one CTA per SM splits the step:
//   * CTAs [0, nd) start with decode (the split-KV body, decode_cta, on
//     warps 0-5; the dynamic longest-first queue in the workspace; items of
//     two kv heads where the shape allows, whose 8 KB boxes raise the
//     per-SM streaming rate that bounds a decode on part of the SMs.  8
//     consumer warps on warps 0-9 measured no faster);
//   * CTAs [nd, N) run the prefill chunks (the tcgen05 body, varlen_cta,
//     with the static snake schedule over those N - nd CTAs), then join the
//     decode queue and take whatever work is left in it.
// Every CTA ends in the decode body, so the decode queue's last-CTA reset
// and the zero rows of empty sequences work as in paged_attn_decode.  No
// warp moves registers (setmaxnreg): both bodies run in the launch's 168 per
// thread.
//
// paged_attn_mixed_append also writes the step's new K/V rows first: every
// CTA appends a slice of them (a warp per token, as paged_kv_append), then
// all CTAs meet at a grid barrier (every CTA is resident: one per SM; the
// wait is bounded) before any work reads the pools.
#include "decode_body.cuh"
#include "tmap.h"
#include "varlen_body.cuh"

namespace pkv {

struct MixedArgs {
  DecodeArgs dec;
  VarlenArgs var;
  // the fused append (num_new > 0): rows of num_new tokens, vpt 16-byte
  // vectors each, to the pools at slot_mapping; bar: two grid-barrier
  // counters in the workspace (zero between calls)
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_pool;
  uint4* v_pool;
  const int64_t* slot_mapping;
  int64_t num_slots;
  int32_t num_new, vpt, vpr;
  int32_t* bar;
  int32_t has_dec, has_var;
  int32_t var_first;  // first CTA that starts with the prefill
};

// the prefill shape of the mixed step (head_dim 128): two Q tiles per item,
// 128-key tiles, K ring 3, V ring 2
constexpr int kMixD = 128, kMixNQ = 2, kMixBN = 128, kMixNS = 1, kMixNKS = 3, kMixNVS = 2;
constexpr int kMixThreads = varlen_threads<kMixNQ>();  // 384
static_assert(kMixThreads == 384, "three warpgroups");
#ifndef PKV_MIX_DEC_NW
#define PKV_MIX_DEC_NW 4
#endif
constexpr int kMixDecNW = PKV_MIX_DEC_NW;  // decode consumer warps (+ producer + epilogue)
static_assert((kMixDecNW + 2) * 32 <= kMixThreads, "decode warps fit the block");

// The step's new rows: a warp takes kMixTokPerPass tokens at once (4
// vectors of K and of V per lane per token), so that a prefill-sized step's
// reads are all in flight together on the launch's 12 warps per SM; then
// the grid barrier.
constexpr int kMixTokPerPass = 4;
__device__ __forceinline__ void mixed_append_rows(const MixedArgs& m) {
  pdl_wait();  // the rows may come from the previous kernel
  constexpr int TP = kMixTokPerPass;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int nw = gridDim.x * wpb;
  const int P = m.dec.P, H_kv = m.dec.H_kv;
  const int hstride = P * m.vpr;
  // warp w takes tokens w + (k * TP + i) * nw, i < TP, in pass k
  for (int tok0 = blockIdx.x * wpb + (threadIdx.x >> 5); tok0 < m.num_new; tok0 += nw * TP) {
    int64_t slot[TP];
#pragma unroll
    for (int i = 0; i < TP; ++i) {
      const int tok = tok0 + i * nw;
      slot[i] = tok < m.num_new ? __ldg(m.slot_mapping + tok) : -1;
    }
    for (int v0 = 0; v0 < m.vpt; v0 += 128) {
      uint4 kv[TP][4], vv[TP][4];
#pragma unroll
      for (int i = 0; i < TP; ++i) {
        const int tok = tok0 + i * nw;
        const int64_t src0 = (int64_t)tok * m.vpt;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int v = v0 + lane + 32 * j;
          if (tok < m.num_new && v < m.vpt) {
            kv[i][j] = __ldg(m.k_new + src0 + v);
            vv[i][j] = __ldg(m.v_new + src0 + v);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < TP; ++i) {
        if (slot[i] < 0) continue;  // padding row, or no token
        if (slot[i] >= m.num_slots) {
          if (lane == 0 && v0 == 0) raise_err(m.dec.err, PKV_DEVERR_SLOT);
          continue;
        }
        const int64_t page = slot[i] / P;
        const int row = (int)(slot[i] - page * P);
        uint4* kd = m.k_pool + (page * H_kv * P + row) * m.vpr;
        uint4* vd = m.v_pool + (kd - m.k_pool);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int v = v0 + lane + 32 * j;
          if (v < m.vpt) {
            const int h = v / m.vpr;
            const int off = h * hstride + (v - h * m.vpr);
            kd[off] = kv[i][j];
            vd[off] = vv[i][j];
          }
        }
      }
    }
  }
  // the rows are read by TMA (the async proxy) in every CTA
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    atomicAdd(m.bar, 1);
    const unsigned long long t0 = globaltimer();
    while (ld_volatile_i32(m.bar) < (int)gridDim.x) {
      __nanosleep(32);
      if (globaltimer() - t0 > kWaitTimeoutNs) {
        raise_err(m.dec.err, PKV_DEVERR_TIMEOUT);
        break;
      }
    }
    __threadfence();
    // the last CTA past the wait resets both counters for the next call
    if (atomicAdd(m.bar + 1, 1) == (int)gridDim.x - 1) {
      m.bar[0] = 0;
      m.bar[1] = 0;
    }
  }
  __syncthreads();
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// APPEND: paged_attn_mixed_append's build (the plain launch carries none of
// the append's code)
template <int NSTAGE_DEC, int HP, bool APPEND>
__global__ void __launch_bounds__(kMixThreads, 1)
    mixed_step_kernel(const MixedArgs m, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmKv,
                      const __grid_constant__ CUtensorMap tmVv,
                      const __grid_constant__ CUtensorMap tmKd,
                      const __grid_constant__ CUtensorMap tmVd) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int nd = m.var_first;
  if (APPEND) mixed_append_rows(m);
  if (m.has_var && (int)blockIdx.x >= nd)
    varlen_cta<kMixD, kMixNQ, kMixBN, kMixNS, kMixNKS, kMixNVS, true>(
        m.var, tmQ, tmKv, tmVv, smem, (int)blockIdx.x - nd, (int)gridDim.x - nd);
  if (m.has_dec && warp < kMixDecNW + 2)
    decode_cta<kMixD, kMixDecNW, NSTAGE_DEC, true, false, HP>(m.dec, tmKd, tmVd, smem,
                                                              blockIdx.x);
}

// CTAs that start with decode when the caller leaves the split open: the
// smallest count whose decode time (HBM bound, or the per-SM rate below
// that) does not exceed the prefill time of the remaining CTAs, from the
// host's estimates of the work (half of the longest decode context per row,
// prefill pairs from the packed lengths).  Prefill CTAs join the decode
// queue when they are done, so the estimate may err towards fewer.
static int mixed_decode_ctas(int num_sms, int64_t dec_batch, int64_t dec_max_seq_len,
                             int64_t total_q, int64_t max_seqlen_q, int64_t max_seqlen_k,
                             int H_q, int H_kv, int D) {
  const double dec_bytes = (double)dec_batch * (double)(dec_max_seq_len / 2 + 1) * H_kv * D * 4.0;
  double pairs_per_q = (double)max_seqlen_k - 0.5 * (double)max_seqlen_q;
  if (pairs_per_q < 1.0) pairs_per_q = 1.0;
  const double var_flops = (double)total_q * pairs_per_q * 4.0 * D * H_q;
  // per-SM decode rate measured with 72 decode CTAs: ~73 GB/s with items of
  // two kv heads, ~60 GB/s with one
  const double per_sm_bw = decode_heads_per_item(D, H_kv, H_q / H_kv) == 2 ? 73e9 : 55e9;
  const double hbm = 6.5e12, per_sm_flops = 4.4e12;
  for (int nd = 1; nd < num_sms; ++nd) {
    double bw = nd * per_sm_bw;
    if (bw > hbm) bw = hbm;
    const double t_dec = dec_bytes / bw;
    const double t_var = var_flops / ((num_sms - nd) * per_sm_flops);
    if (t_dec <= t_var) return nd;
  }
  return num_sms - 1;
}

template <int NSTAGE_DEC, int HP, bool APPEND>
static cudaError_t launch_mixed_k(MixedArgs& m, const VarlenMaps& vmaps, const void* k_cache,
                                  const void* v_cache, size_t smem, cudaStream_t stream,
                                  int num_sms) {
  auto kern = mixed_step_kernel<NSTAGE_DEC, HP, APPEND>;
  CUtensorMap tmKd, tmVd;
  if (!encode_pool_map_groups(&tmKd, k_cache, kMixD, m.dec.P, m.dec.num_pages, m.dec.H_kv, kTile,
                              0, HP) ||
      !encode_pool_map_groups(&tmVd, v_cache, kMixD, m.dec.P, m.dec.num_pages, m.dec.H_kv, kTile,
                              0, HP))
    return cudaErrorInvalidValue;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < (int)smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = (int)smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms);
  cfg.blockDim = dim3(kMixThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, m, vmaps.q, vmaps.k, vmaps.v, tmKd, tmVd);
}

template <int NSTAGE_DEC, int HP>
static cudaError_t launch_mixed_t(MixedArgs& m, const VarlenMaps& vmaps, const void* k_cache,
                                  const void* v_cache, size_t smem, cudaStream_t stream,
                                  int num_sms) {
  if (m.num_new > 0)
    return launch_mixed_k<NSTAGE_DEC, HP, true>(m, vmaps, k_cache, v_cache, smem, stream,
                                                num_sms);
  return launch_mixed_k<NSTAGE_DEC, HP, false>(m, vmaps, k_cache, v_cache, smem, stream,
                                               num_sms);
}

cudaError_t launch_mixed(const MixedLaunch& L, const VarlenMaps& vmaps, cudaStream_t stream,
                         int num_sms) {
  if (L.D != kMixD) return cudaErrorNotSupported;
  MixedArgs m;
  m.has_dec = L.dec_batch > 0;
  m.has_var = L.pre_batch > 0 && L.total_q > 0 && L.max_seqlen_q > 0;
  // ---- decode arguments (as launch_decode)
  DecodeArgs& a = m.dec;
  a.q = static_cast<const __nv_bfloat16*>(L.dec_q);
  a.out = static_cast<__nv_bfloat16*>(L.dec_out);
  a.block_table = L.dec_block_table;
  a.seq_lens = L.dec_seq_lens;
  a.max_blocks = L.dec_max_blocks;
  a.batch = L.dec_batch;
  a.H_q = L.H_q;
  a.H_kv = L.H_kv;
  a.G = L.H_q / L.H_kv;
  a.P = L.P;
  a.num_pages = L.num_pages;
  a.window = L.window;
  a.scale_log2 = L.scale * 1.4426950408889634f;
  a.prefix_lens = nullptr;
  a.k_new = a.v_new = nullptr;
  a.k_pool = a.v_pool = nullptr;
  a.group_size = 1;
  a.pre_o = nullptr;
  a.pre_lse = nullptr;
  a.err = L.err;
  decode_workspace_split(a, L.workspace, L.workspace_bytes, L.dec_batch, L.H_kv, L.D, num_sms);
  // ---- the fused append (paged_attn_mixed_append)
  m.num_new = L.num_new > 0 ? L.num_new : 0;
  m.k_new = static_cast<const uint4*>(L.k_new);
  m.v_new = static_cast<const uint4*>(L.v_new);
  m.k_pool = static_cast<uint4*>(const_cast<void*>(L.k_cache));
  m.v_pool = static_cast<uint4*>(const_cast<void*>(L.v_cache));
  m.slot_mapping = L.slot_mapping;
  m.num_slots = L.num_pages * L.P;
  m.vpr = L.D / 8;
  m.vpt = L.H_kv * m.vpr;
  m.bar = a.queue + 5;  // queue[5..6]: free slots of the decode workspace's counters
  // ---- prefill arguments (as launch_varlen)
  VarlenArgs& v = m.var;
  const int QP = 128 / a.G;
  v.out = static_cast<__nv_bfloat16*>(L.pre_out);
  v.cu_q = L.cu_q;
  v.cu_k = L.cu_k;
  v.block_table = L.pre_block_table;
  v.batch = L.pre_batch;
  v.max_blocks = L.pre_max_blocks;
  v.max_q = L.max_seqlen_q;
  v.R = (L.max_seqlen_q + 2 * QP - 1) / (2 * QP);
  v.pairs_max = L.pre_batch * v.R;
  v.H_q = L.H_q;
  v.H_kv = L.H_kv;
  v.G = a.G;
  v.log2G = 0;
  while ((1 << v.log2G) < v.G) ++v.log2G;
  v.P = L.P;
  v.box_rows = L.P < kMixBN ? L.P : kMixBN;
  v.num_pages = L.num_pages;
  v.scale_log2 = a.scale_log2;
  v.causal = 1;
  v.window = L.window;
  v.out_v8 = (reinterpret_cast<uintptr_t>(L.pre_out) & 31) == 0 ? 1 : 0;
  v.err = L.err;
  // ---- the split
  int nd = L.decode_ctas;
  if (nd <= 0)
    nd = mixed_decode_ctas(num_sms, L.dec_batch, L.dec_max_seq_len, L.total_q, L.max_seqlen_q,
                           L.max_seqlen_k, L.H_q, L.H_kv, L.D);
  if (m.has_var && m.has_dec) nd = nd < 1 ? 1 : (nd > num_sms - 1 ? num_sms - 1 : nd);
  if (!m.has_var) nd = num_sms;  // decode only: every CTA starts with decode
  if (!m.has_dec) nd = 0;        // prefill only: every CTA runs the prefill
  m.var_first = nd;
  a.cta_count = num_sms;
  a.share_ctas = nd > 0 ? nd : num_sms;
  // ---- shared memory: the larger of the two plans
  using VS = VarlenSmem<kMixD, kMixNQ, kMixBN, kMixNS, kMixNKS, kMixNVS>;
  const size_t var_smem = m.has_var ? VS::bytes(v.batch, v.pairs_max) : 0;
  constexpr size_t kMax = 227 * 1024;
  if (var_smem > kMax) return cudaErrorNotSupported;
  if (decode_heads_per_item(L.D, L.H_kv, a.G) == 2) {
    // two kv heads per decode item: 12 stages of 16 KB, or 8
    const size_t dec12 = DecodePlan<kMixD, kMixDecNW, 12, 2>(a.G, a.batch).total;
    const size_t dec8 = DecodePlan<kMixD, kMixDecNW, 8, 2>(a.G, a.batch).total;
    if (!m.has_dec || dec12 <= kMax) {
      const size_t smem = var_smem > dec12 ? var_smem : dec12;
      return launch_mixed_t<12, 2>(m, vmaps, L.k_cache, L.v_cache, smem, stream, num_sms);
    }
    if (dec8 > kMax) return cudaErrorNotSupported;
    const size_t smem = var_smem > dec8 ? var_smem : dec8;
    return launch_mixed_t<8, 2>(m, vmaps, L.k_cache, L.v_cache, smem, stream, num_sms);
  }
  const size_t dec24 = DecodePlan<kMixD, kMixDecNW, 24>(a.G, a.batch).total;
  const size_t dec16 = DecodePlan<kMixD, kMixDecNW, 16>(a.G, a.batch).total;
  if (!m.has_dec || dec24 <= kMax) {
    const size_t smem = var_smem > dec24 ? var_smem : dec24;
    return launch_mixed_t<24, 1>(m, vmaps, L.k_cache, L.v_cache, smem, stream, num_sms);
  }
  if (dec16 > kMax) return cudaErrorNotSupported;
  const size_t smem = var_smem > dec16 ? var_smem : dec16;
  return launch_mixed_t<16, 1>(m, vmaps, L.k_cache, L.v_cache, smem, stream, num_sms);
}

}  // namespace pkv
