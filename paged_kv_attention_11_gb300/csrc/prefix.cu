// Prefix pass of the shared-prefix (cascade) decode.
//
// GRPO rollouts decode several generations of one prompt side by side: the
// generations' block tables alias the prompt's pages (grpo_equivalence page:
// num_generations = 4 per prompt; the flex paged-KV engine's page table lets
// block tables share physical pages).  Plain decode reads those prefix pages
// once per generation.  The cascade splits each such sequence's keys into
// the shared prefix [0, prefix_len) and its own suffix [prefix_len, len):
//
//   this kernel      for each (group, kv head): the prefix tiles are read
//                    once and attended by the query rows of every member
//                    (group_size x G rows), giving a partial (o, lse) per
//                    (sequence, q head);
//   decode kernel    the suffix of each member as an ordinary segment, then
//                    the log-sum-exp merge of its partials with the prefix
//                    partial (the same merge that joins split chunks).
//
// The result is the plain decode result (softmax over all keys), only the
// order of the sums differs.  A member whose length does not exceed the
// prefix gets no prefix partial and is decoded whole.
//
// Design: one persistent CTA per SM walks the (group, kv head) items in a
// static order.  A producer warp streams the prefix's 16-key K/V tiles with
// TMA into a ring (the decode kernel's tile layout); four consumer warps take
// the tiles round-robin and run S^T = K Q^T and O^T = V^T P^T with mma.sync
// over NTQ tiles of 8 query rows, with an exp2 online softmax.  At the end of
// an item the warps' states are combined through shared memory and written
// as normalised o (fp32) and a base-2 log-sum-exp of the scaled scores.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tile16.cuh"
#include "tmap.h"

namespace pkv {

struct PrefixArgs {
  const __nv_bfloat16* q;      // [B, H_q, D]
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* seq_lens;     // [B]
  const int32_t* prefix_lens;  // [n_groups]
  int32_t max_blocks, batch, group_size, n_groups;
  int32_t H_q, H_kv, G, P;
  int64_t num_pages;
  float scale_log2;
  float* pre_o;    // [B * H_q, D]
  float* pre_lse;  // [B * H_q]
  int32_t* err;
};

constexpr int kPfxConsumers = 4;

template <int D, int NTQ, int NSTAGE>
struct PrefixPlan {
  static constexpr int R = 8 * NTQ;                    // query rows per item
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;   // K + V
  static constexpr int kCombStride = D + 4;
  static constexpr int kComb = NSTAGE * kStageBytes;
  static constexpr int kMl = kComb + kPfxConsumers * R * kCombStride * 4;
  static constexpr int kBars = kMl + kPfxConsumers * R * 2 * 4;
  static constexpr int kOk = kBars + 2 * NSTAGE * 8;
  static constexpr int kTotal = 1024 + kOk + NSTAGE * 4;
};

// item i -> group, kv head, shared prefix tiles (0: nothing to do), and the
// members whose length exceeds the prefix (bit m)
struct PfxItem {
  int j, g, n, b0, nm;
  uint32_t elig;
};

__device__ __forceinline__ PfxItem prefix_item(const PrefixArgs& a, int i, bool flag) {
  PfxItem it;
  it.j = i / a.H_kv;
  it.g = i - it.j * a.H_kv;
  it.b0 = it.j * a.group_size;
  it.nm = min(a.group_size, a.batch - it.b0);
  const int cap = a.max_blocks * a.P;
  if (flag) {
    const int raw = __ldg(a.prefix_lens + it.j);
    if (raw != 0 && shared_prefix_len(a.prefix_lens, it.j, a.P, cap) == 0)
      raise_err(a.err, PKV_DEVERR_LEN);
  }
  const int pl = shared_prefix_len(a.prefix_lens, it.j, a.P, cap);
  it.elig = 0;
  for (int m = 0; m < it.nm; ++m) {
    int len = __ldg(a.seq_lens + it.b0 + m);
    len = len < 0 ? 0 : (len > cap ? cap : len);
    if (pl > 0 && len > pl) it.elig |= 1u << m;
  }
  it.n = it.elig ? pl / kTile : 0;
  return it;
}

template <int D, int NTQ, int NSTAGE>
__global__ void __launch_bounds__((kPfxConsumers + 1) * 32, 1)
    prefix_pass_kernel(const PrefixArgs a, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
  static_assert(NSTAGE % kPfxConsumers == 0, "a stage always feeds the same warp");
  using P_ = PrefixPlan<D, NTQ, NSTAGE>;
  constexpr int KS = D / 16;
  constexpr int R = P_::R;
  constexpr int CS = P_::kCombStride;
  constexpr int kIssueLanes = NSTAGE < 16 ? NSTAGE : 16;
  static_assert(kIssueLanes < 32, "a run of free stages ends inside the warp");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* comb = reinterpret_cast<float*>(smem + P_::kComb);  // [W][R][CS]
  float* ml = reinterpret_cast<float*>(smem + P_::kMl);      // [W][R][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P_::kBars);
  uint64_t* empty = full + NSTAGE;
  int* stage_ok = reinterpret_cast<int*>(smem + P_::kOk);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const int n_items = a.n_groups * a.H_kv;

  if (warp == kPfxConsumers) {
    // ============================ producer warp ============================
    bool dead = false;
    int it = 0;  // CTA-wide tile counter
    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
      const PfxItem item = prefix_item(a, i, lane == 0);
      const int* bt = a.block_table + (int64_t)item.b0 * a.max_blocks;
      for (int k0 = 0; k0 < item.n; k0 += 32) {
        int page = -1;
        if (k0 + lane < item.n) page = __ldg(bt + ((k0 + lane) * kTile) / a.P);
        const int cnt = min(32, item.n - k0);
        // in order, each tile as soon as its stage is free (as in the decode
        // producer: a run of free stages per warp instruction)
        for (int j = 0; j < cnt;) {
          const int jj = j + lane;
          const int pg = __shfl_sync(0xffffffffu, page, jj & 31);
          const int t = it + jj;
          const int s = t % NSTAGE;
          const int r = t / NSTAGE;
          const bool mine = lane < kIssueLanes && jj < cnt;
          const bool free_ = mine && (r == 0 || mbar_test_wait(empty + s, (r - 1) & 1));
          const uint32_t fm = __ballot_sync(0xffffffffu, free_);
          int run = __ffs(~fm) - 1;
          if (run == 0) {
            if (lane == 0) mbar_wait(empty + s, (r - 1) & 1, a.err, dead);
            __syncwarp();
            run = 1;
            if (__shfl_sync(0xffffffffu, (int)dead, 0)) dead = true;
          }
          if (lane < run) {
            const bool ok = pg >= 0 && (int64_t)pg < a.num_pages;
            stage_ok[s] = ok ? 1 : 0;
            if (ok) {
              uint8_t* st = smem + s * P_::kStageBytes;
              mbar_arrive_expect_tx(full + s, P_::kStageBytes);
              const int row = ((k0 + jj) * kTile) % a.P;
              const int z = pg * a.H_kv + item.g;
              tma_load_5d(st, &tmK, full + s, 0, 0, 0, row / 8, z);
              tma_load_5d(st + P_::kTileBytes, &tmV, full + s, 0, 0, 0, row / 8, z);
            } else {
              raise_err(a.err, PKV_DEVERR_PAGE);
              mbar_arrive(full + s);
            }
          }
          __syncwarp();
          j += run;
        }
        it += cnt;
      }
    }
    // every issued load lands before the CTA exits
    if (lane == 0) {
      for (int t = (it > NSTAGE ? it - NSTAGE : 0); t < it; ++t)
        mbar_wait(full + (t % NSTAGE), (t / NSTAGE) & 1, a.err, dead);
    }
  } else {
    // ============================ consumer warps ===========================
    const int quad = lane >> 2;  // key row (QK) / query row within an n tile
    const int qlan = lane & 3;
    bool dead = false;
    int it_base = 0;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
      const PfxItem item = prefix_item(a, i, false);
      if (item.n == 0) continue;
      // Q^T fragments of n tile t: query row t*8 + quad = member m, head h
      uint32_t qb[KS][NTQ][2];
#pragma unroll
      for (int t = 0; t < NTQ; ++t) {
        const int rr = t * 8 + quad;
        const int m = rr / a.G, h = rr - (rr / a.G) * a.G;
        const bool hv = m < item.nm && ((item.elig >> m) & 1u);
        const __nv_bfloat16* qrow =
            a.q + ((int64_t)(item.b0 + (hv ? m : 0)) * a.H_q + item.g * a.G + h) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qb[ks][t][0] = hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * qlan))
                            : 0u;
          qb[ks][t][1] =
              hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * qlan)) : 0u;
        }
      }
      float o[KS][NTQ][4];
#pragma unroll
      for (int md = 0; md < KS; ++md)
#pragma unroll
        for (int t = 0; t < NTQ; ++t) o[md][t][0] = o[md][t][1] = o[md][t][2] = o[md][t][3] = 0.f;
      float mA[NTQ], mB[NTQ], lA[NTQ], lB[NTQ];
#pragma unroll
      for (int t = 0; t < NTQ; ++t) {
        mA[t] = mB[t] = -INFINITY;
        lA[t] = lB[t] = 0.f;
      }
      const int n = item.n;
      const int r0 = ((warp - it_base) % kPfxConsumers + kPfxConsumers) % kPfxConsumers;
      for (int kk = r0; kk < n; kk += kPfxConsumers) {
        const int tt = it_base + kk;
        const int s = tt % NSTAGE;
        const bool landed = mbar_wait(full + s, (tt / NSTAGE) & 1, a.err, dead);
        const bool ok = landed && stage_ok[s] != 0;
        const uint32_t stK = smem_u32(smem + s * P_::kStageBytes);
        const uint32_t stV = stK + P_::kTileBytes;
        // ---- S^T = K Q^T: 16 keys x 8 rows per n tile ----
        float sc[NTQ][4];
#pragma unroll
        for (int t = 0; t < NTQ; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
        {
          const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(tile_addr<D>(stK, key, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < NTQ; ++t)
              mma_bf16_16816(sc[t], a0, a1, a2, a3, qb[ks][t][0], qb[ks][t][1]);
          }
        }
        // every key of a prefix tile is attended by every eligible row
        uint32_t pb[NTQ][2];
#pragma unroll
        for (int t = 0; t < NTQ; ++t) {
          const float x0A = ok ? sc[t][0] * a.scale_log2 : -INFINITY;
          const float x0B = ok ? sc[t][1] * a.scale_log2 : -INFINITY;
          const float x1A = ok ? sc[t][2] * a.scale_log2 : -INFINITY;
          const float x1B = ok ? sc[t][3] * a.scale_log2 : -INFINITY;
          float tA = fmaxf(x0A, x1A), tB = fmaxf(x0B, x1B);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, off));
            tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, off));
          }
          const float nA = fmaxf(mA[t], tA), nB = fmaxf(mB[t], tB);
          const float uA = nA == -INFINITY ? 0.f : nA;
          const float uB = nB == -INFINITY ? 0.f : nB;
          const float alA = exp2f(mA[t] - uA), alB = exp2f(mB[t] - uB);
          const float p0A = exp2f(x0A - uA), p0B = exp2f(x0B - uB);
          const float p1A = exp2f(x1A - uA), p1B = exp2f(x1B - uB);
          lA[t] = lA[t] * alA + p0A + p1A;
          lB[t] = lB[t] * alB + p0B + p1B;
          mA[t] = nA;
          mB[t] = nB;
#pragma unroll
          for (int md = 0; md < KS; ++md) {
            o[md][t][0] *= alA;
            o[md][t][1] *= alB;
            o[md][t][2] *= alA;
            o[md][t][3] *= alB;
          }
          pb[t][0] = movmatrix_t(pack_bf16(p0A, p0B));
          pb[t][1] = movmatrix_t(pack_bf16(p1A, p1B));
        }
        // ---- O^T += V^T P^T ----
        {
          const int jq = lane >> 3;
          const int key = (lane & 7) + (jq >> 1) * 8;
#pragma unroll
          for (int md = 0; md < KS; ++md) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(tile_addr<D>(stV, key, 2 * md + (jq & 1)), a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < NTQ; ++t)
              mma_bf16_16816(o[md][t], a0, a1, a2, a3, pb[t][0], pb[t][1]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);
      }
      it_base += n;

      // ---- combine the four warps' states through shared memory ----
      float* co = comb + (warp * R) * CS;
      float* cm = ml + (warp * R) * 2;
#pragma unroll
      for (int t = 0; t < NTQ; ++t) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          lA[t] += __shfl_xor_sync(0xffffffffu, lA[t], off);
          lB[t] += __shfl_xor_sync(0xffffffffu, lB[t], off);
        }
        const int hA = t * 8 + 2 * qlan, hB = hA + 1;
#pragma unroll
        for (int md = 0; md < KS; ++md) {
          const int d = md * 16 + quad;
          co[hA * CS + d] = o[md][t][0];
          co[hA * CS + d + 8] = o[md][t][2];
          co[hB * CS + d] = o[md][t][1];
          co[hB * CS + d + 8] = o[md][t][3];
        }
        if (quad == 0) {
          cm[hA * 2] = mA[t];
          cm[hA * 2 + 1] = lA[t];
          cm[hB * 2] = mB[t];
          cm[hB * 2 + 1] = lB[t];
        }
      }
      named_bar_sync(1, kPfxConsumers * 32);
      for (int idx = tid; idx < R * (D / 4); idx += kPfxConsumers * 32) {
        const int rr = idx / (D / 4), d4 = idx - rr * (D / 4);
        const int m = rr / a.G, h = rr - (rr / a.G) * a.G;
        if (m >= item.nm || !((item.elig >> m) & 1u)) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kPfxConsumers; ++w) M = fmaxf(M, ml[(w * R + rr) * 2]);
        float lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kPfxConsumers; ++w) {
          const float mw = ml[(w * R + rr) * 2];
          const float sc = M == -INFINITY ? 0.f : exp2f(mw - M);
          lsum += sc * ml[(w * R + rr) * 2 + 1];
          const float4 v = *reinterpret_cast<const float4*>(comb + (w * R + rr) * CS + d4 * 4);
          acc.x += sc * v.x;
          acc.y += sc * v.y;
          acc.z += sc * v.z;
          acc.w += sc * v.w;
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
        const int64_t row = (int64_t)(item.b0 + m) * a.H_q + item.g * a.G + h;
        *reinterpret_cast<float4*>(a.pre_o + row * D + d4 * 4) = acc;
        if (d4 == 0) a.pre_lse[row] = lsum > 0.f ? M + log2f(lsum) : -INFINITY;
      }
      named_bar_sync(1, kPfxConsumers * 32);  // comb is free for the next item
    }
  }
}

// --------------------------------------------------------------- host side
template <int D>
struct PrefixCfg;
template <> struct PrefixCfg<64> { static constexpr int NSTAGE = 16, MAX_NTQ = 4; };
template <> struct PrefixCfg<128> { static constexpr int NSTAGE = 16, MAX_NTQ = 2; };
template <> struct PrefixCfg<256> { static constexpr int NSTAGE = 8, MAX_NTQ = 1; };

int prefix_max_rows(int D) {
  switch (D) {
    case 64: return 8 * PrefixCfg<64>::MAX_NTQ;
    case 128: return 8 * PrefixCfg<128>::MAX_NTQ;
    case 256: return 8 * PrefixCfg<256>::MAX_NTQ;
    default: return 0;
  }
}

template <int D, int NTQ>
static cudaError_t launch_prefix_t(const PrefixArgs& a, const void* k_cache, const void* v_cache,
                                   cudaStream_t stream, int num_sms) {
  constexpr int NSTAGE = PrefixCfg<D>::NSTAGE;
  using P_ = PrefixPlan<D, NTQ, NSTAGE>;
  auto kern = prefix_pass_kernel<D, NTQ, NSTAGE>;
  CUtensorMap tmK, tmV;
  const bool enc_ok =
      encode_pool_map_groups(&tmK, k_cache, D, a.P, a.num_pages, a.H_kv, kTile) &&
      encode_pool_map_groups(&tmV, v_cache, D, a.P, a.num_pages, a.H_kv, kTile);
  if (!enc_ok) return cudaErrorInvalidValue;
  static_assert(P_::kTotal <= 227 * 1024, "prefix pass shared memory");
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_::kTotal);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int n_items = a.n_groups * a.H_kv;
  const int grid = n_items < num_sms ? n_items : num_sms;
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((kPfxConsumers + 1) * 32);
  cfg.dynamicSmemBytes = P_::kTotal;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, tmK, tmV);
}

template <int D>
static cudaError_t launch_prefix_d(const PrefixArgs& a, const void* k_cache, const void* v_cache,
                                   cudaStream_t stream, int num_sms) {
  const int rows = a.group_size * a.G;
  if (rows <= 8) return launch_prefix_t<D, 1>(a, k_cache, v_cache, stream, num_sms);
  if (PrefixCfg<D>::MAX_NTQ >= 2 && rows <= 16)
    return launch_prefix_t<D, (PrefixCfg<D>::MAX_NTQ >= 2 ? 2 : 1)>(a, k_cache, v_cache, stream,
                                                                     num_sms);
  if (PrefixCfg<D>::MAX_NTQ >= 4 && rows <= 32)
    return launch_prefix_t<D, (PrefixCfg<D>::MAX_NTQ >= 4 ? 4 : 1)>(a, k_cache, v_cache, stream,
                                                                     num_sms);
  return cudaErrorNotSupported;
}

cudaError_t launch_prefix_pass(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* seq_lens, const int32_t* prefix_lens,
                               int32_t batch, int32_t group_size, int32_t H_q, int32_t H_kv,
                               int32_t D, int32_t P, int64_t num_pages, float scale,
                               float* pre_o, float* pre_lse, int32_t* err, cudaStream_t stream,
                               int num_sms) {
  PrefixArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.prefix_lens = prefix_lens;
  a.max_blocks = max_blocks;
  a.batch = batch;
  a.group_size = group_size;
  a.n_groups = (batch + group_size - 1) / group_size;
  a.H_q = H_q;
  a.H_kv = H_kv;
  a.G = H_q / H_kv;
  a.P = P;
  a.num_pages = num_pages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.pre_o = pre_o;
  a.pre_lse = pre_lse;
  a.err = err;
  switch (D) {
    case 64: return launch_prefix_d<64>(a, k_cache, v_cache, stream, num_sms);
    case 128: return launch_prefix_d<128>(a, k_cache, v_cache, stream, num_sms);
    case 256: return launch_prefix_d<256>(a, k_cache, v_cache, stream, num_sms);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pkv
