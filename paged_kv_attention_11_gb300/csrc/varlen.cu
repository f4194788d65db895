// paged_attn_varlen: packed variable-length (prefill) attention over the
// paged cache on the tcgen05 tensor cores.
//
// Semantics: cb_sync_driver.py commit message (phase-2 fixes: a paged varlen
// forward is described by cu_seq_lens_q / cu_seq_lens_k), README
// "Integration notes" (max_seqlen_q / max_seqlen_k), scripts/benchmarks
// commit log: the packed-prefill "document causal" mask (queries see keys of
// their own sequence up to their position) and the Gemma-4 sliding window
// (q_pos - k_pos < window, strict).  Chunks sit on top of a cached prefix:
// query i of a chunk with q_len queries and k_len keys is at position
// k_len - q_len + i.
//
// Design (GB300):
//  * One CTA per (128-row Q tile, kv head, chunk).  The 128 MMA rows pack
//    128/G query positions x the G query heads that share the kv head, so a
//    K/V tile staged once in shared memory feeds the whole GQA group.
//  * Warp 0: TMA producer (Q once; K and V tiles through two 2-deep rings;
//    page lookups in the block table, one box per page slice, 128-byte
//    swizzle).  Boxes outside the attended key range or the pool are
//    fetched at an out-of-range coordinate, which fills zeros.
//  * Warp 1: allocates 512 TMEM columns and issues tcgen05.mma
//    (cta_group::1, kind::f16, bf16 in, fp32 accumulate):
//        S[buf] = Q K^T   (M=128, N=BN, K=D; two S buffers in TMEM)
//        O     += P V     (M=128, N=D,  K=BN; P from smem, V MN-major)
//    S for tile j+1 is issued before PV of tile j, so the tensor core works
//    on the next QK^T while the softmax warps handle the current tile.
//  * Warps 2-5 (one thread per row): tcgen05.ld the S row, mask, online
//    softmax in the exp2 domain, write P (bf16, swizzled) to smem, rescale
//    O in TMEM only when the running max grew by more than 2^8 (the stale
//    max is exact math because O and l share it), epilogue O / l -> bf16.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {

struct VarlenArgs {
  __nv_bfloat16* out;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_table;
  int32_t max_blocks;
  int32_t num_qtiles;
  int32_t H_q, H_kv, G, log2G, P, box_rows;
  int64_t num_pages;
  float scale_log2;
  int32_t causal, window;
  int32_t* err;
};

template <int D, int BN>
struct VarlenSmem {
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kKVChunk = BN * 128;          // one 64-column chunk of a tile
  static constexpr int kKVBytes = (D / 64) * kKVChunk;
  static constexpr int kPBytes = 128 * BN * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + 2 * kKVBytes;
  static constexpr int kPOff = kVOff + 2 * kKVBytes;
  static constexpr int kBarOff = kPOff + kPBytes;
  static constexpr int kNumBars = 15;
  static constexpr int kTmemOff = kBarOff + kNumBars * 8;
  static constexpr int kEnd = kTmemOff + 16;
  // at least 116 KB so that only one CTA (and its 512 TMEM columns) fits
  // on an SM
  static constexpr int kBytes = 1024 + (kEnd > 116 * 1024 ? kEnd : 116 * 1024);
};

template <int D, int BN>
__global__ void __launch_bounds__(192, 1)
    varlen_fwd_kernel(const VarlenArgs a, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using S_ = VarlenSmem<D, BN>;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, BN, false);
  constexpr uint32_t kIdescO = tc::idesc_bf16_f32(128, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S_::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2]
  uint64_t* s_free = bars + 11;  // [2]
  uint64_t* p_full = bars + 13;
  uint64_t* o_done = bars + 14;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S_::kTmemOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int g = blockIdx.y;
  const int qt = a.num_qtiles - 1 - (int)blockIdx.x;  // long (late) tiles first
  const int QP = 128 >> a.log2G;                       // query positions per tile

  pdl_wait();  // inputs may come from the previous kernel in the stream
  pdl_launch_dependents();
  const int q0 = __ldg(a.cu_q + b);
  int q_len = __ldg(a.cu_q + b + 1) - q0;
  int k_len = __ldg(a.cu_k + b + 1) - __ldg(a.cu_k + b);
  const bool leader = threadIdx.x == 0 && g == 0;
  if (q_len < 0) {
    if (leader && qt == 0) raise_err(a.err, PKV_DEVERR_LEN);
    return;
  }
  if (q_len > a.num_qtiles * QP) {
    if (leader && qt == 0) raise_err(a.err, PKV_DEVERR_LEN);
    q_len = a.num_qtiles * QP;
  }
  const int kcap = a.max_blocks * a.P;
  if (k_len < 0 || k_len > kcap) {
    if (leader && qt == 0) raise_err(a.err, PKV_DEVERR_LEN);
    k_len = k_len < 0 ? 0 : kcap;
  }
  const int p_begin = qt * QP;
  if (p_begin >= q_len) return;
  const int p_end = min(p_begin + QP, q_len);
  const int off = k_len - q_len;  // position of chunk row 0

  int kv_lo = 0, kv_hi = k_len;
  if (a.causal) {
    kv_hi = min(k_len, off + p_end);
    if (a.window > 0) kv_lo = max(0, off + p_begin - a.window + 1);
  }
  const int t_lo = kv_lo / BN;
  const int n = kv_hi > kv_lo ? (kv_hi + BN - 1) / BN - t_lo : 0;

  if (n == 0) {  // every row of this tile sees no key: zero output rows
    if (warp >= 2) {
      const int r = (warp & 3) * 32 + lane;
      const int p = p_begin + (r >> a.log2G);
      if (p < p_end) {
        uint4* dst = reinterpret_cast<uint4*>(
            a.out + ((int64_t)(q0 + p) * a.H_q + g * a.G + (r & (a.G - 1))) * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- setup
  if (warp == 0 && lane == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
      mbar_init(s_full + i, 1);
      mbar_init(s_free + i, 128);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  const uint32_t sQ = smem_u32(smem + S_::kQOff);
  const uint32_t sK = smem_u32(smem + S_::kKOff);
  const uint32_t sV = smem_u32(smem + S_::kVOff);
  const uint32_t sP = smem_u32(smem + S_::kPOff);

  if (warp == 0) {
    // ============================== TMA producer ============================
    bool dead = false;
    const int* bt = a.block_table + (int64_t)b * a.max_blocks;
    const int R = a.box_rows;
    const int nsub = BN / R;
    const int oob = (int)(a.num_pages * a.H_kv);  // first z past the pool: zero fill
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, S_::kQBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(smem + S_::kQOff + c * 16384, &tmQ, q_full, c * 64, 0, g, q0 + p_begin);
    }
    for (int j = 0; j < n; ++j) {
      const int key_base = (t_lo + j) * BN;
      int z = oob, row = 0;
      if (lane < nsub) {
        const int key0 = key_base + lane * R;
        row = key0 % a.P;
        if (key0 < kv_hi && key0 + R > kv_lo) {
          const int pg = __ldg(bt + key0 / a.P);
          if (pg >= 0 && (int64_t)pg < a.num_pages) z = pg * a.H_kv + g;
          else raise_err(a.err, PKV_DEVERR_PAGE);
        }
      }
      int zs[8], rows[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        zs[i] = __shfl_sync(0xffffffffu, z, i);
        rows[i] = __shfl_sync(0xffffffffu, row, i);
      }
      if (lane == 0) {
        const int s = j & 1;
        if (j >= 2) mbar_wait(k_empty + s, ((j >> 1) - 1) & 1, a.err, dead);
        mbar_arrive_expect_tx(k_full + s, S_::kKVBytes);
        uint8_t* kdst = smem + S_::kKOff + s * S_::kKVBytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < nsub) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(kdst + c * S_::kKVChunk + i * R * 128, &tmK, k_full + s, c * 64,
                          rows[i], zs[i]);
          }
        }
        if (j >= 2) mbar_wait(v_empty + s, ((j >> 1) - 1) & 1, a.err, dead);
        mbar_arrive_expect_tx(v_full + s, S_::kKVBytes);
        uint8_t* vdst = smem + S_::kVOff + s * S_::kKVBytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < nsub) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(vdst + c * S_::kKVChunk + i * R * 128, &tmV, v_full + s, c * 64,
                          rows[i], zs[i]);
          }
        }
      }
      __syncwarp();
    }
    if (lane == 0) {  // every issued copy must land before the CTA exits
      for (int j = (n > 2 ? n - 2 : 0); j < n; ++j) {
        mbar_wait(k_full + (j & 1), (j >> 1) & 1, a.err, dead);
        mbar_wait(v_full + (j & 1), (j >> 1) & 1, a.err, dead);
      }
    }
  } else if (warp == 1) {
    // =============================== MMA issuer =============================
    if (lane == 0) {
      bool dead = false;
      mbar_wait(q_full, 0, a.err, dead);
      auto pv = [&](int i) {
        const int vb = i & 1;
        mbar_wait(v_full + vb, (i >> 1) & 1, a.err, dead);
        mbar_wait(p_full, i & 1, a.err, dead);
        tc::fence_after_sync();
        const uint32_t vbase = sV + vb * S_::kKVBytes;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t ad = tc::smem_desc_sw128(sP + (ks >> 2) * 16384 + (ks & 3) * 32, 16,
                                                  1024);
          const uint64_t bd = tc::smem_desc_sw128(vbase + ks * 2048, S_::kKVChunk, 1024);
          tc::mma_ss(tmem + 2 * BN, ad, bd, kIdescO, (i > 0 || ks > 0) ? 1u : 0u);
        }
        tc::commit(o_done);
        tc::commit(v_empty + vb);
      };
      for (int j = 0; j < n; ++j) {
        const int sb = j & 1;
        mbar_wait(k_full + sb, (j >> 1) & 1, a.err, dead);
        if (j >= 2) mbar_wait(s_free + sb, ((j >> 1) - 1) & 1, a.err, dead);
        tc::fence_after_sync();
        const uint32_t kbase = sK + sb * S_::kKVBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ad = tc::smem_desc_sw128(sQ + (ks >> 2) * 16384 + (ks & 3) * 32, 16,
                                                  1024);
          const uint64_t bd = tc::smem_desc_sw128(kbase + (ks >> 2) * S_::kKVChunk + (ks & 3) * 32,
                                                  16, 1024);
          tc::mma_ss(tmem + sb * BN, ad, bd, kIdescS, ks > 0 ? 1u : 0u);
        }
        tc::commit(s_full + sb);
        tc::commit(k_empty + sb);
        if (j >= 1) pv(j - 1);
      }
      pv(n - 1);
      // the stage-release arrivals must land before the CTA (and its smem)
      // goes away
      for (int j = (n > 2 ? n - 2 : 0); j < n; ++j) {
        mbar_wait(k_empty + (j & 1), (j >> 1) & 1, a.err, dead);
        mbar_wait(v_empty + (j & 1), (j >> 1) & 1, a.err, dead);
      }
    }
  } else {
    // ============================ softmax warps 2..5 ========================
    bool dead = false;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const int p = p_begin + (r >> a.log2G);
    const bool row_valid = p < p_end;
    const int qpos = off + p;
    int khi = k_len, klo = 0;
    if (a.causal) {
      khi = min(k_len, qpos + 1);
      if (a.window > 0) klo = max(0, qpos - a.window + 1);
    }
    float m = -INFINITY, l = 0.f;
    const float sl2 = a.scale_log2;
    for (int j = 0; j < n; ++j) {
      const int sb = j & 1;
      mbar_wait(s_full + sb, (j >> 1) & 1, a.err, dead);
      tc::fence_after_sync();
      uint32_t s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
        tc::ld_32x32b_x32(lane_addr + sb * BN + c * 32,
                          *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
      tc::wait_ld();
      tc::fence_before_sync();
      mbar_arrive(s_free + sb);

      const int key0 = (t_lo + j) * BN;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        const int k = key0 + c;
        const float v = (k >= klo && k < khi) ? __uint_as_float(s[c]) * sl2 : -INFINITY;
        s[c] = __float_as_uint(v);
        mx = fmaxf(mx, v);
      }
      const float m_new = fmaxf(m, mx);
      const bool resc = m_new > m + 8.0f;  // false while both are -inf
      float alpha = 1.f;
      if (resc) {
        alpha = exp2f(m - m_new);  // 0 when m = -inf
        m = m_new;
      }
      const float mu = m == -INFINITY ? 0.f : m;
      l *= alpha;

      if (j >= 1) {
        mbar_wait(o_done, (j - 1) & 1, a.err, dead);
        tc::fence_after_sync();
      }
      // P row -> smem (bf16, K-major, 128-byte swizzle), 8 keys per 16 B
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < BN / 8; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = exp2f(__uint_as_float(s[u * 8 + 2 * e]) - mu);
          const float p1 = exp2f(__uint_as_float(s[u * 8 + 2 * e + 1]) - mu);
          sum += p0 + p1;
          w[e] = pack_bf16(p0, p1);
        }
        const uint32_t addr = sP + (u >> 3) * 16384 + r * 128 + (((u & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      l += sum;
      // O *= alpha (rows whose max grew by > 2^8); warp-collective TMEM access
      if (j >= 1 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::ld_32x32b_x32(lane_addr + 2 * BN + c * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::st_32x32b_x32(lane_addr + 2 * BN + c * 32, o);
        }
        tc::wait_st();
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(p_full);
    }
    // epilogue: O / l -> bf16 rows
    mbar_wait(o_done, (n - 1) & 1, a.err, dead);
    tc::fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(
        a.out + ((int64_t)(q0 + (row_valid ? p : p_begin)) * a.H_q + g * a.G +
                 (r & (a.G - 1))) * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tc::ld_32x32b_x32(lane_addr + 2 * BN + c * 32, o);
      tc::wait_ld();
      if (row_valid) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 pk;
          pk.x = pack_bf16(__uint_as_float(o[v * 8 + 0]) * inv, __uint_as_float(o[v * 8 + 1]) * inv);
          pk.y = pack_bf16(__uint_as_float(o[v * 8 + 2]) * inv, __uint_as_float(o[v * 8 + 3]) * inv);
          pk.z = pack_bf16(__uint_as_float(o[v * 8 + 4]) * inv, __uint_as_float(o[v * 8 + 5]) * inv);
          pk.w = pack_bf16(__uint_as_float(o[v * 8 + 6]) * inv, __uint_as_float(o[v * 8 + 7]) * inv);
          dst[c * 4 + v] = pk;
        }
      }
    }
    tc::fence_before_sync();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------- host side
template <int D, int BN>
static cudaError_t launch_varlen_t(const VarlenArgs& a, const VarlenMaps& maps, int batch,
                                   cudaStream_t stream) {
  using S_ = VarlenSmem<D, BN>;
  auto kern = varlen_fwd_kernel<D, BN>;
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S_::kBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_qtiles, a.H_kv, batch);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = S_::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, maps.q, maps.k, maps.v);
}

cudaError_t launch_varlen(void* out, const VarlenMaps& maps, const int32_t* cu_q,
                          const int32_t* cu_k, const int32_t* block_table, int32_t max_blocks,
                          int32_t batch, int32_t max_seqlen_q, int32_t total_q, int32_t H_q,
                          int32_t H_kv, int32_t D, int32_t P, int64_t num_pages, float scale,
                          int32_t causal, int32_t window, int32_t* err, cudaStream_t stream,
                          int num_sms) {
  (void)total_q;
  (void)num_sms;
  VarlenArgs a;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.cu_q = cu_q;
  a.cu_k = cu_k;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.H_q = H_q;
  a.H_kv = H_kv;
  a.G = H_q / H_kv;
  a.log2G = 0;
  while ((1 << a.log2G) < a.G) ++a.log2G;
  if ((1 << a.log2G) != a.G || a.G > 128) return cudaErrorNotSupported;
  const int QP = 128 / a.G;
  a.num_qtiles = (max_seqlen_q + QP - 1) / QP;
  if (a.num_qtiles == 0) return cudaSuccess;
  if (a.num_qtiles > 65535 * 32) return cudaErrorNotSupported;
  a.P = P;
  a.num_pages = num_pages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal;
  a.window = window;
  a.err = err;
  if (batch > 65535 || H_kv > 65535) return cudaErrorNotSupported;
  switch (D) {
    case 64: a.box_rows = P < 128 ? P : 128; return launch_varlen_t<64, 128>(a, maps, batch, stream);
    case 128: a.box_rows = P < 128 ? P : 128; return launch_varlen_t<128, 128>(a, maps, batch, stream);
    case 256: a.box_rows = P < 64 ? P : 64; return launch_varlen_t<256, 64>(a, maps, batch, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pkv
