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
//  * Persistent: one CTA per SM walks a work list.  A work item is NQ
//    consecutive 128-row Q tiles of one (chunk, kv head); the 128 MMA rows
//    of a Q tile pack 128/G query positions x the G query heads sharing
//    the kv head, so a K/V tile staged once in shared memory feeds the
//    whole GQA group and, with NQ = 2, two Q tiles.
//  * Every CTA derives the same schedule from cu_seq_lens in its prologue:
//    items are ordered by their distance from the end of their chunk (the
//    last item of each chunk -- the one that sees the most keys -- first),
//    chunks with more items first; CTA c takes items c, c+grid, ...
//  * Warp 0: TMA producer (Q tiles per item; K and V 64-key tiles through
//    two 2-deep rings, one box per page slice, 128-byte swizzle).  Boxes
//    outside the attended key range or the pool are fetched at an
//    out-of-range coordinate, which fills zeros.
//  * Warp 1: allocates 512 TMEM columns and issues tcgen05.mma
//    (cta_group::1, kind::f16, bf16 in, fp32 accumulate):
//        S_x  = Q_x K^T   (M=128, N=64, K=D)   one S buffer per Q tile
//        O_x += P_x V     (M=128, N=D,  K=64)  P from smem, V MN-major
//  * One softmax warpgroup per Q tile (one thread per row): tcgen05.ld the
//    S row, mask, online softmax in the exp2 domain, write P (bf16,
//    swizzled) to smem, rescale O in TMEM only when the running max grew
//    by more than 2^8 (the stale max is exact math: O and l share it),
//    epilogue O / l -> bf16.  The two warpgroups alternate with the tensor
//    core: while one runs its softmax the MMAs of the other proceed.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {

constexpr int kVBN = 64;  // keys per K/V tile
constexpr int kMaxSortPairs = 256;  // (chunk, item) pairs ordered by exact length

struct VarlenArgs {
  __nv_bfloat16* out;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* block_table;
  int32_t batch;
  int32_t max_blocks;
  int32_t max_q;       // clamp for q_len (max_seqlen_q)
  int32_t R;           // max items per (chunk, head) = ceil(max_q / (NQ*QP))
  int32_t pairs_max;   // batch * R: an upper bound of the (chunk, item) pairs
  int32_t H_q, H_kv, G, log2G, P, box_rows;
  int64_t num_pages;
  float scale_log2;
  int32_t causal, window;
  int32_t* err;
};

template <int D, int NQ, int NKV>
struct VarlenSmem {
  static constexpr int kQBytes = 128 * D * 2;            // one Q tile
  static constexpr int kKVChunk = kVBN * 128;            // one 64-column chunk of a K/V tile
  static constexpr int kKVBytes = (D / 64) * kKVChunk;   // one K (or V) tile
  static constexpr int kPBytes = 128 * kVBN * 2;         // one P tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + NQ * kQBytes;
  static constexpr int kVOff = kKOff + NKV * kKVBytes;
  static constexpr int kPOff = kVOff + NKV * kKVBytes;
  static constexpr int kBarOff = kPOff + NQ * kPBytes;
  // q_full, q_empty, k_full[NKV], k_empty[NKV], v_full[NKV], v_empty[NKV],
  // s_full[NQ], s_free[NQ], p_full[NQ], o_done[NQ]
  static constexpr int kNumBars = 2 + 4 * NKV + 4 * NQ;
  static constexpr int kTmemOff = kBarOff + kNumBars * 8;
  static constexpr int kSchedOff = kTmemOff + 16;
  // then: q_len[B] k_len[B] pair_prefix[B+1] key[P] order[P] with
  // P = min(pairs, kMaxSortPairs)
  static size_t bytes(int batch, int pairs) {
    const size_t np = (size_t)(pairs < kMaxSortPairs ? pairs : kMaxSortPairs);
    const size_t need = kSchedOff + (size_t)batch * 8 + (size_t)(batch + 1) * 4 + np * 8 + 16;
    // at least 116 KB so that only one CTA (and its 512 TMEM columns) fits
    // on an SM
    return 1024 + (need > 116 * 1024 ? need : 116 * 1024);
  }
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x on the FMA/ALU pipes, for x <= 8 (the softmax's stale-max bound):
// x = n + f with n = round(x) (added to the exponent field) and
// f in [-1/2, 1/2]; 2^f by a cubic fitted here to minimise relative error on
// that interval (max relative error 2.2e-4, below bf16 resolution of P).
// x < -125 returns 0 like the hardware exp2 of a masked (-inf) score.
__device__ __forceinline__ float poly_exp2(float x) {
  const float xc = fmaxf(x, -125.f);
  const float t = xc + 12582912.f;  // 1.5 * 2^23: rounds xc to an integer
  const int n = __float_as_int(t) - 0x4B400000;
  const float f = xc - (t - 12582912.f);
  float p = fmaf(0.05286737531423569f, f, 0.24215202033519745f);
  p = fmaf(p, f, 0.6935867667198181f);
  p = fmaf(p, f, 0.9999627470970154f);
  const float y = __int_as_float(__float_as_int(p) + (n << 23));
  return x < -125.f ? 0.f : y;
}

// Item geometry shared by every role of the CTA.
struct Item {
  int b, g, qp;          // chunk, kv head, index of the item within the chunk
  int q0, q_len, k_len;  // chunk's first row in q/out, its query and key counts
  int p_begin;           // first chunk row of the item
  int t_lo, n;           // first KV tile, number of KV tiles (0: no key for any row)
  int kv_lo, kv_hi;      // attended key range of the item
};

template <int NQ>
__device__ __forceinline__ Item make_item(const VarlenArgs& a, int b, int g, int qp, int q0,
                                          int q_len, int k_len) {
  Item it;
  it.b = b;
  it.g = g;
  it.qp = qp;
  it.q0 = q0;
  it.q_len = q_len;
  it.k_len = k_len;
  const int QP = 128 >> a.log2G;
  it.p_begin = qp * NQ * QP;
  const int p_end = min(it.p_begin + NQ * QP, q_len);
  const int off = k_len - q_len;
  int lo = 0, hi = k_len;
  if (a.causal) {
    hi = min(k_len, off + p_end);
    if (a.window > 0) lo = max(0, off + it.p_begin - a.window + 1);
  }
  it.kv_lo = lo;
  it.kv_hi = hi;
  it.t_lo = lo / kVBN;
  it.n = hi > lo ? (hi + kVBN - 1) / kVBN - it.t_lo : 0;
  return it;
}

template <int D, int NQ, int NKV>
__global__ void __launch_bounds__((3 + 4 * NQ) * 32, 1)
    varlen_fwd_kernel(const VarlenArgs a, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  using S_ = VarlenSmem<D, NQ, NKV>;
  constexpr int NT = (3 + 4 * NQ) * 32;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, kVBN, false);
  constexpr uint32_t kIdescO = tc::idesc_bf16_f32(128, D, true);
  constexpr int kOCol = NQ * kVBN;  // O_x at kOCol + x*D; S_x at x*kVBN

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S_::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;               // [NKV]
  uint64_t* k_empty = k_full + NKV;          // [NKV]
  uint64_t* v_full = k_empty + NKV;          // [NKV]
  uint64_t* v_empty = v_full + NKV;          // [NKV]
  uint64_t* s_full = v_empty + NKV;          // [NQ]
  uint64_t* s_free = s_full + NQ;            // [NQ]
  uint64_t* p_full = s_free + NQ;            // [NQ]
  uint64_t* o_done = p_full + NQ;            // [NQ]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S_::kTmemOff);
  int* s_qlen = reinterpret_cast<int*>(smem + S_::kSchedOff);  // clamped q_len per chunk
  int* s_klen = s_qlen + a.batch;                              // clamped k_len per chunk
  int* s_pfx = s_klen + a.batch;                               // [B+1] pairs before chunk b
  int* s_key = s_pfx + a.batch + 1;                            // KV tiles of pair p
  int* s_porder = s_key + min(a.pairs_max, kMaxSortPairs);     // pairs, most tiles first

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int B = a.batch;
  const int QP = 128 >> a.log2G;

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < NKV; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int x = 0; x < NQ; ++x) {
      mbar_init(s_full + x, 1);
      mbar_init(s_free + x, 128);
      mbar_init(p_full + x, 128);
      mbar_init(o_done + x, 1);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::tmem_relinquish();
  }
  pdl_wait();  // inputs may come from the previous kernel in the stream

  // ------------------------------------------------ schedule (every CTA)
  // A pair (chunk b, item qp) covers NQ Q tiles of chunk b; with the H_kv
  // heads it makes H_kv work items of equal cost.  Pairs are ordered by
  // their number of KV tiles, most first (exactly, up to kMaxSortPairs
  // pairs; beyond that in chunk order), and the sorted items are dealt to
  // the CTAs in a snake (0..N-1, N-1..0, ...) so that every CTA gets a
  // similar total.
  const int kcap = a.max_blocks * a.P;
  for (int b = tid; b < B; b += NT) {
    const int q0 = __ldg(a.cu_q + b);
    int ql = __ldg(a.cu_q + b + 1) - q0;
    int kl = __ldg(a.cu_k + b + 1) - __ldg(a.cu_k + b);
    ql = ql < 0 ? 0 : (ql > a.max_q ? a.max_q : ql);
    kl = kl < 0 ? 0 : (kl > kcap ? kcap : kl);
    s_qlen[b] = ql;
    s_klen[b] = kl;
  }
  __syncthreads();
  if (tid == 0) {  // pair prefix over chunks (B <= 1024)
    int run = 0;
    for (int b = 0; b < B; ++b) {
      s_pfx[b] = run;
      int ni = (s_qlen[b] + NQ * QP - 1) / (NQ * QP);
      run += ni < a.R ? ni : a.R;
    }
    s_pfx[B] = run;
  }
  __syncthreads();
  const int TP = s_pfx[B];
  const bool sorted = TP <= kMaxSortPairs;
  auto pair_at = [&](int p, int& b, int& qp) {
    int lo = 0, hi = B;  // s_pfx[lo] <= p < s_pfx[lo+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pfx[mid] <= p) lo = mid; else hi = mid;
    }
    b = lo;
    qp = p - s_pfx[lo];
  };
  if (sorted) {
    for (int p = tid; p < TP; p += NT) {
      int b, qp;
      pair_at(p, b, qp);
      s_key[p] = make_item<NQ>(a, b, 0, qp, 0, s_qlen[b], s_klen[b]).n;
    }
    __syncthreads();
    for (int p = tid; p < TP; p += NT) {
      const int kp = s_key[p];
      int rank = 0;
      for (int j = 0; j < TP; ++j) {
        const int kj = s_key[j];
        rank += (kj > kp || (kj == kp && j < p)) ? 1 : 0;
      }
      s_porder[rank] = p;
    }
  }
  __syncthreads();
  const int T = TP * a.H_kv;
  pdl_launch_dependents();

  // item i (sorted order) -> (chunk, head, item within chunk); identical in
  // every role
  auto item_at = [&](int i) -> Item {
    const int sp = i / a.H_kv;
    const int g = i - sp * a.H_kv;
    const int p = sorted ? s_porder[sp] : sp;
    int b, qp;
    pair_at(p, b, qp);
    return make_item<NQ>(a, b, g, qp, __ldg(a.cu_q + b), s_qlen[b], s_klen[b]);
  };
  // the k-th item of this CTA (snake over the CTAs)
  const int NC = gridDim.x;
  auto my_item = [&](int k) -> int {
    const int c = (k & 1) ? NC - 1 - (int)blockIdx.x : (int)blockIdx.x;
    return k * NC + c;
  };

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  const uint32_t sQ = smem_u32(smem + S_::kQOff);
  const uint32_t sK = smem_u32(smem + S_::kKOff);
  const uint32_t sV = smem_u32(smem + S_::kVOff);
  const uint32_t sP = smem_u32(smem + S_::kPOff);

  if (blockIdx.x == 0 && tid == 0) {  // report clamped lengths once
    for (int b = 0; b < B; ++b) {
      const int ql = __ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b);
      const int kl = __ldg(a.cu_k + b + 1) - __ldg(a.cu_k + b);
      if (ql < 0 || ql > a.max_q || ql > a.R * NQ * QP || kl < 0 ||
          kl > a.max_blocks * a.P)
        raise_err(a.err, PKV_DEVERR_LEN);
    }
  }

  if (warp == 0 || warp == 2 + 4 * NQ) {
    // ========================= TMA producers (K and V) ======================
    // Warp 0 loads Q and K, the last warp loads V: the two rings run
    // independently, so a K tile never waits for a V stage to be released
    // (which would tie the K prefetch to the PV progress).
    const bool isK = warp == 0;
    bool dead = false;
    const int R = a.box_rows;
    const int nsub = kVBN / R;
    const int oob = (int)(a.num_pages * a.H_kv);  // first z past the pool: zero fill
    uint64_t* ring_full = isK ? k_full : v_full;
    uint64_t* ring_empty = isK ? k_empty : v_empty;
    const CUtensorMap* tm = isK ? &tmK : &tmV;
    const int ring_off = isK ? S_::kKOff : S_::kVOff;
    int t = 0;      // KV tiles issued by this CTA
    int nitem = 0;  // non-empty items loaded by this CTA
    for (int kk_ = 0, i = my_item(0); i < T; ++kk_, i = my_item(kk_)) {
      const Item it = item_at(i);
      if (it.n == 0) continue;
      const int* bt = a.block_table + (int64_t)it.b * a.max_blocks;
      if (isK && lane == 0) {
        if (nitem > 0) mbar_wait(q_empty, (nitem - 1) & 1, a.err, dead);
        mbar_arrive_expect_tx(q_full, NQ * S_::kQBytes);
#pragma unroll
        for (int x = 0; x < NQ; ++x)
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(smem + S_::kQOff + x * S_::kQBytes + c * 16384, &tmQ, q_full, c * 64, 0,
                        it.g, it.q0 + it.p_begin + x * QP);
      }
      ++nitem;
      for (int j = 0; j < it.n; ++j, ++t) {
        const int key_base = (it.t_lo + j) * kVBN;
        int z = oob, row = 0;
        if (lane < nsub) {
          const int key0 = key_base + lane * R;
          row = key0 % a.P;
          if (key0 < it.kv_hi && key0 + R > it.kv_lo) {
            const int pg = __ldg(bt + key0 / a.P);
            if (pg >= 0 && (int64_t)pg < a.num_pages) z = pg * a.H_kv + it.g;
            else if (isK) raise_err(a.err, PKV_DEVERR_PAGE);
          }
        }
        int zs[4], rows[4];
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          zs[i2] = __shfl_sync(0xffffffffu, z, i2);
          rows[i2] = __shfl_sync(0xffffffffu, row, i2);
        }
        if (lane == 0) {
          const int s = t % NKV;
          const int rr = t / NKV;
          if (rr >= 1) mbar_wait(ring_empty + s, (rr - 1) & 1, a.err, dead);
          mbar_arrive_expect_tx(ring_full + s, S_::kKVBytes);
          uint8_t* dst = smem + ring_off + s * S_::kKVBytes;
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2)
            if (i2 < nsub)
#pragma unroll
              for (int c = 0; c < D / 64; ++c)
                tma_load_3d(dst + c * S_::kKVChunk + i2 * R * 128, tm, ring_full + s, c * 64,
                            rows[i2], zs[i2]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {  // every issued copy must land before the CTA exits
      for (int u = (t > NKV ? t - NKV : 0); u < t; ++u)
        mbar_wait(ring_full + (u % NKV), (u / NKV) & 1, a.err, dead);
      if (isK && nitem > 0) mbar_wait(q_full, (nitem - 1) & 1, a.err, dead);
    }
  } else if (warp == 1) {
    // =============================== MMA issuer =============================
    if (lane == 0) {
      bool dead = false;
      int t = 0, nitem = 0;
      // descriptor low halves of the operand bases (K-major Q, K, P: LBO 16;
      // MN-major V: LBO = the 64-column chunk stride); all share one high half
      constexpr uint32_t kHi = tc::sw128_hi(1024);
      const uint32_t q_lo0 = tc::sw128_lo(sQ, 16);
      const uint32_t k_lo0 = tc::sw128_lo(sK, 16);
      const uint32_t p_lo0 = tc::sw128_lo(sP, 16);
      const uint32_t v_lo0 = tc::sw128_lo(sV, S_::kKVChunk);
      // O_x += P_x V(u) for Q tile x; V(u) must have landed
      auto pv_x = [&](int u, int x, bool first) {
        const int vb = u % NKV;
        mbar_wait(v_full + vb, (u / NKV) & 1, a.err, dead);
        mbar_wait(p_full + x, u & 1, a.err, dead);
        tc::fence_after_sync();
        const uint32_t alo = p_lo0 + x * (S_::kPBytes >> 4);
        const uint32_t blo = v_lo0 + vb * (S_::kKVBytes >> 4);
#pragma unroll
        for (int ks = 0; ks < kVBN / 16; ++ks)
          tc::mma_ss_h(tmem + kOCol + x * D, alo + ks * (32 >> 4), kHi, blo + ks * (2048 >> 4),
                       kHi, kIdescO, (!first || ks > 0) ? 1u : 0u);
        tc::commit(o_done + x);
      };
      for (int kk_ = 0, i = my_item(0); i < T; ++kk_, i = my_item(kk_)) {
        const Item it = item_at(i);
        if (it.n == 0) continue;
        mbar_wait(q_full, nitem & 1, a.err, dead);
        for (int j = 0; j < it.n; ++j, ++t) {
          const int kb = t % NKV;
          mbar_wait(k_full + kb, (t / NKV) & 1, a.err, dead);
          const uint32_t klo = k_lo0 + kb * (S_::kKVBytes >> 4);
          // per Q tile: S_x of this KV tile, then PV_x of the previous one, so
          // one warpgroup's softmax never waits on the other's progress
#pragma unroll
          for (int x = 0; x < NQ; ++x) {
            if (t >= 1) mbar_wait(s_free + x, (t - 1) & 1, a.err, dead);
            tc::fence_after_sync();
            const uint32_t qlo = q_lo0 + x * (S_::kQBytes >> 4);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              tc::mma_ss_h(tmem + x * kVBN, qlo + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), kHi,
                           klo + (((ks >> 2) * S_::kKVChunk + (ks & 3) * 32) >> 4), kHi,
                           kIdescS, ks > 0 ? 1u : 0u);
            tc::commit(s_full + x);
            if (j >= 1) pv_x(t - 1, x, j == 1);
          }
          if (j == it.n - 1) tc::commit(q_empty);
          tc::commit(k_empty + kb);
          if (j >= 1) tc::commit(v_empty + ((t - 1) % NKV));
        }
#pragma unroll
        for (int x = 0; x < NQ; ++x) pv_x(t - 1, x, it.n == 1);
        tc::commit(v_empty + ((t - 1) % NKV));
        ++nitem;
      }
      // the stage-release arrivals must land before the CTA (and its smem)
      // goes away
      for (int u = (t > NKV ? t - NKV : 0); u < t; ++u) {
        mbar_wait(k_empty + (u % NKV), (u / NKV) & 1, a.err, dead);
        mbar_wait(v_empty + (u % NKV), (u / NKV) & 1, a.err, dead);
      }
      if (nitem > 0) mbar_wait(q_empty, (nitem - 1) & 1, a.err, dead);
    }
  } else {
    // ======================== softmax warpgroups ============================
    bool dead = false;
    const int x = (warp - 2) >> 2;  // which Q tile of the item
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_addr = lane_base + x * kVBN;
    const uint32_t o_addr = lane_base + kOCol + x * D;
    const uint32_t prow = sP + x * S_::kPBytes + r * 128;
    const float sl2 = a.scale_log2;
    int t = 0;
    for (int kk_ = 0, i = my_item(0); i < T; ++kk_, i = my_item(kk_)) {
      const Item it = item_at(i);
      const int p = it.p_begin + x * QP + (r >> a.log2G);  // chunk row of this thread
      const bool row_valid = p < it.q_len;
      const int hh = r & (a.G - 1);
      __nv_bfloat16* orow =
          a.out + ((int64_t)(it.q0 + (row_valid ? p : 0)) * a.H_q + it.g * a.G + hh) * D;
      if (it.n == 0) {  // no key for any row of the item: zero rows
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int qpos = it.k_len - it.q_len + p;
      int khi = it.k_len, klo = 0;
      if (a.causal) {
        khi = min(it.k_len, qpos + 1);
        if (a.window > 0) klo = max(0, qpos - a.window + 1);
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n; ++j, ++t) {
        mbar_wait(s_full + x, t & 1, a.err, dead);
        tc::fence_after_sync();
        uint32_t s[kVBN];
        tc::ld_32x32b_x32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tc::ld_32x32b_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tc::wait_ld();
        tc::fence_before_sync();
        mbar_arrive(s_free + x);

        // mask only where a key of this tile falls outside a row's range
        const int key0 = (it.t_lo + j) * kVBN;
        const bool inside = key0 >= klo && key0 + kVBN <= khi;
        float mxp[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mxp[c] = -INFINITY;
        if (__all_sync(0xffffffffu, inside)) {
#pragma unroll
          for (int c = 0; c < kVBN; ++c) mxp[c & 7] = fmaxf(mxp[c & 7], __uint_as_float(s[c]));
        } else {
#pragma unroll
          for (int c = 0; c < kVBN; ++c) {
            const int k = key0 + c;
            const float v = (k >= klo && k < khi) ? __uint_as_float(s[c]) : -INFINITY;
            s[c] = __float_as_uint(v);
            mxp[c & 7] = fmaxf(mxp[c & 7], v);
          }
        }
        const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                               fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
        // running max in the log2 domain (scale > 0 commutes with max)
        const float mt = mx * sl2;
        const float m_new = fmaxf(m, mt);
        const bool resc = m_new > m + 8.0f;  // false while both are -inf
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m - m_new);  // 0 when m = -inf
          m = m_new;
        }
        const float mu = m == -INFINITY ? 0.f : m;
        l *= alpha;

        if (t >= 1) {  // PV of the previous tile must be done with P and O
          mbar_wait(o_done + x, (t - 1) & 1, a.err, dead);
          tc::fence_after_sync();
        }
        float sp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < kVBN / 8; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // half of the exponentials on the SFU, half on the FMA pipes
            const float x0 = fmaf(__uint_as_float(s[u * 8 + 2 * e]), sl2, -mu);
            const float x1 = fmaf(__uint_as_float(s[u * 8 + 2 * e + 1]), sl2, -mu);
            const float p0 = (u & 1) ? poly_exp2(x0) : fast_exp2(x0);
            const float p1 = (u & 1) ? poly_exp2(x1) : fast_exp2(x1);
            sp[e] += p0 + p1;
            w[e] = pack_bf16(p0, p1);
          }
          const uint32_t addr = prow + ((u ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]),
                       "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
        l += (sp[0] + sp[1]) + (sp[2] + sp[3]);
        if (j >= 1 && __any_sync(0xffffffffu, resc)) {  // O *= alpha (warp-collective)
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc::ld_32x32b_x32(o_addr + c * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st_32x32b_x32(o_addr + c * 32, o);
          }
          tc::wait_st();
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        mbar_arrive(p_full + x);
      }
      // epilogue: O / l -> bf16 rows
      mbar_wait(o_done + x, (t - 1) & 1, a.err, dead);
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::ld_32x32b_x32(o_addr + c * 32, o);
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
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// --------------------------------------------------------------- host side
template <int D, int NQ, int NKV>
static cudaError_t launch_varlen_t(const VarlenArgs& a, const VarlenMaps& maps,
                                   cudaStream_t stream, int num_sms) {
  using S_ = VarlenSmem<D, NQ, NKV>;
  auto kern = varlen_fwd_kernel<D, NQ, NKV>;
  const size_t smem = S_::bytes(a.batch, a.pairs_max);
  if (smem > 227 * 1024) {
    // the deep K/V ring does not fit next to this batch's schedule: use 2 stages
    if (NKV > 2) return launch_varlen_t<D, NQ, 2>(a, maps, stream, num_sms);
    return cudaErrorNotSupported;
  }
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
  // persistent grid: one CTA per SM, never more CTAs than work items
  const int64_t items_max = (int64_t)a.batch * a.H_kv * a.R;
  const int64_t grid = items_max < num_sms ? items_max : num_sms;
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((3 + 4 * NQ) * 32);
  cfg.dynamicSmemBytes = smem;
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
  VarlenArgs a;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.cu_q = cu_q;
  a.cu_k = cu_k;
  a.block_table = block_table;
  a.batch = batch;
  a.max_blocks = max_blocks;
  a.max_q = max_seqlen_q;
  a.H_q = H_q;
  a.H_kv = H_kv;
  a.G = H_q / H_kv;
  a.log2G = 0;
  while ((1 << a.log2G) < a.G) ++a.log2G;
  if ((1 << a.log2G) != a.G || a.G > 128) return cudaErrorNotSupported;
  if (batch > 1024) return cudaErrorNotSupported;
  const int QP = 128 / a.G;
  a.P = P;
  a.box_rows = P < kVBN ? P : kVBN;
  a.num_pages = num_pages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal;
  a.window = window;
  a.err = err;
  if (max_seqlen_q <= 0) return cudaSuccess;
  switch (D) {
    case 64:
      a.R = (max_seqlen_q + 2 * QP - 1) / (2 * QP);
      a.pairs_max = batch * a.R;
      return launch_varlen_t<64, 2, 4>(a, maps, stream, num_sms);
    case 128:
      a.R = (max_seqlen_q + 2 * QP - 1) / (2 * QP);
      a.pairs_max = batch * a.R;
      return launch_varlen_t<128, 2, 4>(a, maps, stream, num_sms);
    case 256:
      a.R = (max_seqlen_q + QP - 1) / QP;
      a.pairs_max = batch * a.R;
      return launch_varlen_t<256, 1, 2>(a, maps, stream, num_sms);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace pkv
