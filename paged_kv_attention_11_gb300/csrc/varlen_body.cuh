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
//    (chunk, item) pairs sorted by their number of KV tiles, most first (up
//    to 256 pairs; beyond that in chunk order), dealt to the CTAs in a snake
//    so that every CTA gets a similar total.
//  * The CTA's items form one stream of KV tiles; no role drains at an
//    item boundary.  Two producer warps load with TMA (128-byte swizzle, one
//    box per page slice, lane-parallel issue): one the K tiles (and the Q
//    tiles when the stream enters an item), one the V tiles, each through
//    its own ring.
//  * The MMA warp (warp 4*NQ+1) allocates 512 TMEM columns and issues
//    tcgen05.mma (cta_group::1, kind::f16, bf16 in, fp32 accumulate) as a
//    converged warp, one elected lane per operation:
//        S_x(t)  = Q_x K(t)^T        smem x smem -> TMEM  (M=128, N=BN)
//        O_x    += P_x(t) V(t)       TMEM x smem -> TMEM  (M=128, N=D)
//    P_x(t) is written by the softmax into the TMEM columns of S_x(t), as
//    bf16 pairs, and read from there by the PV MMA.  Per tile t and Q tile
//    x the issue order is PV_x(t), QK_x(t+NS): the tensor pipe runs one
//    thread's MMAs in issue order, so S_x(t+NS) may reuse the columns P_x(t)
//    was read from.
//    With NQ = 2 (NS = 1) the two Q tiles' softmaxes alternate with the
//    tensor core; with NQ = 1 (NS = 2, head_dim 256) S is double-buffered
//    so that QK of the next tile runs under the softmax of this one.
//  * One softmax warpgroup per Q tile (one thread per row): tcgen05.ld the
//    S row, mask (boundary tiles only), online softmax in the exp2 domain
//    (packed f32x2 arithmetic; an eighth of the exponentials on the FMA
//    pipes, the rest on the SFU), P -> TMEM, rescale O in TMEM only when the
//    running max grew by more than 2^8 (the stale max is exact math: O and
//    l share it), epilogue O / l -> bf16.
#pragma once

#include <math.h>

#include "common.cuh"
#include "exp2_math.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkv {

// (chunk, item) pairs ordered by exact length; head_dim 512 keeps fewer, its
// tiles leave less shared memory for the schedule
template <int D>
constexpr int max_sort_pairs() {
  return D >= 512 ? 32 : 256;
}

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
  int32_t out_v8;  // out is 32-byte aligned: the epilogue writes 32-byte words
  int32_t* err;
};

#ifndef PKV_VAR_EPI_BATCH
#define PKV_VAR_EPI_BATCH 1
#endif

// One 32-byte global store of 8 words (dst 32-byte aligned).
__device__ __forceinline__ void st_global_v8(uint32_t* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// DV: the width of O (and of the V columns) one work item computes; D / DV
// items cover a Q tile (head_dim 512: two halves of 256, each recomputing S)
template <int D, int NQ, int BN, int NS, int NKS, int NVS, int DV = D>
struct VarlenSmem {
  static constexpr int kQBytes = 128 * D * 2;              // one Q tile
  // a K/V tile is [row group][64-column chunk][8 rows][128 B]: 8-row atoms
  // of a chunk kAtomStride apart (K: D/64 chunks; V: DV/64), chunks 1024 B
  // apart
  static constexpr int kAtomStride = (D / 64) * 1024;
  static constexpr int kVAtomStride = (DV / 64) * 1024;
  static constexpr int kSlotBytes = BN * D * 2;            // one K tile
  static constexpr int kVSlotBytes = BN * DV * 2;          // one V tile (DV columns)
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + NQ * kQBytes;   // K ring: NKS tiles
  static constexpr int kVOff = kKOff + NKS * kSlotBytes;  // V ring: NVS tiles
  static constexpr int kBarOff = kVOff + NVS * kVSlotBytes;
  // q_full[NQ] q_empty[NQ] k_full[NKS] k_empty[NKS] v_full[NVS] v_empty[NVS]
  // s_full[NQ*NS] p_full[NQ*NS] o_done[NQ]
  static constexpr int kNumBars = 2 * NQ + 2 * NKS + 2 * NVS + 2 * NQ * NS + NQ;
  static constexpr int kTmemOff = kBarOff + kNumBars * 8;
  static constexpr int kSchedOff = kTmemOff + 16;
  // then: q_len[B] k_len[B] pair_prefix[B+1] key[P] order[P] with
  // P = min(pairs, max_sort_pairs<D>())
  static size_t bytes(int batch, int pairs) {
    constexpr int kMaxSortPairs = max_sort_pairs<D>();
    const size_t np = (size_t)(pairs < kMaxSortPairs ? pairs : kMaxSortPairs);
    const size_t need = kSchedOff + (size_t)batch * 8 + (size_t)(batch + 1) * 4 + np * 8 + 16;
    // at least 116 KB so that only one CTA (and its 512 TMEM columns) fits
    // on an SM
    return 1024 + (need > 116 * 1024 ? need : 116 * 1024);
  }
};

// Item geometry shared by every role of the CTA.
struct Item {
  int b, g, qp;          // chunk, kv head, index of the item within the chunk
  int half;              // which DV-wide part of O (0 when DV == D)
  int q0, q_len, k_len;  // chunk's first row in q/out, its query and key counts
  int p_begin;           // first chunk row of the item
  int t_lo, n;           // first KV tile, number of KV tiles (0: no key for any row)
  int kv_lo, kv_hi;      // attended key range of the item
};

template <int NQ, int BN>
__device__ __forceinline__ Item make_item(const VarlenArgs& a, int b, int g, int qp, int q0,
                                          int q_len, int k_len, int half = 0) {
  Item it;
  it.b = b;
  it.g = g;
  it.qp = qp;
  it.half = half;
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
  it.t_lo = lo / BN;
  it.n = hi > lo ? (hi + BN - 1) / BN - it.t_lo : 0;
  return it;
}

// Position in the CTA's stream of KV tiles: item ordinal k of this CTA,
// tile j of that item, and m, the ordinal of the item among the CTA's
// non-empty items (the phase count of the Q buffers).
struct Cursor {
  int k, j, m;
  Item it;
};

// Warps: 4*NQ softmax warps (warpgroup x = Q tile x), then one warpgroup
// holding the TMA producer, the MMA issuer and two idle warps (whole
// warpgroups, so that registers can move to the softmax with setmaxnreg).
template <int NQ>
__host__ __device__ constexpr int varlen_threads() {
  return (4 * NQ + 4) * 32;
}

// The varlen work of one CTA (all varlen_threads<NQ>() threads of the
// block).  `cta` is this CTA's index among the `ncta` CTAs that share the
// static schedule; smem is the 1024-aligned dynamic shared memory.  HOSTED:
// the block runs other work afterwards (the mixed-step kernel): every warp
// keeps the launch's register count (no setmaxnreg moves, so each code path
// after the body sees the same budget) and the body invalidates its
// mbarriers before it returns.
template <int D, int NQ, int BN, int NS, int NKS, int NVS, bool HOSTED, int DV = D>
__device__ __forceinline__ void varlen_cta(const VarlenArgs& a, const CUtensorMap& tmQ,
                                           const CUtensorMap& tmK, const CUtensorMap& tmV,
                                           uint8_t* smem, int cta, int ncta) {
  using S_ = VarlenSmem<D, NQ, BN, NS, NKS, NVS, DV>;
  constexpr int NH = D / DV;  // O parts per Q tile
  static_assert(D % DV == 0 && DV % 64 == 0, "O parts");
  constexpr int NT = varlen_threads<NQ>();
  constexpr int kProdWarp = 4 * NQ;
  constexpr int kMmaWarp = 4 * NQ + 1;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, BN, false);
  constexpr uint32_t kIdescO = tc::idesc_bf16_f32(128, DV, true);
  constexpr int kOCol = NQ * NS * BN;  // S/P buffer (x, b) at (x*NS + b)*BN; O_x at kOCol + x*DV
  static_assert(kOCol + NQ * DV <= (int)kTmemCols, "TMEM columns");
  static_assert(BN == 32 || BN == 64 || BN == 128, "KV tile");

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S_::kBarOff);
  uint64_t* q_full = bars;                     // [NQ]
  uint64_t* q_empty = q_full + NQ;             // [NQ]
  uint64_t* k_full = q_empty + NQ;             // [NKS]
  uint64_t* k_empty = k_full + NKS;            // [NKS]
  uint64_t* v_full = k_empty + NKS;            // [NVS]
  uint64_t* v_empty = v_full + NVS;            // [NVS]
  uint64_t* s_full = v_empty + NVS;            // [NQ*NS]
  uint64_t* p_full = s_full + NQ * NS;         // [NQ*NS]
  uint64_t* o_done = p_full + NQ * NS;         // [NQ]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S_::kTmemOff);
  int* s_qlen = reinterpret_cast<int*>(smem + S_::kSchedOff);  // clamped q_len per chunk
  int* s_klen = s_qlen + a.batch;                              // clamped k_len per chunk
  int* s_pfx = s_klen + a.batch;                               // [B+1] pairs before chunk b
  int* s_key = s_pfx + a.batch + 1;                            // KV tiles of pair p
  constexpr int kMaxSortPairs = max_sort_pairs<D>();
  int* s_porder = s_key + min(a.pairs_max, kMaxSortPairs);     // pairs, most tiles first

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int B = a.batch;
  const int QP = 128 >> a.log2G;

  if (tid == 0) {
    for (int x = 0; x < NQ; ++x) {
      mbar_init(q_full + x, 1);
      mbar_init(q_empty + x, 1);
      mbar_init(o_done + x, 1);
    }
    for (int i = 0; i < NKS; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < NVS; ++i) {
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < NQ * NS; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 1);  // one arrive per warpgroup, after a named barrier
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_holder, kTmemCols);
    tc::tmem_relinquish();
  }
  pdl_wait();  // inputs may come from the previous kernel in the stream

  // ------------------------------------------------ schedule (every CTA)
  // A pair (chunk b, item qp) covers NQ Q tiles of chunk b; with the H_kv
  // heads it makes H_kv work items of equal cost.  Pairs are ordered by
  // their number of KV tiles, most first (exactly, up to max_sort_pairs
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
      s_key[p] = make_item<NQ, BN>(a, b, 0, qp, 0, s_qlen[b], s_klen[b]).n;
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
  const int T = TP * a.H_kv * NH;
  pdl_launch_dependents();

  // item i (sorted order) -> (chunk, head, item within chunk, O part);
  // identical in every role
  auto item_at = [&](int i) -> Item {
    const int sp = i / (a.H_kv * NH);
    const int r = i - sp * (a.H_kv * NH);
    const int g = r / NH, half = r - (r / NH) * NH;
    const int p = sorted ? s_porder[sp] : sp;
    int b, qp;
    pair_at(p, b, qp);
    return make_item<NQ, BN>(a, b, g, qp, __ldg(a.cu_q + b), s_qlen[b], s_klen[b], half);
  };
  // the k-th item of this CTA (snake over the CTAs)
  const int NC = ncta;
  auto my_item = [&](int k) -> int {
    const int c = (k & 1) ? NC - 1 - cta : cta;
    return k * NC + c;
  };
  // step to the next KV tile of the CTA's stream (skipping items without
  // keys); false at the end.  Start from {k = -1, j = 0, m = -1, it.n = 0}.
  auto next_tile = [&](Cursor& c) -> bool {
    if (++c.j < c.it.n) return true;
    while (true) {
      const int i = my_item(++c.k);
      if (i >= T) {
        c.it.n = 0;
        return false;
      }
      c.it = item_at(i);
      if (c.it.n > 0) {
        c.j = 0;
        ++c.m;
        return true;
      }
    }
  };
  auto cursor0 = []() {
    Cursor c;
    c.k = -1;
    c.j = 0;
    c.m = -1;
    c.it = Item{0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    return c;
  };

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  const uint32_t sQ = smem_u32(smem + S_::kQOff);

  if (cta == 0 && tid == 0) {  // report clamped lengths once
    for (int b = 0; b < B; ++b) {
      const int ql = __ldg(a.cu_q + b + 1) - __ldg(a.cu_q + b);
      const int kl = __ldg(a.cu_k + b + 1) - __ldg(a.cu_k + b);
      if (ql < 0 || ql > a.max_q || ql > a.R * NQ * QP || kl < 0 ||
          kl > a.max_blocks * a.P)
        raise_err(a.err, PKV_DEVERR_LEN);
    }
  }

  // the producer and the MMA issuer hold few registers, the softmax many;
  // each role's code sits under its own register change.  Launch: 384
  // threads x 168 registers; after the change 4 warps x 104 + 8 warps x 200
  // use the same total, and every SM sub-partition holds at most 504 per lane.
  if (warp >= kProdWarp) {
    if (NQ == 2 && !HOSTED) asm volatile("setmaxnreg.dec.sync.aligned.u32 104;" ::: "memory");
  if (warp == kProdWarp || warp == kProdWarp + 2) {
    // ====================== TMA producers: K (+Q) and V ======================
    // Warp kProdWarp loads the Q tiles and the K tiles, warp kProdWarp+2 the
    // V tiles, each through its own ring (one issuing warp sustains about
    // half the box rate of two).
    const bool isK = warp == kProdWarp;
    bool dead = false;
    const int R = a.box_rows;
    const int nbox = BN / R;                      // boxes (page slices) per tile
    const int oob = (int)(a.num_pages * a.H_kv);  // first z past the pool: zero fill
    // This lane's box of the cursor's tile: its row in the page and the
    // block-table entry, requested two tiles ahead and checked only when
    // the box is issued (box_z).  Boxes outside the attended range (or on a
    // bad page) are fetched at z = oob: zeros.
    struct Box {
      int pg, row, g;
      bool inr;
    };
    auto box_req = [&](const Cursor& c) -> Box {
      Box bx = {0, 0, c.it.g, false};
      if (lane < nbox) {
        const int key0 = (c.it.t_lo + c.j) * BN + lane * R;
        bx.row = key0 % a.P;
        bx.inr = key0 < c.it.kv_hi && key0 + R > c.it.kv_lo;
        if (bx.inr) bx.pg = __ldg(a.block_table + (int64_t)c.it.b * a.max_blocks + key0 / a.P);
      }
      return bx;
    };
    auto box_z = [&](const Box& bx) -> int {
      if (!bx.inr) return oob;
      if (bx.pg >= 0 && (int64_t)bx.pg < a.num_pages) return bx.pg * a.H_kv + bx.g;
      raise_err(a.err, PKV_DEVERR_PAGE);
      return oob;
    };
    auto load_q = [&](const Cursor& c) {  // lane 0: the Q tiles of the cursor's item
#pragma unroll
      for (int x = 0; x < NQ; ++x) {
        if (c.m >= 1) mbar_wait(q_empty + x, (c.m - 1) & 1, a.err, dead);
        mbar_arrive_expect_tx(q_full + x, S_::kQBytes);
#pragma unroll
        for (int ch = 0; ch < D / 64; ++ch)
          tma_load_4d(smem + S_::kQOff + x * S_::kQBytes + ch * 16384, &tmQ, q_full + x, ch * 64,
                      0, c.it.g, c.it.q0 + c.it.p_begin + x * QP);
      }
    };
    const int nring = isK ? NKS : NVS;
    uint64_t* rfull = isK ? k_full : v_full;
    uint64_t* rempty = isK ? k_empty : v_empty;
    uint8_t* rbase = smem + (isK ? S_::kKOff : S_::kVOff);
    const int slot_bytes = isK ? S_::kSlotBytes : S_::kVSlotBytes;
    const int row_bytes = (isK ? D : DV) * 2;  // one key's columns in the slot
    const CUtensorMap* tm = isK ? &tmK : &tmV;
    const Box none = {0, 0, 0, false};
    Cursor c0 = cursor0();  // tile being loaded
    bool h0 = next_tile(c0);
    Cursor c1 = c0;  // the next one
    bool h1 = h0 && next_tile(c1);
    Box b0 = h0 ? box_req(c0) : none;
    Box b1 = h1 ? box_req(c1) : none;
    int t = 0, s = 0, ph = 0;  // tiles loaded; ring slot and its phase
    while (h0) {
      if (lane == 0) {
        if (t >= nring) mbar_wait(rempty + s, ph ^ 1, a.err, dead);
        mbar_arrive_expect_tx(rfull + s, slot_bytes);
      }
      __syncwarp();
      const int z = box_z(b0);
      // V: the item's DV-wide column part, starting at 64-column chunk
      // half * DV / 64 of the pool rows
      const int chunk0 = isK ? 0 : c0.it.half * (DV / 64);
      if (lane < nbox)  // one box: this lane's page slice of the tile, its columns
        tma_load_5d(rbase + s * slot_bytes + lane * R * row_bytes, tm, rfull + s, 0, 0, chunk0,
                    b0.row / 8, z);
      if (isK && c0.j == 0 && lane == 0) {
        // a new item: its Q tiles (after the K tile, which does not wait for
        // the previous item's last QK), and an L2 prefetch of the Q tiles of
        // the item after it
        load_q(c0);
        const int inext = my_item(c0.k + 1);
        if (inext < T) {
          const Item nx = item_at(inext);
#pragma unroll
          for (int x = 0; x < NQ; ++x)
#pragma unroll
            for (int ch = 0; ch < D / 64; ++ch)
              tma_prefetch_l2_4d(&tmQ, ch * 64, 0, nx.g, nx.q0 + nx.p_begin + x * QP);
        }
      }
      ++t;
      if (++s == nring) {
        s = 0;
        ph ^= 1;
      }
      c0 = c1;
      h0 = h1;
      b0 = b1;
      if (h1) {
        h1 = next_tile(c1);
        if (h1) b1 = box_req(c1);
      }
    }
    if (lane == 0) {  // every issued copy must land before the CTA exits
      for (int u = (t > nring ? t - nring : 0); u < t; ++u)
        mbar_wait(rfull + (u % nring), (u / nring) & 1, a.err, dead);
      if (isK && c0.m >= 0)
#pragma unroll
        for (int x = 0; x < NQ; ++x) mbar_wait(q_full + x, c0.m & 1, a.err, dead);
    }
  } else if (warp == kMmaWarp) {
    // =============================== MMA issuer =============================
    {  // the whole warp runs the loop; one elected lane issues each tcgen05 op
      bool dead = false;
      // descriptor halves of the operand bases: K-major Q (atoms 1024 B
      // apart) and K (atoms kAtomStride apart), LBO 16 (unused); MN-major V:
      // LBO = the 1024 B chunk stride, atoms along the keys kAtomStride apart
      constexpr uint32_t kHi = tc::sw128_hi(1024);
      constexpr uint32_t kHiKV = tc::sw128_hi(S_::kAtomStride);
      constexpr uint32_t kHiV = tc::sw128_hi(S_::kVAtomStride);
      const uint32_t q_lo0 = tc::sw128_lo(sQ, 16);
      const uint32_t k_lo0 = tc::sw128_lo(smem_u32(smem + S_::kKOff), 16);
      const uint32_t v_lo0 = tc::sw128_lo(smem_u32(smem + S_::kVOff), 1024);
      // Every wait is followed by __syncwarp() (mbar_wait_converged): the
      // lanes leave a spin at different times, and the issue below runs
      // several times faster from a converged warp.
      // S_x(ta) = Q_x K(ta)^T into S buffer (x, ta % NS)
      auto qk_x = [&](const Cursor& c, int ta, int x) {
        const int sk = ta % NKS;
        if (x == 0) mbar_wait_converged(k_full + sk, (ta / NKS) & 1, a.err, dead);
        if (c.j == 0) mbar_wait_converged(q_full + x, c.m & 1, a.err, dead);
        tc::fence_after_sync();
        const uint32_t qlo = q_lo0 + x * (S_::kQBytes >> 4);
        const uint32_t klo = k_lo0 + sk * (S_::kSlotBytes >> 4);
        const int sb = x * NS + ta % NS;
        // K=16 steps: 32 B apart inside a 64-column chunk; chunks 16 KB
        // apart in Q and 1 KB apart in K
#pragma unroll
        for (int ch = 0; ch < D / 64; ++ch)
          tc::mma_ss_x4<2, 2>(tmem + sb * BN, qlo + ch * (16384 >> 4), kHi, klo + ch * (1024 >> 4),
                              kHiKV, kIdescS, ch > 0 ? 1u : 0u);
        tc::commit_w(s_full + sb);
        if (c.j == c.it.n - 1) tc::commit_w(q_empty + x);  // last use of this item's Q_x
        if (x == NQ - 1) tc::commit_w(k_empty + sk);       // last use of K(ta)
      };
      Cursor ca = cursor0();  // tile of the next QK (NS ahead of the PV)
      bool ha = next_tile(ca);
      int ta = 0;
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        if (ha) {
          for (int x = 0; x < NQ; ++x) qk_x(ca, ta, x);
          ++ta;
          ha = next_tile(ca);
        }
      }
      Cursor cv = cursor0();
      int t = 0;
      while (next_tile(cv)) {
        const int sv = t % NVS;
        for (int x = 0; x < NQ; ++x) {
          // O_x (+)= P_x(t) V(t): A = P in the TMEM columns of S buffer (x, t % NS)
          const int sb = x * NS + t % NS;
          if (x == 0) mbar_wait_converged(v_full + sv, (t / NVS) & 1, a.err, dead);
          const uint32_t blo = v_lo0 + sv * (S_::kVSlotBytes >> 4);
          // K=16 steps: 8 P columns and two 8-key atoms of V apart
          constexpr uint32_t kVStep = (2 * S_::kVAtomStride) >> 4;
          mbar_wait_converged(p_full + sb, (t / NS) & 1, a.err, dead);
          tc::fence_after_sync();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (BN == 128) {
              tc::mma_ts_x4<kVStep>(tmem + kOCol + x * DV, tmem + sb * BN + h * 32,
                                    blo + h * 4 * kVStep, kHiV, kIdescO,
                                    (cv.j > 0 || h > 0) ? 1u : 0u);
            } else {
#pragma unroll
              for (int ks = h * (BN / 32); ks < (h + 1) * (BN / 32); ++ks)
                tc::mma_ts_w(tmem + kOCol + x * DV, tmem + sb * BN + ks * 8, blo + ks * kVStep,
                             kHiV, kIdescO, (cv.j > 0 || ks > 0) ? 1u : 0u);
            }
          }
          // O_x is read back only at the item's end (and, with two S
          // buffers, before a rescale): commit o_done only then
          if (NS > 1 || cv.j == cv.it.n - 1) tc::commit_w(o_done + x);
          if (x == NQ - 1) tc::commit_w(v_empty + sv);  // last use of V(t)
          if (ha) qk_x(ca, ta, x);
        }
        if (ha) {
          ++ta;
          ha = next_tile(ca);
        }
        ++t;
      }
      // the stage-release arrivals must land before the CTA (and its smem)
      // goes away
      for (int u = (ta > NKS ? ta - NKS : 0); u < ta; ++u)
        mbar_wait(k_empty + (u % NKS), (u / NKS) & 1, a.err, dead);
      for (int u = (t > NVS ? t - NVS : 0); u < t; ++u)
        mbar_wait(v_empty + (u % NVS), (u / NVS) & 1, a.err, dead);
      if (cv.m >= 0)
        for (int x = 0; x < NQ; ++x) mbar_wait(q_empty + x, cv.m & 1, a.err, dead);
    }
  }
  } else {
    if (NQ == 2 && !HOSTED) asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
    // ======================== softmax warpgroups ============================
    bool dead = false;
    const int x = warp >> 2;  // which Q tile of the item
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t o_addr = lane_base + kOCol + x * DV;
    const float sl2 = a.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    int t = 0;
    int mi = 0;  // items with keys done by this warpgroup
    for (int kk_ = 0, i = my_item(0); i < T; ++kk_, i = my_item(kk_)) {
      const Item it = item_at(i);
      const int p = it.p_begin + x * QP + (r >> a.log2G);  // chunk row of this thread
      const bool row_valid = p < it.q_len;
      const int hh = r & (a.G - 1);
      // this item's DV columns of the output row
      __nv_bfloat16* orow =
          a.out + ((int64_t)(it.q0 + (row_valid ? p : 0)) * a.H_q + it.g * a.G + hh) * D +
          it.half * DV;
      if (it.n == 0) {  // no key for any row of the item: zero rows
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int v = 0; v < DV / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
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
        const int sb = x * NS + t % NS;
        const uint32_t s_addr = lane_base + sb * BN;
        mbar_wait(s_full + sb, (t / NS) & 1, a.err, dead);
        tc::fence_after_sync();
        uint32_t s[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          tc::ld_32x32b_x32(s_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
        tc::wait_ld();

        // mask only where a key of this tile falls outside a row's range
        const int key0 = (it.t_lo + j) * BN;
        const bool inside = key0 >= klo && key0 + BN <= khi;
        if (!__all_sync(0xffffffffu, inside)) {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int k = key0 + c;
            if (k < klo || k >= khi) s[c] = __float_as_uint(-INFINITY);
          }
        }
        float mxp[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          mxp[c] = fmaxf(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1]));
#pragma unroll
        for (int c = 16; c < BN; c += 2)
          mxp[(c >> 1) & 7] =
              max3f(mxp[(c >> 1) & 7], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
        const float mx = fmaxf(max3f(mxp[0], mxp[1], mxp[2]),
                               fmaxf(max3f(mxp[3], mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
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

        if (NS > 1 && j >= 1) {
          // With two S buffers nothing else orders PV(t-1) before this
          // point.  Wait for it on every tile: O may then be rescaled, and
          // the waits on o_done advance one phase at a time, which a parity
          // wait needs (at the epilogue a wait two phases ahead of the
          // barrier would return at once).  With one S buffer, S(t) itself
          // comes after PV(t-1).
          mbar_wait(o_done + x, (t - 1) & 1, a.err, dead);
          tc::fence_after_sync();
        }
        // P = 2^(s*scale_log2 - m) as bf16 pairs over the S columns, stored
        // in two halves of the keys; an eighth of the pairs on the FMA pipes
        const uint64_t negm = f2(-mu, -mu);
        uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = h * (BN / 4); c < (h + 1) * (BN / 4); ++c) {
            const uint64_t xx =
                f2_fma(f2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sl2x2, negm);
            uint64_t pp;
            if ((c & 7) == 7) {
              pp = poly_exp2x2(xx);
            } else {
              float x0, x1;
              f2_split(xx, x0, x1);
              pp = f2(fast_exp2(x0), fast_exp2(x1));
            }
            sum2[c & 3] = (c < 4) ? pp : f2_add(sum2[c & 3], pp);
            float p0, p1;
            f2_split(pp, p0, p1);
            s[c] = pack_bf16(p0, p1);  // P pair c over the consumed S column c
          }
          if (BN == 128)
            tc::st_32x32b_x32(s_addr + h * 32,
                              *reinterpret_cast<const uint32_t(*)[32]>(&s[h * 32]));
          else
            (BN == 64) ? tc::st_32x32b_x16(s_addr + h * 16, &s[h * 16])
                       : tc::st_32x32b_x8(s_addr + h * 8, &s[h * 8]);
          if (h == 0) {
            // O must be rescaled before the first half's PV; done here, once
            // the first half of the S row is dead, to keep registers free
            if (j >= 1 && __any_sync(0xffffffffu, resc)) {  // O *= alpha (warp-collective)
              const uint64_t al2 = f2(alpha, alpha);
              // rare (the running max grew by more than 2^8): kept rolled,
              // so that the tile loop's code stays small
#pragma unroll 1
              for (int c = 0; c < DV / 32; ++c) {
                uint32_t o[32];
                tc::ld_32x32b_x32(o_addr + c * 32, o);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  float o0, o1;
                  f2_split(f2_mul(f2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), al2),
                           o0, o1);
                  o[2 * e] = __float_as_uint(o0);
                  o[2 * e + 1] = __float_as_uint(o1);
                }
                tc::st_32x32b_x32(o_addr + c * 32, o);
              }
            }
          }
        }
        tc::wait_st();
        tc::fence_before_sync();
        // the whole warpgroup's P (and O) stores are done: one arrive
        named_bar_sync(1 + x, 128);
        if (r == 0) mbar_arrive(p_full + sb);
        float l0, l1;
        f2_split(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), l0, l1);
        l += l0 + l1;
      }
      // epilogue: O / l -> bf16 rows (after the item's last PV).  o_done
      // completes once per tile with two S buffers, once per item with one.
      mbar_wait(o_done + x, (NS > 1 ? (t - 1) : mi) & 1, a.err, dead);
      ++mi;
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
#if PKV_VAR_EPI_BATCH
      // two 32-column loads per wait; each 32 columns leave as two 32-byte
      // (or four 16-byte) stores of the thread's row
      static_assert((DV / 32) % 2 == 0, "pairs of 32-column chunks");
#pragma unroll
      for (int c = 0; c < DV / 32; c += 2) {
        uint32_t o[2][32];
        tc::ld_32x32b_x32(o_addr + c * 32, o[0]);
        tc::ld_32x32b_x32(o_addr + (c + 1) * 32, o[1]);
        tc::wait_ld();
        if (row_valid) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16(__uint_as_float(o[e][2 * i]) * inv,
                                __uint_as_float(o[e][2 * i + 1]) * inv);
            uint32_t* dst = reinterpret_cast<uint32_t*>(orow + (c + e) * 32);
            if (a.out_v8) {
#pragma unroll
              for (int h = 0; h < 2; ++h) st_global_v8(dst + 8 * h, pk + 8 * h);
            } else {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                reinterpret_cast<uint4*>(dst)[v] =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        }
      }
#else
      uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
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
#endif
      tc::fence_before_sync();
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (HOSTED) {
    // the shared memory is reused by the next phase: retire the barriers
    for (int i = tid; i < S_::kNumBars; i += NT) mbar_inval(bars + i);
    __syncthreads();
  }
}

}  // namespace pkv
