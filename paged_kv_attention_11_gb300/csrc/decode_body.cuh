// paged_attn_decode: one query per sequence over its paged K/V prefix.
//
// Semantics: scripts/benchmarks commit log, "Why this works" (decode reads
// the pool through the page table; the new token is written first, so the
// query at position len-1 sees keys 0..len-1) and the Gemma-4 sliding-window
// commit (key allowed iff q_pos - k_pos < window).
//
// Design (GB300):
//  * Work item = a (sequence, kv head) "segment" of 16-key tiles, or a chunk
//    of one: a segment longer than half of a CTA's fair share of the batch
//    is cut into equal chunks (unless the longest segment is within a
//    merge's cost of that length).  With HP = 2 (head_dim 128, an even
//    kv-head count, GQA group <= 4) a segment covers two kv heads of the
//    sequence: one TMA box per tile spans both heads' slice of a page.  One
//    persistent CTA per SM takes items from a device-side queue (an atomic
//    counter in the workspace) in longest-first order, so the SMs finish
//    together whatever the length mix, and only the few long segments need
//    a merge.
//  * Producer warp: grabs the next item, writes a record (sequence, head,
//    tiles, ...) and the item's query rows into a 4-deep record ring in
//    shared memory, then streams the item's K and V tiles: page ids from
//    the block table (32 per coalesced load), one TMA box per 16-key K or V
//    tile (5-D page view, 128-byte swizzle) into a deep NSTAGE ring, each
//    tile as soon as its stage is free.  The fused append (APPEND) writes
//    the sequence's newest K/V row before the copies of the tile that
//    holds it.
//  * NW consumer warps: take the tiles of each item round-robin (with two
//    heads per item, each warp of a pair takes one head of the pair's
//    tiles).  Per tile a warp computes S^T = K Q^T (16 keys x 8 heads, GQA
//    group padded to 8) with mma.sync, does the online softmax (exp2, warp
//    shuffles), transposes P in registers with movmatrix and accumulates
//    O^T = V^T P^T with mma.sync.  At the end of an item it hands its
//    (m, l, O) state to the epilogue warp through a double buffer and goes
//    straight on: no CTA-wide barrier in the stream.
//  * Epilogue warp: combines the consumer states of an item (log-sum-exp
//    weights); a whole segment is written as the bf16 output, a chunk as a
//    partial (o, lse) in the workspace.  The CTA that delivers the last
//    chunk of a segment (per-segment arrival counter) posts it to a merge
//    queue; CTAs that have run out of items merge the posted segments with
//    all their warps.  The last CTA to find the queue empty resets it.
//  * K/V bytes are read from HBM exactly once.  Launched with programmatic
//    dependent launch: the prologue overlaps the previous kernel in the
//    stream; griddepcontrol.wait precedes every read of the inputs.
#pragma once

#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tile16.cuh"

namespace pkv {

constexpr int kNRec = 4;   // piece records in flight
constexpr int kEpiScratch = 10 * kGP;  // epilogue weights: [NW][G] per warp, then the join's two
// Shortest chunk a segment is cut into (tiles).  Small batches (a few long
// windowed segments) then still spread over every SM instead of one segment
// per CTA; large batches cut at half a CTA's share, far above this floor.
#ifndef PKV_DEC_MIN_CHUNK_KB
#define PKV_DEC_MIN_CHUNK_KB 0
#endif
constexpr int kMinChunkTiles = 16;
// and at least this many bytes of K+V per chunk (0: no byte floor)
constexpr int kMinChunkBytes = PKV_DEC_MIN_CHUNK_KB * 1024;
// What a merge costs, as bytes one CTA would stream in the same time (~8 us
// at ~60 GB/s per SM, measured on the sliding-window step; the merge code
// runs once per CTA, so its instructions come cold from memory).
#ifndef PKV_DEC_MERGE_COST_KB
#define PKV_DEC_MERGE_COST_KB 480
#endif
constexpr int kMergeCostBytes = PKV_DEC_MERGE_COST_KB * 1024;
constexpr int kMaxSortSeq = 512;  // longest-first queue order up to this batch
// Batches up to this size keep each sequence's clamped length in shared
// memory, so the producer maps a queue index to its item without a global
// load; larger ones re-read seq_lens.
constexpr int kLenCacheSeq = 1024;

// a compile-time int carried by value (for generic lambdas)
template <int N>
struct IntC {
  static constexpr int value = N;
};

struct DecodeArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t max_blocks;
  int32_t batch;
  int32_t H_q, H_kv, G, P;
  int64_t num_pages;
  int32_t window;
  float scale_log2;
  int32_t* seg_count;   // [batch * H_kv] arrival counters, zero between calls
  int32_t* merge_jobs;  // [batch * H_kv] completed chunked segments (+1), zero between calls
  int32_t* queue;       // [8]: next item, CTAs done with items; next merge job, jobs
                        // posted, CTAs done merging; zero between calls
  float* part_lse;     // [(S + N) * G]
  float* part_o;       // [(S + N) * G * D]
  // shared-prefix (cascade) decode: null prefix_lens = plain decode.  A
  // sequence of group b / group_size whose length exceeds the group's shared
  // prefix attends only its suffix here, and its result is merged with the
  // prefix pass's partial (pre_o, pre_lse at row b * H_q + head).
  const int32_t* prefix_lens;
  int32_t group_size;
  const float* pre_o;
  const float* pre_lse;
  // CTAs that run the decode body (the last of them to find the queue empty
  // resets it), and the CTA count a segment's fair share is taken over
  int32_t cta_count;
  int32_t share_ctas;
  // fused append (null k_new: none): row b of k_new / v_new [batch, H_kv, D]
  // is sequence b's newest token, written to position seq_lens[b] - 1 of
  // its pages (k_pool / v_pool) before that tile is read
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_pool;
  uint4* v_pool;
  int32_t* err;
};

// Keys [lo, L) of sequence b are attended here; returns the tile range and
// whether a prefix partial covers keys [0, lo).
// The attended keys [lo, len) of sequence b of (clamped) length len and its
// 16-key tiles [t_lo, t_hi): the window, or the shared prefix of a cascade
// (pfx = 1: a prefix partial joins the merge).
__device__ __forceinline__ void extent_of_len(const DecodeArgs& a, int b, int len, int& lo,
                                              int& t_lo, int& t_hi, int* pfx) {
  const int cap = a.max_blocks * a.P;
  lo = (a.window > 0 && len > a.window) ? len - a.window : 0;
  int has_pfx = 0;
  if (a.prefix_lens != nullptr) {
    const int pl = shared_prefix_len(a.prefix_lens, b / a.group_size, a.P, cap);
    if (pl > 0 && len > pl) {
      lo = pl;
      has_pfx = 1;
    }
  }
  if (pfx) *pfx = has_pfx;
  t_lo = lo / kTile;
  t_hi = (len + kTile - 1) / kTile;
}

// Length of sequence b from seq_lens, clamped to the block table (flag:
// raise PKV_DEVERR_LEN for an out-of-range length), and its extent.
__device__ __forceinline__ void seq_extent(const DecodeArgs& a, int b, int& L, int& lo,
                                           int& t_lo, int& t_hi, bool flag, int* pfx = nullptr) {
  int len = __ldg(a.seq_lens + b);
  const int cap = a.max_blocks * a.P;
  if (len < 0 || len > cap) {
    if (flag) raise_err(a.err, PKV_DEVERR_LEN);
    len = len < 0 ? 0 : cap;
  }
  L = len;
  extent_of_len(a, b, len, lo, t_lo, t_hi, pfx);
}

// A piece as the producer hands it to the consumers and the epilogue.
struct PieceRec {
  int b, g;          // sequence, kv head
  int first_tile;    // first 16-key tile (absolute, within the sequence)
  int n;             // tiles in the item; -1 terminates the stream
  int L, lo;         // attended keys [lo, L)
  int nch;           // chunks of the segment (1: the item is the whole segment)
  int slot0;         // partial slot of chunk 0 of the segment
  int chunk;         // this item's chunk
  int pfx;           // 1: a prefix partial joins the merge (cascade)
};

// Head dims of 512 and more keep the query rows in shared memory (read with
// ldmatrix per tile) instead of registers, which then hold only O.
template <int D>
struct DecodeLayout {
  static constexpr bool kQSmem = D >= 512;
  // query rows in a record slot: kQSmem: kGP rows padded by 16 bytes (rows
  // G..kGP-1 zero), so that the 8 rows of an ldmatrix hit distinct banks
  static constexpr int kQRowBytes = kQSmem ? D * 2 + 16 : D * 2;
};

// Shared-memory plan (byte offsets from the 1024-aligned base); depends on
// the runtime GQA group and batch.  HP: kv heads per work item (a stage
// holds the item's HP heads of one 16-key tile, K then V).
template <int D, int NW, int NSTAGE, int HP = 1>
struct DecodePlan {
  using Lay = DecodeLayout<D>;
  static constexpr int kTileBytes = kTile * D * 2;      // one K (or V) tile of one head
  static constexpr int kStageBytes = 2 * HP * kTileBytes;  // K + V
  static constexpr int kCombStride = D + 4;             // padded row (floats)
  // consumer states reach the epilogue through two combine buffers, or one
  // where the buffer is large (head_dim 512, or 8 consumer warps)
  static constexpr int kNComb = (Lay::kQSmem || NW >= 8) ? 1 : 2;
  int rec, qbuf, qslot, comb, ml, bars, ok, misc, scan, cum, total;
  __host__ __device__ DecodePlan(int G, int batch) {
    int o = NSTAGE * kStageBytes;
    rec = o;   o += kNRec * (int)sizeof(PieceRec);
    qslot = (Lay::kQSmem ? kGP : G * HP) * Lay::kQRowBytes;
    qbuf = o;  o += kNRec * qslot;
    comb = o;  o += kNComb * NW * G * kCombStride * 4;
    ml = o;    o += kNComb * NW * G * 2 * 4;
    bars = o;  o += (2 * NSTAGE + 2 * kNRec + 2 * kNComb) * 8;
    ok = o;    o += NSTAGE * 4;
    misc = o;  o += 2 * kGP * 4 + 16 + kEpiScratch * 4;
    scan = o;  o += (NW + 2) * 4 + 8 + 16 + (NW + 2) * 4;
    // natural prefix, sorted prefix, order; lengths up to kLenCacheSeq sequences
    cum = o;   o += (batch + 1) * 4 * (batch <= kLenCacheSeq ? 4 : 3);
    total = 1024 + o;
  }
};

// The decode work of one CTA: (NW + 2) warps, threads 0 .. (NW+2)*32-1 of
// the block.  SUBSET: the block has more threads (the mixed-step kernel
// hosts this body on part of its warps), so the body synchronises on a
// named barrier of its own threads instead of the whole block.  `cta` is
// this CTA's index among the a.cta_count CTAs that run the body; smem is the
// 1024-aligned base of the dynamic shared memory.  APPEND: the fused append
// of paged_attn_decode_append (a.k_new set); compiled out otherwise.
// HP: kv heads per work item.  With HP = 2 an item is (sequence, pair of kv
// heads, chunk): one TMA box carries both heads' 16-key slice of a page
// (half the boxes per byte), the item's 2G query rows are handled as one
// group ("virtual head" g of H_kv / 2), and consumer warp w takes head
// w % 2 of the stages of its pair w / 2.  The host requires H_kv % HP == 0
// and HP * G <= 8.
template <int D, int NW, int NSTAGE, bool SUBSET, bool APPEND = false, int HP = 1>
__device__ __forceinline__ void decode_cta(const DecodeArgs& a, const CUtensorMap& tmK,
                                           const CUtensorMap& tmV, uint8_t* smem, int cta) {
  static_assert(HP == 1 || HP == 2, "one or two kv heads per item");
  static_assert(NW % HP == 0, "whole warp pairs");
  constexpr int NWH = NW / HP;  // consumer warps per head
  static_assert(NSTAGE % NWH == 0, "each stage must always feed the same warps");
  static_assert(D % 64 == 0, "head_dim must be a multiple of 64");
  static_assert(HP == 1 || !DecodeLayout<D>::kQSmem, "query rows in registers");
  using P_ = DecodePlan<D, NW, NSTAGE, HP>;
  using Lay = DecodeLayout<D>;
  constexpr bool QS = Lay::kQSmem;
  constexpr int NCB = P_::kNComb;
  constexpr int NT = (NW + 2) * 32;
  constexpr int KS = D / 16;  // mma k-steps for QK, m-tiles for PV
  constexpr int CS = P_::kCombStride;
  constexpr int kIssueLanes = NSTAGE < 16 ? NSTAGE : 16;  // producer lanes testing stages
  static_assert(kIssueLanes < 32, "a run of free stages ends inside the warp");
  const int G = a.G;        // query heads per kv head
  const int GV = G * HP;    // query rows per item
  const int HV = a.H_kv / HP;  // items per (sequence, chunk)
  const P_ plan(G, a.batch);

  auto block_sync = [&]() {
    if (SUBSET) named_bar_sync(1, NT);
    else __syncthreads();
  };
  PieceRec* recs = reinterpret_cast<PieceRec*>(smem + plan.rec);
  uint8_t* qbuf = smem + plan.qbuf;
  float* comb_o = reinterpret_cast<float*>(smem + plan.comb);   // [2][NW][G][CS]
  float* comb_ml = reinterpret_cast<float*>(smem + plan.ml);    // [2][NW][G][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + NSTAGE;
  uint64_t* rec_full = empty + NSTAGE;
  uint64_t* rec_empty = rec_full + kNRec;
  uint64_t* comb_full = rec_empty + kNRec;  // [NCB]
  uint64_t* comb_empty = comb_full + NCB;   // [NCB]
  int* stage_ok = reinterpret_cast<int*>(smem + plan.ok);
  float* merge_m = reinterpret_cast<float*>(smem + plan.misc);
  float* merge_inv = merge_m + kGP;
  float* epi_w = merge_inv + kGP + 4;  // [kEpiScratch]
  int* scan_tmp = reinterpret_cast<int*>(smem + plan.scan);
  int* s_misc = scan_tmp + NW + 4;                              // [4]
  int* s_nat = reinterpret_cast<int*>(smem + plan.cum);         // [B+1] items before b
  int* s_sp = s_nat + (a.batch + 1);                            // [B+1] sorted prefix
  int* s_order = s_sp + (a.batch + 1);                          // [B] sequences, longest first
  int* s_len = a.batch <= kLenCacheSeq ? s_order + (a.batch + 1) : nullptr;  // [B] lengths

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int B = a.batch;

  // one barrier per thread (the block has more threads than barriers)
  static_assert(2 * NSTAGE + 2 * kNRec + 2 * NCB <= NT, "barrier init");
  {
    const int i = tid;
    if (i < NSTAGE) {
      mbar_init(full + i, 1);
    } else if (i < 2 * NSTAGE) {
      mbar_init(full + i, HP);  // empty[i - NSTAGE]: the stage's consumer warps
    } else if (i < 2 * NSTAGE + kNRec) {
      mbar_init(rec_full + (i - 2 * NSTAGE), 32);
    } else if (i < 2 * NSTAGE + 2 * kNRec) {
      mbar_init(rec_full + (i - 2 * NSTAGE), NW * 32 + 32);  // rec_empty
    } else if (i < 2 * NSTAGE + 2 * kNRec + NCB) {
      mbar_init(comb_full + (i - 2 * NSTAGE - 2 * kNRec), NW * 32);
    } else if (i < 2 * NSTAGE + 2 * kNRec + 2 * NCB) {
      mbar_init(comb_full + (i - 2 * NSTAGE - 2 * kNRec), 32);  // comb_empty
    }
    if (i < 2 * NSTAGE + 2 * kNRec + 2 * NCB) fence_mbar_init();
  }
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (QS) {
    // rows G..kGP-1 of every query slot stay zero (the padded heads of the
    // mma N dimension); rows < G are written per item
    for (int i = tid; i < kNRec * (kGP - G) * (Lay::kQRowBytes / 16); i += NT) {
      const int per = (kGP - G) * (Lay::kQRowBytes / 16);
      const int sl = i / per, j = i - sl * per;
      reinterpret_cast<uint4*>(qbuf + sl * plan.qslot + G * Lay::kQRowBytes)[j] =
          make_uint4(0, 0, 0, 0);
    }
  }
  pdl_wait();  // inputs may come from the previous kernel in the stream
  // the producer's first queue grab is issued now; its latency hides behind
  // the prologue
  int first_grab = 0;
  if (warp == NW && lane == 0) first_grab = atomicAdd(a.queue, 1);
  {
    // the query rows and block tables, spread over the grid, into L2: the
    // producers' first items then find them there
    const int64_t qlines = ((int64_t)B * a.H_q * D * 2 + 127) / 128;
    const int64_t blines = ((int64_t)B * a.max_blocks * 4 + 127) / 128;
    const char* qp = reinterpret_cast<const char*>(a.q);
    const char* bp = reinterpret_cast<const char*>(a.block_table);
    for (int64_t l = (int64_t)cta * NT + tid; l < qlines + blines;
         l += (int64_t)a.cta_count * NT) {
      const char* p = l < qlines ? qp + l * 128 : bp + (l - qlines) * 128;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
  }

  // ---- work items (every CTA computes the same list, in smem) ----
  // tiles of sequence b: t_b; units W = sum t_b * H_kv; a segment longer
  // than S_max = max(kMinChunkTiles, W / (2N)) tiles is cut into nch_b
  // equal chunks -- unless the longest segment is within the cost of a
  // merge of S_max (kMergeCostBytes of streaming), where cutting would not
  // end the call sooner: then nothing is cut.
  {
    int local = 0, lmax = 0;
    for (int b = tid; b < B; b += NT) {
      int L, lo, tl, th;
      seq_extent(a, b, L, lo, tl, th, cta == 0);
      const int t = th - tl;
      s_nat[b] = t;  // tiles, for now
      if (s_len) s_len[b] = L;
      local += t;
      lmax = t > lmax ? t : lmax;
      // zero-length sequences have no work item: their zero rows are written here
      if (t == 0 && b % a.cta_count == cta) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + (int64_t)b * a.H_q * D);
        for (int i = 0; i < a.H_q * D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      local += __shfl_xor_sync(0xffffffffu, local, o);
      lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    }
    if (lane == 0) {
      scan_tmp[warp] = local;
      s_misc[4 + warp] = lmax;  // free until the prefix scan below
    }
    block_sync();
    if (tid == 0) {
      int64_t tot = 0;
      int tmax = 0;
      for (int w = 0; w < NT / 32; ++w) {
        tot += scan_tmp[w];
        tmax = max(tmax, s_misc[4 + w]);
      }
      // units: an item's tile (HP heads of 16 keys, K and V: 64 * D * HP bytes)
      const int64_t W = tot * HV;
      const int64_t half_share = (W + 2 * (int64_t)a.share_ctas - 1) / (2 * (int64_t)a.share_ctas);
      int64_t floor_tiles = kMinChunkTiles;
      if ((int64_t)kMinChunkBytes / (64 * D * HP) > floor_tiles)
        floor_tiles = kMinChunkBytes / (64 * D * HP);
      int64_t cut = half_share > floor_tiles ? half_share : floor_tiles;
      if ((int64_t)tmax <= cut + kMergeCostBytes / (64 * D * HP)) cut = tmax > 0 ? tmax : 1;
      s_misc[0] = (int)cut;  // S_max
      s_misc[1] = 0;  // sequences cut into more than one chunk
    }
    block_sync();
  }
  const int smax = s_misc[0];
  auto nch_of = [&](int t) { return (t + smax - 1) / smax; };
  // items per sequence (natural order) and chunk length (queue order key)
  {
    int chunked = 0;
    for (int b = tid; b < B; b += NT) {
      const int t = s_nat[b];
      const int nch = nch_of(t);
      s_nat[b] = nch * HV;
      s_sp[b] = t == 0 ? 0 : (t + nch - 1) / nch;
      chunked += nch > 1 ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) chunked += __shfl_xor_sync(0xffffffffu, chunked, o);
    if (lane == 0 && chunked) atomicAdd(s_misc + 1, chunked);
  }
  block_sync();
  // queue order: sequences by chunk length, longest first, ties by index
  // (up to kMaxSortSeq sequences; beyond, the natural order).  The rank of b
  // is the number of sequences that come before it.  Up to one sequence per
  // thread, each thread counts its own; beyond, the B x B comparisons run in
  // rows of 32 spread over all threads, ranks accumulate in s_order, and
  // every thread then scatters its sequences to their ranks.
  if (B <= NT) {
    // one thread per sequence: its rank is the number of keys ahead of it
    if (tid < B) {
      const int kb = s_sp[tid];
      int r = 0;
#pragma unroll 8
      for (int c = 0; c < B; ++c) {
        const int kc = s_sp[c];
        r += (kc > kb || (kc == kb && c < tid)) ? 1 : 0;
      }
      s_order[r] = tid;
    }
  } else if (B <= kMaxSortSeq) {
    for (int b = tid; b < B; b += NT) s_order[b] = 0;
    block_sync();
    const int nc = (B + 31) / 32;
    for (int u = tid; u < B * nc; u += NT) {
      const int b = u / nc, c0 = (u - b * nc) * 32;
      const int kb = s_sp[b];
      const int c1 = min(B, c0 + 32);
      int r = 0;
      for (int c = c0; c < c1; ++c) {
        const int kc = s_sp[c];
        r += (kc > kb || (kc == kb && c < b)) ? 1 : 0;
      }
      if (r) atomicAdd(s_order + b, r);
    }
    block_sync();
    int rk[(kMaxSortSeq + NT - 1) / NT];
#pragma unroll
    for (int k = 0; k < (kMaxSortSeq + NT - 1) / NT; ++k) {
      const int b = tid + k * NT;
      rk[k] = b < B ? s_order[b] : 0;
    }
    block_sync();
#pragma unroll
    for (int k = 0; k < (kMaxSortSeq + NT - 1) / NT; ++k) {
      const int b = tid + k * NT;
      if (b < B) s_order[rk[k]] = b;
    }
  } else {
    for (int b = tid; b < B; b += NT) s_order[b] = b;
  }
  block_sync();
  for (int k = tid; k < B; k += NT) s_sp[k] = s_nat[s_order[k]];  // items, queue order
  // both exclusive prefixes in one pass: each thread scans a contiguous run
  {
    const int per = (B + NT - 1) / NT;
    const int i0 = tid * per;
    block_sync();
    int l1 = 0, l2 = 0;
    for (int i = i0; i < i0 + per && i < B; ++i) {
      l1 += s_nat[i];
      l2 += s_sp[i];
    }
    int c1 = l1, c2 = l2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v1 = __shfl_up_sync(0xffffffffu, c1, o);
      const int v2 = __shfl_up_sync(0xffffffffu, c2, o);
      if (lane >= o) {
        c1 += v1;
        c2 += v2;
      }
    }
    if (lane == 31) {
      scan_tmp[warp] = c1;
      s_misc[4 + warp] = c2;
    }
    block_sync();
    int r1 = c1 - l1, r2 = c2 - l2;
    for (int w = 0; w < warp; ++w) {
      r1 += scan_tmp[w];
      r2 += s_misc[4 + w];
    }
    for (int i = i0; i < i0 + per && i < B; ++i) {
      const int v1 = s_nat[i], v2 = s_sp[i];
      s_nat[i] = r1;
      s_sp[i] = r2;
      r1 += v1;
      r2 += v2;
    }
    if (tid == NT - 1) {
      s_nat[B] = r1;
      s_sp[B] = r2;
    }
    block_sync();
  }
  pdl_launch_dependents();
  const int T = s_nat[B];  // work items in the batch

  if (warp == NW) {
    // ============================ producer warp ============================
    // Items come from the queue one at a time; the next item's query rows
    // and first 32 page ids are loaded into registers before the current
    // item is streamed, so no global-memory latency sits between items.
    constexpr int QV = D / 32;  // query vectors per lane for a group of <= 8 heads
    bool dead = false;
    const int qvec = GV * D / 8;  // 16-byte vectors of the item's query rows
    struct Item {
      bool more;
      int b, g, L, lo, first_tile, n, nch, slot0, chunk, pfx;
    };
    auto grab = [&]() -> int {
      int i = 0;
      if (lane == 0) i = atomicAdd(a.queue, 1);
      return __shfl_sync(0xffffffffu, i, 0);
    };
    // queue index -> item (sorted sequences; heads; chunks)
    auto item_at = [&](int i) -> Item {
      Item it;
      it.more = i < T;
      it.b = it.g = it.L = it.lo = it.first_tile = it.nch = it.slot0 = it.chunk = it.pfx = 0;
      it.n = -1;
      if (!it.more) return it;
      int lo = 0, hi = B;  // s_sp[lo] <= i < s_sp[lo+1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_sp[mid] <= i) lo = mid; else hi = mid;
      }
      const int b = s_order[lo];
      const int j = i - s_sp[lo];
      int L, klo, t_lo, t_hi, pfx;
      if (s_len) {
        L = s_len[b];
        extent_of_len(a, b, L, klo, t_lo, t_hi, &pfx);
      } else {
        seq_extent(a, b, L, klo, t_lo, t_hi, false, &pfx);
      }
      const int t = t_hi - t_lo;
      const int nch = nch_of(t);
      const int csz = (t + nch - 1) / nch;
      const int g = j / nch, chunk = j - (j / nch) * nch;
      it.b = b;
      it.g = g;
      it.L = L;
      it.lo = klo;
      it.first_tile = t_lo + chunk * csz;
      it.n = min(csz, t - chunk * csz);
      it.nch = nch;
      it.slot0 = s_nat[b] + g * nch;
      it.chunk = chunk;
      it.pfx = pfx;
      return it;
    };
    // fused append: the item whose tiles hold key L-1 writes the new K/V
    // rows of its (sequence, kv heads) first.  Lane l holds 16-byte vector l
    // of the HP K rows then of the HP V rows (kNV per lane).
    constexpr int kRowVec = D / 8;                      // vectors of one row
    constexpr int kNV = (2 * HP * kRowVec + 31) / 32;   // per lane
    uint4 nrow[kNV];
    int npage = -1;  // page of key L-1 (-1: nothing to write)
    auto prefetch_new = [&](const Item& p) {
      npage = -1;
      if (!APPEND || !p.more || p.n <= 0 || p.L <= 0) return;
      const int last = (p.L - 1) / kTile;
      if (last < p.first_tile || last >= p.first_tile + p.n) return;
      npage = __ldg(a.block_table + (int64_t)p.b * a.max_blocks + (p.L - 1) / a.P);
      const int64_t row = (int64_t)p.b * a.H_kv + HP * p.g;  // the item's first head
#pragma unroll
      for (int i = 0; i < kNV; ++i) {
        const int v = lane + 32 * i;
        if (v < HP * kRowVec) nrow[i] = __ldg(a.k_new + row * kRowVec + v);
        else if (v < 2 * HP * kRowVec)
          nrow[i] = __ldg(a.v_new + row * kRowVec + (v - HP * kRowVec));
      }
    };
    auto write_new = [&](const Item& p) {
      if (!APPEND || npage < 0) return;
      if ((int64_t)npage >= a.num_pages) {
        if (lane == 0) raise_err(a.err, PKV_DEVERR_PAGE);
        return;
      }
      // head h's row sits P * kRowVec vectors after head h - 1's
      const int64_t dst =
          (((int64_t)npage * a.H_kv + HP * p.g) * a.P + (p.L - 1) % a.P) * kRowVec;
#pragma unroll
      for (int i = 0; i < kNV; ++i) {
        const int v = lane + 32 * i;
        const int w = v < HP * kRowVec ? v : v - HP * kRowVec;  // vector in the K or V rows
        const int64_t off = dst + (int64_t)(w / kRowVec) * a.P * kRowVec + (w % kRowVec);
        if (v < HP * kRowVec) a.k_pool[off] = nrow[i];
        else if (v < 2 * HP * kRowVec) a.v_pool[off] = nrow[i];
      }
      // the rows must be seen by the TMA (async proxy) copies of this item
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
    };
    auto prefetch = [&](const Item& p, uint4 (&qr)[QV], int& pages) {
      pages = -1;
      prefetch_new(p);
      if (!p.more) return;
      // page ids first: the first TMA copies need them, the query rows only
      // the record
      if (lane < p.n)
        pages = __ldg(a.block_table + (int64_t)p.b * a.max_blocks +
                      ((p.first_tile + lane) * kTile) / a.P);
      const uint4* qsrc =
          reinterpret_cast<const uint4*>(a.q + ((int64_t)p.b * a.H_q + p.g * GV) * D);
#pragma unroll
      for (int i = 0; i < QV; ++i) {
        const int v = lane + 32 * i;
        if (v < qvec) qr[i] = __ldg(qsrc + v);
      }
    };

    Item cur = item_at(__shfl_sync(0xffffffffu, first_grab, 0));
    uint4 qcur[QV];
    int pcur;
    prefetch(cur, qcur, pcur);
    int it = 0;  // CTA-wide tile counter
    int k = 0;   // item counter
    while (true) {
      // ---- the item record and its query rows, to the consumers and the
      //      epilogue.  It goes out right after the item's first issue
      //      instruction (up to 16 tiles), and always before a wait on a
      //      busy stage (the item's own consumers may be the ones to free
      //      it), so a CTA's first copies leave without waiting for the
      //      query rows. ----
      bool published = false;
      auto publish = [&]() {
        const int slot = k % kNRec;
        if (k >= kNRec) mbar_wait(rec_empty + slot, ((k / kNRec) - 1) & 1, a.err, dead);
        if (cur.more) {
          uint4* qdst = reinterpret_cast<uint4*>(qbuf + slot * plan.qslot);
#pragma unroll
          for (int i = 0; i < QV; ++i) {
            const int v = lane + 32 * i;
            if (v < qvec) {
              if (QS) {  // padded rows: vector v of head v / (D/8)
                const int h = v / (D / 8);
                qdst[v + h] = qcur[i];
              } else {
                qdst[v] = qcur[i];
              }
            }
          }
        }
        if (lane == 0) {
          PieceRec& r = recs[slot];
          r.b = cur.b;
          r.g = cur.g;
          r.first_tile = cur.first_tile;
          r.n = cur.n;
          r.L = cur.L;
          r.lo = cur.lo;
          r.nch = cur.nch;
          r.slot0 = cur.slot0;
          r.chunk = cur.chunk;
          r.pfx = cur.pfx;
        }
        __syncwarp();
        mbar_arrive(rec_full + slot);  // all 32 lanes: each releases its own writes
        ++k;
        published = true;
      };
      if (!cur.more) {
        publish();
        break;
      }
      // ---- stream the item's tiles (after the fused append's row) ----
      write_new(cur);
      const int* bt = a.block_table + (int64_t)cur.b * a.max_blocks;
      const int n = cur.n;
      int page = pcur;
      for (int k0 = 0; k0 < n; k0 += 32) {
        int page_ahead = -1;  // page ids of the following 32 tiles
        if (k0 + 32 + lane < n)
          page_ahead = __ldg(bt + ((cur.first_tile + k0 + 32 + lane) * kTile) / a.P);
        const int cnt = min(32, n - k0);
        // Tiles go out in order, each as soon as its own stage is free:
        // lanes test the stages of the next kIssueLanes tiles (distinct
        // stages, so no test can see a phase two rounds old), and the run of
        // free stages from the first one is issued by one warp instruction.
        // When the first stage is still busy, lane 0 waits on it alone; the
        // consumers free stages in order, so it is the next to free.
        for (int j = 0; j < cnt;) {
          const int jl = j + lane;
          const int pg = __shfl_sync(0xffffffffu, page, jl & 31);
          const int itj = it + jl;
          const int s = itj % NSTAGE;
          const int r = itj / NSTAGE;
          const bool mine = lane < kIssueLanes && jl < cnt;
          const bool free_ = mine && (r == 0 || mbar_test_wait(empty + s, (r - 1) & 1));
          const uint32_t fm = __ballot_sync(0xffffffffu, free_);
          int run = __ffs(~fm) - 1;  // free stages in a row from tile j
          if (run == 0) {
            if (!published) publish();
            if (lane == 0) mbar_wait(empty + s, (r - 1) & 1, a.err, dead);
            __syncwarp();
            run = 1;
            if (__shfl_sync(0xffffffffu, (int)dead, 0)) dead = true;
          }
          if (lane < run) {
            const int key0 = (cur.first_tile + k0 + jl) * kTile;
            const bool ok = pg >= 0 && (int64_t)pg < a.num_pages;
            stage_ok[s] = ok ? 1 : 0;
            if (ok) {
              uint8_t* st = smem + s * P_::kStageBytes;
              mbar_arrive_expect_tx(full + s, P_::kStageBytes);
              const int row = key0 % a.P;
              const int z = pg * a.H_kv + HP * cur.g;
              // one box per tile: 16 keys x all D columns of one page and
              // the item's HP heads
              tma_load_5d(st, &tmK, full + s, 0, 0, 0, row / 8, z);
              tma_load_5d(st + HP * P_::kTileBytes, &tmV, full + s, 0, 0, 0, row / 8, z);
            } else {
              raise_err(a.err, PKV_DEVERR_PAGE);
              mbar_arrive(full + s);
            }
          }
          __syncwarp();
          j += run;
          // the consumers start on the first copies while the rest go out
          if (!published) publish();
        }
        it += cnt;
        page = page_ahead;
      }
      // ---- next item: grabbed only once this one is issued, so no CTA holds
      //      work in reserve at the end; the stage ring covers the latency ----
      cur = item_at(grab());
      prefetch(cur, qcur, pcur);
    }
    // queue exhausted for this CTA: the last CTA to get here resets it
    if (lane == 0) {
      __threadfence();
      const int done = atomicAdd(a.queue + 1, 1);
      if (done == a.cta_count - 1) {
        a.queue[0] = 0;
        a.queue[1] = 0;
      }
    }
    // drain: every issued load must land before the CTA may exit
    if (lane == 0) {
      const int first = it > NSTAGE ? it - NSTAGE : 0;
      for (int i = first; i < it; ++i)
        mbar_wait(full + (i % NSTAGE), (i / NSTAGE) & 1, a.err, dead);
    }
  } else if (warp < NW) {
    // ============================== consumer warps ==========================
    const int quad = lane >> 2;  // 0..7: key row (QK) / head (Q frag)
    const int qlan = lane & 3;   // 0..3: head pair (2*qlan, 2*qlan+1)
    const int hd = warp % HP;    // the item's kv head this warp takes
    const int team = warp / HP;  // this warp's place among the head's warps
    bool dead = false;
    int it_base = 0;
    for (int k = 0;; ++k) {
      const int slot = k % kNRec;
      if (!mbar_wait(rec_full + slot, (k / kNRec) & 1, a.err, dead)) break;
      const PieceRec rec = recs[slot];
      // Q^T fragments (B operand of S^T = K Q^T): head = quad, dims by qlan.
      // Registers (head dims up to 256), or per tile from shared memory.
      uint32_t qb[QS ? 1 : KS][2];
      if (!QS) {
        const bool hv = rec.n >= 0 && quad < G;
        const uint8_t* qrow = qbuf + slot * plan.qslot + (hv ? hd * G + quad : 0) * D * 2;
#pragma unroll
        for (int ks = 0; ks < (QS ? 1 : KS); ++ks) {
          qb[ks][0] = hv ? *reinterpret_cast<const uint32_t*>(qrow + (ks * 16 + 2 * qlan) * 2)
                         : 0u;
          qb[ks][1] =
              hv ? *reinterpret_cast<const uint32_t*>(qrow + (ks * 16 + 8 + 2 * qlan) * 2) : 0u;
        }
        mbar_arrive(rec_empty + slot);  // record and query rows copied to registers
      }
      // ldmatrix row address of this lane in the smem query slot: row
      // lane % 8 (a head), 8 dims at (lane / 8) * 8 of each 32-dim step
      const uint32_t q_lane_addr = smem_u32(qbuf + slot * plan.qslot) +
                                   (lane & 7) * Lay::kQRowBytes + (lane >> 3) * 16;
      if (rec.n < 0) {
        if (QS) mbar_arrive(rec_empty + slot);
        break;
      }

      float o[KS][4];
#pragma unroll
      for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
      const int n = rec.n;
      // this warp takes the item's tiles kk = r, r+NWH, ...; r depends only
      // on where the item starts in the stage ring, and the epilogue
      // combines the warps in r order, so the result does not depend on the
      // CTA
      const int r0 = ((team - it_base) % NWH + NWH) % NWH;
      for (int kk = r0; kk < n; kk += NWH) {
        const int it = it_base + kk;
        const int s = it % NSTAGE;
        const bool landed = mbar_wait(full + s, (it / NSTAGE) & 1, a.err, dead);
        const bool ok = landed && stage_ok[s] != 0;
        // head hd's K tile, then (after the HP K tiles) its V tile
        const uint32_t stK = smem_u32(smem + s * P_::kStageBytes) + hd * P_::kTileBytes;
        const uint32_t stV = stK + HP * P_::kTileBytes;
        const int key0 = (rec.first_tile + kk) * kTile;

        // ---- S^T = K Q^T: 16 keys x 8 heads, two accumulation chains ----
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
          if (QS) {
            // two k-steps per ldmatrix of the query rows
#pragma unroll
            for (int ks = 0; ks < KS; ks += 2) {
              uint32_t b00, b01, b10, b11;
              ldsm_x4(q_lane_addr + ks * 32, b00, b01, b10, b11);
              uint32_t a0, a1, a2, a3;
              ldsm_x4(tile_addr<D>(stK, key, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
              mma_bf16_16816(sa, a0, a1, a2, a3, b00, b01);
              ldsm_x4(tile_addr<D>(stK, key, 2 * ks + 2 + (lane >> 4)), a0, a1, a2, a3);
              mma_bf16_16816(sb, a0, a1, a2, a3, b10, b11);
            }
          } else {
#pragma unroll
            for (int ks = 0; ks < (QS ? 1 : KS); ++ks) {
              const uint32_t addr = tile_addr<D>(stK, key, 2 * ks + (lane >> 4));
              uint32_t a0, a1, a2, a3;
              ldsm_x4(addr, a0, a1, a2, a3);
              if (ks & 1) mma_bf16_16816(sb, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
              else mma_bf16_16816(sa, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            }
          }
        }
        // rows: key0+quad (regs 0,1) and key0+quad+8 (regs 2,3); cols: heads 2*qlan, +1
        const int kA = key0 + quad, kB = kA + 8;
        const bool vA = ok && kA >= rec.lo && kA < rec.L;
        const bool vB = ok && kB >= rec.lo && kB < rec.L;
        const float x0A = vA ? (sa[0] + sb[0]) * a.scale_log2 : -INFINITY;
        const float x0B = vA ? (sa[1] + sb[1]) * a.scale_log2 : -INFINITY;
        const float x1A = vB ? (sa[2] + sb[2]) * a.scale_log2 : -INFINITY;
        const float x1B = vB ? (sa[3] + sb[3]) * a.scale_log2 : -INFINITY;
        float tA = fmaxf(x0A, x1A), tB = fmaxf(x0B, x1B);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, off));
          tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, off));
        }
        const float nA = fmaxf(mA, tA), nB = fmaxf(mB, tB);
        const float uA = nA == -INFINITY ? 0.f : nA;
        const float uB = nB == -INFINITY ? 0.f : nB;
        const float alA = exp2f(mA - uA), alB = exp2f(mB - uB);
        const float p0A = exp2f(x0A - uA), p0B = exp2f(x0B - uB);
        const float p1A = exp2f(x1A - uA), p1B = exp2f(x1B - uB);
        lA = lA * alA + p0A + p1A;
        lB = lB * alB + p0B + p1B;
        mA = nA;
        mB = nB;
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          o[i][0] *= alA;
          o[i][1] *= alB;
          o[i][2] *= alA;
          o[i][3] *= alB;
        }
        // P^T as the B operand: transpose the 8x8 (key x head) blocks in registers
        const uint32_t pb0 = movmatrix_t(pack_bf16(p0A, p0B));
        const uint32_t pb1 = movmatrix_t(pack_bf16(p1A, p1B));

        // ---- O^T += V^T P^T: D/16 m-tiles of 16 dims x 8 heads ----
        {
          const int j = lane >> 3;
          const int key = (lane & 7) + (j >> 1) * 8;
#pragma unroll
          for (int md = 0; md < KS; ++md) {
            const uint32_t addr = tile_addr<D>(stV, key, 2 * md + (j & 1));
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(addr, a0, a1, a2, a3);
            mma_bf16_16816(o[md], a0, a1, a2, a3, pb0, pb1);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);
      }
      it_base += n;
      if (QS) mbar_arrive(rec_empty + slot);  // done reading the query rows

      // ---- hand (m, l, O) of this warp to the epilogue warp ----
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        lA += __shfl_xor_sync(0xffffffffu, lA, off);
        lB += __shfl_xor_sync(0xffffffffu, lB, off);
      }
      const int cb = k % NCB;
      if (k >= NCB) mbar_wait(comb_empty + cb, ((k / NCB) - 1) & 1, a.err, dead);
      float* co = comb_o + ((cb * NW + hd * NWH + r0) * G) * CS;
      float* cml = comb_ml + ((cb * NW + hd * NWH + r0) * G) * 2;
      const int hA = 2 * qlan, hB = hA + 1;
#pragma unroll
      for (int md = 0; md < KS; ++md) {
        const int d = md * 16 + quad;
        if (hA < G) {
          co[hA * CS + d] = o[md][0];
          co[hA * CS + d + 8] = o[md][2];
        }
        if (hB < G) {
          co[hB * CS + d] = o[md][1];
          co[hB * CS + d + 8] = o[md][3];
        }
      }
      if (quad == 0) {
        if (hA < G) {
          cml[hA * 2] = mA;
          cml[hA * 2 + 1] = lA;
        }
        if (hB < G) {
          cml[hB * 2] = mB;
          cml[hB * 2 + 1] = lB;
        }
      }
      mbar_arrive(comb_full + cb);  // every lane releases its own writes
    }
  } else {
    // =============================== epilogue warp ==========================
    bool dead = false;
    for (int k = 0;; ++k) {
      const int slot = k % kNRec;
      if (!mbar_wait(rec_full + slot, (k / kNRec) & 1, a.err, dead)) break;
      const PieceRec rec = recs[slot];
      mbar_arrive(rec_empty + slot);
      if (rec.n < 0) break;
      const int cb = k % NCB;
      mbar_wait(comb_full + cb, (k / NCB) & 1, a.err, dead);
      const int b = rec.b, g = rec.g;
      // a segment in one piece is written here; so is one with a prefix
      // partial (cascade) whose suffix is one piece: the two are joined
      // inline, with the prefix partial's weight from its log-sum-exp
      const bool join_pfx = rec.nch == 1 && rec.pfx == 1;
      const bool whole = rec.nch == 1;
      const int64_t pre_row0 = (int64_t)b * a.H_q + g * GV;
      float* w_item = epi_w + NW * kGP;  // [kGP] weights of the joined outputs
      float* w_pfx = w_item + kGP;           // [kGP]
      const float* co = comb_o + (cb * NW * G) * CS;
      const float* cml = comb_ml + (cb * NW * G) * 2;
      const int64_t pslot = (int64_t)rec.slot0 + rec.chunk;
      // per query row h of the item (kv head h / G, its row h % G, held by
      // warps (h / G) * NWH + r): weight of each warp's state, 1/l,
      // log2-sum-exp
      float* wsc = epi_w;  // [NWH][GV] scratch
      // state of row h from its head's r-th warp: hbase(h) + r * G
      auto hbase = [&](int h) -> int {
        if (HP == 1) return h;
        return (h / G) * NWH * G + (h % G);
      };
      if (lane < GV) {
        const int h = lane;
        const int hb = hbase(h);
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < NWH; ++r) M = fmaxf(M, cml[(hb + r * G) * 2]);
        float lsum = 0.f;
#pragma unroll
        for (int r = 0; r < NWH; ++r) {
          const float sc = M == -INFINITY ? 0.f : exp2f(cml[(hb + r * G) * 2] - M);
          wsc[r * GV + h] = sc;
          lsum += sc * cml[(hb + r * G) * 2 + 1];
        }
        merge_m[h] = lsum > 0.f ? M + log2f(lsum) : -INFINITY;
        merge_inv[h] = lsum > 0.f ? 1.f / lsum : 0.f;
        if (join_pfx) {
          const float li = merge_m[h];
          const float lp = __ldcg(a.pre_lse + pre_row0 + h);
          const float m2 = fmaxf(li, lp);
          const float wi = li == -INFINITY ? 0.f : exp2f(li - m2);
          const float wp = lp == -INFINITY ? 0.f : exp2f(lp - m2);
          const float den = wi + wp;
          w_item[h] = den > 0.f ? wi / den : 0.f;
          w_pfx[h] = den > 0.f ? wp / den : 0.f;
        }
      }
      __syncwarp();
      // 4 slices per lane per pass; the prefix partial's loads (cascade)
      // are issued before any is used
      for (int j0 = lane; j0 < GV * (D / 4); j0 += 128) {
        float4 pv[4];
        if (join_pfx) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + 32 * u < GV * (D / 4) ? j0 + 32 * u : 0;
            const int h = j / (D / 4), d4 = j - h * (D / 4);
            pv[u] = __ldcg(reinterpret_cast<const float4*>(a.pre_o + (pre_row0 + h) * D) + d4);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + 32 * u;
          if (j >= GV * (D / 4)) break;
          const int h = j / (D / 4), d4 = j - h * (D / 4);
          const float* cor = co + hbase(h) * CS + d4 * 4;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int r = 0; r < NWH; ++r) {
            const float sc = wsc[r * GV + h];
            const float4 v = *reinterpret_cast<const float4*>(cor + r * G * CS);
            acc.x += sc * v.x;
            acc.y += sc * v.y;
            acc.z += sc * v.z;
            acc.w += sc * v.w;
          }
          const float inv = merge_inv[h];
          acc.x *= inv;
          acc.y *= inv;
          acc.z *= inv;
          acc.w *= inv;
          if (join_pfx) {
            const float wi = w_item[h], wp = w_pfx[h];
            acc.x = wi * acc.x + wp * pv[u].x;
            acc.y = wi * acc.y + wp * pv[u].y;
            acc.z = wi * acc.z + wp * pv[u].z;
            acc.w = wi * acc.w + wp * pv[u].w;
          }
          if (whole) {
            __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo2);
            pk.y = *reinterpret_cast<uint32_t*>(&hi2);
            *reinterpret_cast<uint2*>(a.out + ((int64_t)b * a.H_q + g * GV + h) * D + d4 * 4) =
                pk;
          } else {
            *reinterpret_cast<float4*>(a.part_o + (pslot * GV + h) * D + d4 * 4) = acc;
            if (d4 == 0) a.part_lse[pslot * GV + h] = merge_m[h];
          }
        }
      }
      __syncwarp();
      mbar_arrive(comb_empty + cb);  // the consumers may refill this buffer
      if (!whole) {
        // arrival counter: the CTA that delivers the last chunk of this
        // segment posts it to the merge queue (nobody waits here; the
        // counter is reset for the next call)
        const int64_t seg = (int64_t)b * HV + g;
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          const int old = atomicAdd(a.seg_count + seg, 1);
          if (old == rec.nch - 1) {
            a.seg_count[seg] = 0;
            __threadfence();  // every chunk's partial before the post
            const int j = atomicAdd(a.queue + 3, 1);
            st_volatile_i32(a.merge_jobs + j, (int)seg + 1);
          }
        }
        __syncwarp();
      }
    }
  }

  // ============================ merge phase ================================
  // Segments cut into chunks are merged by the CTAs that have run out of
  // items, with all their warps: a CTA takes the next posted segment (in
  // the order the segments completed), waits for its post if it is still
  // being computed elsewhere (every CTA of the grid is resident, so the
  // post comes), and combines the chunks' partials with their log-sum-exp
  // weights.  The stage ring is free scratch now: the producer has drained
  // every copy it issued.
  // segments with more than one chunk: each is posted exactly once (none:
  // the CTA ends here, touching no merge counter)
  const int n_jobs = s_misc[1] * HV;
  if (n_jobs > 0) {
    block_sync();
    volatile int* s_job = s_misc + 2;  // [2]: queue index, segment
    float* wts = reinterpret_cast<float*>(smem);  // [np * GV] weights, then [2][GV]
    bool mdead = false;
    while (true) {
      if (tid == 0) s_job[0] = atomicAdd(a.queue + 2, 1);
      block_sync();
      const int idx = s_job[0];
      if (idx >= n_jobs) break;
      if (tid == 0) {
        int v = ld_volatile_i32(a.merge_jobs + idx);
        if (v == 0 && !mdead) {
          const unsigned long long t0 = globaltimer();
          while ((v = ld_volatile_i32(a.merge_jobs + idx)) == 0) {
            __nanosleep(128);  // the posts are far apart; keep the L2 line quiet
            if (globaltimer() - t0 > kWaitTimeoutNs) {
              raise_err(a.err, PKV_DEVERR_TIMEOUT);
              mdead = true;
              break;
            }
          }
        }
        st_volatile_i32(a.merge_jobs + idx, 0);
        s_job[1] = v - 1;
        __threadfence();  // the chunks' partials after the post
      }
      block_sync();
      const int seg = s_job[1];
      if (seg < 0) break;
      const int b = seg / HV, g = seg - b * HV;
      const int nch = (s_nat[b + 1] - s_nat[b]) / HV;
      const int64_t slot0 = (int64_t)s_nat[b] + (int64_t)g * nch;
      int L, klo, t_lo, t_hi, pfx;
      if (s_len) {
        L = s_len[b];
        extent_of_len(a, b, L, klo, t_lo, t_hi, &pfx);
      } else {
        seq_extent(a, b, L, klo, t_lo, t_hi, false, &pfx);
      }
      // the segment's chunks, plus the prefix partial as chunk nch (cascade)
      const int np = nch + pfx;
      const int64_t row0 = (int64_t)b * a.H_q + g * GV;
      auto l_src = [&](int c, int h) -> const float* {
        return c < nch ? a.part_lse + (slot0 + c) * GV + h : a.pre_lse + row0 + h;
      };
      auto o_src = [&](int c, int h) -> const float* {
        return c < nch ? a.part_o + ((slot0 + c) * GV + h) * D : a.pre_o + (row0 + h) * D;
      };
      const int nl = np * GV;
      float* wm = wts + nl;  // [GV] max, [GV] 1 / sum
      for (int i = tid; i < nl; i += NT) wts[i] = __ldcg(l_src(i / GV, i % GV));
      block_sync();
      if (tid < GV) {  // per head: max and 1 / sum of the weights
        const int h = tid;
        float M = -INFINITY, sum = 0.f;
        for (int c = 0; c < np; ++c) M = fmaxf(M, wts[c * GV + h]);
        if (M != -INFINITY)
          for (int c = 0; c < np; ++c) sum += exp2f(wts[c * GV + h] - M);
        wm[h] = M;
        wm[GV + h] = sum > 0.f ? 1.f / sum : 0.f;
      }
      block_sync();
      for (int i = tid; i < nl; i += NT) {
        const int h = i % GV;
        const float M = wm[h];
        wts[i] = M == -INFINITY ? 0.f : exp2f(wts[i] - M) * wm[GV + h];
      }
      block_sync();
      // weighted sum of the chunks' outputs, 4 dims (a slice) per load; each
      // thread keeps kS slices x kMC chunks of loads in flight (two chunks,
      // the common split: twice the slices); every output sums its chunks
      // in chunk order
      auto wsum = [&](auto s_c, auto mc_c) {
        constexpr int kS = decltype(s_c)::value, kMC = decltype(mc_c)::value;
        constexpr int Q4 = D / 4;
        for (int j0 = tid; j0 < GV * Q4; j0 += NT * kS) {
          float4 acc[kS];
          int hh[kS], dd[kS];
#pragma unroll
          for (int u = 0; u < kS; ++u) {
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int j = j0 + NT * u < GV * Q4 ? j0 + NT * u : 0;
            hh[u] = j / Q4;
            dd[u] = j - hh[u] * Q4;
          }
          for (int c0 = 0; c0 < np; c0 += kMC) {
            float4 v[kS][kMC];
#pragma unroll
            for (int u = 0; u < kS; ++u)
#pragma unroll
              for (int cc = 0; cc < kMC; ++cc) {
                const int c = c0 + cc < np ? c0 + cc : np - 1;  // clamped: weight 0 below
                v[u][cc] = __ldcg(reinterpret_cast<const float4*>(o_src(c, hh[u])) + dd[u]);
              }
#pragma unroll
            for (int u = 0; u < kS; ++u)
#pragma unroll
              for (int cc = 0; cc < kMC; ++cc) {
                const float w = c0 + cc < np ? wts[(c0 + cc) * GV + hh[u]] : 0.f;
                acc[u].x += w * v[u][cc].x;
                acc[u].y += w * v[u][cc].y;
                acc[u].z += w * v[u][cc].z;
                acc[u].w += w * v[u][cc].w;
              }
          }
#pragma unroll
          for (int u = 0; u < kS; ++u) {
            if (j0 + NT * u >= GV * Q4) continue;
            __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc[u].x, acc[u].y);
            __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc[u].z, acc[u].w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo2);
            pk.y = *reinterpret_cast<uint32_t*>(&hi2);
            *reinterpret_cast<uint2*>(a.out + (row0 + hh[u]) * D + dd[u] * 4) = pk;
          }
        }
      };
      if (np <= 2)
        wsum(IntC<8>{}, IntC<2>{});
      else
        wsum(IntC<4>{}, IntC<4>{});
      block_sync();  // the next job reuses the weights and the job slots
    }
    // the last CTA out of the merge phase resets its counters
    if (tid == 0) {
      __threadfence();
      const int done = atomicAdd(a.queue + 4, 1);
      if (done == a.cta_count - 1) {
        a.queue[2] = 0;
        a.queue[3] = 0;
        a.queue[4] = 0;
      }
    }
  }
}

// Places the arrival counters, the merge queue, the item queue and the
// partial results of a decode call in its workspace (decode.cu).
void decode_workspace_split(DecodeArgs& a, void* workspace, size_t workspace_bytes,
                            int32_t batch, int32_t H_kv, int32_t D, int num_sms);

}  // namespace pkv
