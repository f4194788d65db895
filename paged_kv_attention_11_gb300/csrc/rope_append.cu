// paged_kv_append_rope: the KV append with the attention input transform
// fused in.  Per new token: each q head and each k head is normalised by a
// per-head RMSNorm over head_dim (Qwen3's q_norm / k_norm: scripts/benchmarks
// commit log, Llama-3.2 support commit) and rotated by the rotary embedding
// of the token's position (rotate-half pairs (i, i + D/2)); q is written
// back in place, k goes to its page slot, and v is copied to the same slot
// unchanged (the cache stores post-rotary K: Gemma-4 shared-KV commit).
//
// HBM-bound elementwise work.  One thread owns one 16-byte vector (8 bf16)
// of a q/k row, so a row of head_dim values spans D/8 consecutive lanes of
// one warp: the sum of squares is a shuffle reduction over those lanes and
// the rotary partner of a lane's 8 values sits HALF = D/16 lanes away
// (one xor-shuffle per value).  The thread that owns a k vector also moves
// the matching v vector.  All arithmetic is fp32 with one rounding to bf16
// at the end.  The cos/sin table row of a token is read by all its heads and
// stays in L1/L2.
//
// pkv_rope_table's kernel fills that table in double precision (CUDA's
// pow and sincos), rounding each entry once to float.
#include "common.cuh"
#include "kernels.h"

namespace pkv {

namespace {

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16(f[0], f[1]);
  v.y = pack_bf16(f[2], f[3]);
  v.z = pack_bf16(f[4], f[5]);
  v.w = pack_bf16(f[6], f[7]);
  return v;
}

}  // namespace

__global__ void __launch_bounds__(256) rope_table_kernel(float* __restrict__ cs, int32_t max_pos,
                                                         int32_t D, double theta) {
  const int32_t half = D / 2;
  const int64_t n = (int64_t)max_pos * half;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
    const int64_t p = e / half;
    const int32_t i = (int32_t)(e - p * half);
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
    double s, c;
    sincos((double)p * inv_freq, &s, &c);
    cs[p * D + i] = (float)c;
    cs[p * D + half + i] = (float)s;
  }
}

// One vector of a q/k row: where it comes from and its raw contents.
struct RopeVec {
  int32_t t, hr, l, pos;
  bool in, live, isq;
  int64_t src;
  uint4 x, v;
};

template <int D>
__device__ __forceinline__ RopeVec rope_load(const RopeAppendArgs& a, int32_t i, int32_t total,
                                             int32_t Hq, int32_t rows_per_tok) {
  constexpr int LPR = D / 8;
  RopeVec r;
  r.in = i < total;
  const int32_t row = r.in ? i / LPR : 0;
  r.l = i & (LPR - 1);
  r.t = row / rows_per_tok;
  r.hr = row - r.t * rows_per_tok;
  r.isq = r.hr < Hq;
  r.pos = r.in ? __ldg(a.positions + r.t) : 0;
  r.live = r.in && r.pos >= 0 && r.pos < a.max_pos;
  r.src = r.isq ? ((int64_t)r.t * Hq + r.hr) * LPR + r.l
                : ((int64_t)r.t * a.H_kv + (r.hr - Hq)) * LPR + r.l;
  r.x = make_uint4(0u, 0u, 0u, 0u);
  r.v = r.x;
  if (r.live) {
    if (r.isq) {
      r.x = static_cast<const uint4*>(a.q)[r.src];
    } else {
      r.x = __ldg(static_cast<const uint4*>(a.k_new) + r.src);
      r.v = __ldg(static_cast<const uint4*>(a.v_new) + r.src);
    }
  }
  return r;
}

// Norm, rotate and store one vector.  Every lane of the warp calls it (the
// shuffles need them all), whatever its vector's state.
template <int D>
__device__ __forceinline__ void rope_finish(const RopeAppendArgs& a, const RopeVec& r,
                                            int32_t Hq) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int HALF = LPR / 2;  // lane distance between rotary partners
  float x[8];
  unpack8(r.x, x);
  // per-head RMSNorm: sum of squares over the row's LPR lanes
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) ss = fmaf(x[k], x[k], ss);
#pragma unroll
  for (int off = HALF; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const uint4* w = static_cast<const uint4*>(r.isq ? a.q_w : a.k_w);
  if (w != nullptr) {
    const float rn = rsqrtf(ss * (1.f / (float)D) + a.eps);
    float wf[8];
    unpack8(__ldg(w + r.l), wf);
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = x[k] * rn * wf[k];
  }
  // rotary: lanes [0, HALF) hold dims i < D/2, lanes [HALF, LPR) dims i + D/2
  float y[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) y[k] = __shfl_xor_sync(0xFFFFFFFFu, x[k], HALF);
  const bool lo = r.l < HALF;
  const int i0 = (lo ? r.l : r.l - HALF) * 8;  // first pair index of this vector
  const float4* cs = reinterpret_cast<const float4*>(a.cos_sin + (int64_t)(r.live ? r.pos : 0) * D);
  const float4 c0 = __ldg(cs + i0 / 4), c1 = __ldg(cs + i0 / 4 + 1);
  const float4 s0 = __ldg(cs + (D / 2 + i0) / 4), s1 = __ldg(cs + (D / 2 + i0) / 4 + 1);
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float o[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    o[k] = lo ? fmaf(x[k], c[k], -y[k] * s[k]) : fmaf(x[k], c[k], y[k] * s[k]);

  if (!r.in) return;
  if (!r.live) {
    if (r.hr == 0 && r.l == 0) raise_err(a.err, PKV_DEVERR_POS);
    return;
  }
  if (r.isq) {
    static_cast<uint4*>(a.q)[r.src] = pack8(o);
    return;
  }
  const int64_t slot = __ldg(a.slot_mapping + r.t);
  if (slot < 0) return;  // padding row: skip the append
  if (slot >= a.num_slots) {
    if (r.hr == Hq && r.l == 0) raise_err(a.err, PKV_DEVERR_SLOT);
    return;
  }
  const int64_t page = slot / a.P;
  const int64_t prow = slot - page * a.P;
  const int64_t dst = ((page * a.H_kv + (r.hr - Hq)) * a.P + prow) * LPR + r.l;
  static_cast<uint4*>(a.k_cache)[dst] = pack8(o);
  static_cast<uint4*>(a.v_cache)[dst] = r.v;
}

template <int D>
__global__ void __launch_bounds__(256, 4) kv_append_rope_kernel(const RopeAppendArgs a) {
  constexpr int LPR = D / 8;
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int32_t Hq = a.q != nullptr ? a.H_q : 0;
  const int32_t rows_per_tok = Hq + a.H_kv;
  const int32_t total = a.T * rows_per_tok * LPR;  // host-checked: < 2^30
  const int32_t nthreads = (int32_t)(gridDim.x * blockDim.x);
  // Whole warps iterate together (the shuffles need every lane); two
  // vectors per thread per step, both loaded before either is finished.
  for (int32_t base = (int32_t)(blockIdx.x * blockDim.x + (threadIdx.x & ~31u)); base < total;
       base += 2 * nthreads) {
    const RopeVec r0 = rope_load<D>(a, base + lane, total, Hq, rows_per_tok);
    const RopeVec r1 = rope_load<D>(a, base + nthreads + lane, total, Hq, rows_per_tok);
    rope_finish<D>(a, r0, Hq);
    rope_finish<D>(a, r1, Hq);
  }
}

cudaError_t launch_rope_table(float* cos_sin, int32_t max_pos, int32_t D, double theta,
                              cudaStream_t stream, int num_sms) {
  const int64_t n = (int64_t)max_pos * (D / 2);
  if (n == 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  rope_table_kernel<<<(unsigned)blocks, 256, 0, stream>>>(cos_sin, max_pos, D, theta);
  return cudaGetLastError();
}

cudaError_t launch_kv_append_rope(const RopeAppendArgs& a, int32_t D, cudaStream_t stream,
                                  int num_sms) {
  const int64_t total = (int64_t)a.T * ((a.q != nullptr ? a.H_q : 0) + a.H_kv) * (D / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 511) / 512;  // two vectors per thread
  const int64_t cap = (int64_t)num_sms * 4;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (D) {
    case 64: return cudaLaunchKernelEx(&cfg, kv_append_rope_kernel<64>, a);
    case 128: return cudaLaunchKernelEx(&cfg, kv_append_rope_kernel<128>, a);
    case 256: return cudaLaunchKernelEx(&cfg, kv_append_rope_kernel<256>, a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pkv
