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

// Work unit: kRopeSteps * (256 / D) consecutive rows of one token's q/k
// rows (q heads first, then kv heads), processed by one warp.  Lane `lane`
// always owns the same 16-byte slice l = lane % (D/8) of a row, so the
// token's position and slot, the lane's cos/sin values and its slice of
// both norm weights are loaded once per unit and reused for every row.
// Each step covers 32 / (D/8) rows; the unit's kRopeSteps steps load their
// rows (and, for kv rows, the v rows) before any is finished.
#ifndef PKV_ROPE_STEPS
#define PKV_ROPE_STEPS 4
#endif
#ifndef PKV_ROPE_MINBLOCKS
#define PKV_ROPE_MINBLOCKS 2
#endif
constexpr int kRopeSteps = PKV_ROPE_STEPS;
constexpr int kRopeBlocksPerSm = PKV_ROPE_MINBLOCKS;

template <int D>
__global__ void __launch_bounds__(256, kRopeBlocksPerSm) kv_append_rope_kernel(
    const RopeAppendArgs a) {
  constexpr int LPR = D / 8;           // lanes per row
  constexpr int HALF = LPR / 2;        // lane distance between rotary partners
  constexpr int RPS = 32 / LPR;        // rows per warp step
  constexpr int U = kRopeSteps;        // steps per unit
  constexpr int R = U * RPS;           // rows per unit
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int l = lane & (LPR - 1);      // the lane's slice of a row
  const int sub = lane / LPR;          // the lane's row within a step
  const bool lo = l < HALF;
  const int i0 = (l & (HALF - 1)) * 8;  // first rotary pair of the slice
  const int32_t Hq = a.q != nullptr ? a.H_q : 0;
  const int32_t rows = Hq + a.H_kv;
  const int32_t units_per_tok = (rows + R - 1) / R;
  const int64_t units = (int64_t)a.T * units_per_tok;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint4* q = static_cast<uint4*>(a.q);
  const uint4* k_new = static_cast<const uint4*>(a.k_new);
  const uint4* v_new = static_cast<const uint4*>(a.v_new);
  // the lane's slices of the two norm weights, kept packed (bf16)
  const uint4 qw = a.q_w ? __ldg(static_cast<const uint4*>(a.q_w) + l) : make_uint4(0u, 0u, 0u, 0u);
  const uint4 kw = a.k_w ? __ldg(static_cast<const uint4*>(a.k_w) + l) : make_uint4(0u, 0u, 0u, 0u);

  for (int64_t unit = (((int64_t)blockIdx.x * blockDim.x) >> 5) + (threadIdx.x >> 5);
       unit < units; unit += nwarps) {  // warp-uniform
    const int32_t t = (int32_t)(unit / units_per_tok);
    const int32_t row0 = (int32_t)(unit - (int64_t)t * units_per_tok) * R;
    const int32_t pos = __ldg(a.positions + t);
    const bool live = pos >= 0 && pos < a.max_pos;
    // the rows: loads first
    uint4 x[U], v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t hr = row0 + u * RPS + sub;
      x[u] = make_uint4(0u, 0u, 0u, 0u);
      v[u] = x[u];
      if (live && hr < rows) {
        if (hr < Hq) {
          x[u] = q[((int64_t)t * Hq + hr) * LPR + l];
        } else {
          const int64_t src = ((int64_t)t * a.H_kv + (hr - Hq)) * LPR + l;
          x[u] = __ldg(k_new + src);
          v[u] = __ldg(v_new + src);
        }
      }
    }
    if (!live) {  // warp-uniform: the whole unit belongs to token t
      if (row0 == 0 && lane == 0) raise_err(a.err, PKV_DEVERR_POS);
      continue;
    }
    const float4* cs = reinterpret_cast<const float4*>(a.cos_sin + (int64_t)pos * D);
    float c[8], s[8];
    {
      const float4 c0 = __ldg(cs + i0 / 4), c1 = __ldg(cs + i0 / 4 + 1);
      const float4 s0 = __ldg(cs + (D / 2 + i0) / 4), s1 = __ldg(cs + (D / 2 + i0) / 4 + 1);
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
      c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
      s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
      s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
    }
    const bool has_kv = row0 + R > Hq;
    int64_t slot = -1;
    if (has_kv) slot = __ldg(a.slot_mapping + t);
    if (has_kv && slot >= a.num_slots && lane == 0 && row0 <= Hq) raise_err(a.err, PKV_DEVERR_SLOT);
    const bool store_kv = slot >= 0 && slot < a.num_slots;
    int64_t page = 0, prow = 0;
    if (store_kv) {
      page = a.P_shift >= 0 ? (slot >> a.P_shift) : slot / a.P;
      prow = slot - page * a.P;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t hr = row0 + u * RPS + sub;
      const bool isq = hr < Hq;
      float f[8];
      unpack8(x[u], f);
      // per-head RMSNorm: sum of squares over the row's LPR lanes
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(f[k], f[k], ss);
#pragma unroll
      for (int off = HALF; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
      if (isq ? a.q_w != nullptr : a.k_w != nullptr) {
        const float rn = rsqrtf(ss * (1.f / (float)D) + a.eps);
        float wf[8];
        unpack8(isq ? qw : kw, wf);
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = f[k] * rn * wf[k];
      }
      // rotary: lanes [0, HALF) of a row hold dims i < D/2, the rest i + D/2
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float y = __shfl_xor_sync(0xFFFFFFFFu, f[k], HALF);
        o[k] = lo ? fmaf(f[k], c[k], -y * s[k]) : fmaf(f[k], c[k], y * s[k]);
      }
      if (hr >= rows) continue;
      if (isq) {
        static_cast<uint4*>(a.q)[((int64_t)t * Hq + hr) * LPR + l] = pack8(o);
      } else if (store_kv) {
        const int64_t dst = ((page * a.H_kv + (hr - Hq)) * a.P + prow) * LPR + l;
        static_cast<uint4*>(a.k_cache)[dst] = pack8(o);
        static_cast<uint4*>(a.v_cache)[dst] = v[u];
      }
    }
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
  const int64_t rows = (a.q != nullptr ? a.H_q : 0) + a.H_kv;
  const int64_t R = (int64_t)kRopeSteps * (256 / D);
  const int64_t units = (int64_t)a.T * ((rows + R - 1) / R);  // one warp each
  if (units == 0) return cudaSuccess;
  int64_t blocks = (units + 7) / 8;
  const int64_t cap = (int64_t)num_sms * kRopeBlocksPerSm;  // the resident blocks
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
