// paged_kv_append_rope: the KV append with the attention input transform
// fused in.  Per new token: each q head and each k head is normalised by a
// per-head RMSNorm over head_dim (Qwen3's q_norm / k_norm: scripts/benchmarks
// commit log, Llama-3.2 support commit) and rotated by the rotary embedding
// of the token's position (rotate-half pairs (i, i + D/2)); q is written
// back in place, k goes to its page slot, and v is copied to the same slot
// unchanged (the cache stores post-rotary K: Gemma-4 shared-KV commit).
//
// HBM-bound elementwise work (the layout of the work is described at the
// kernel).  All arithmetic is fp32 with one rounding to bf16 at the end.
//
// pkv_rope_table's kernel fills that table in double precision (CUDA's
// pow and sincos), rounding each entry once to float.
#include "common.cuh"
#include "kernels.h"

namespace pkv {


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

// Work unit: R = kRopeSteps * (512 / D) consecutive q/k rows of one token
// (q heads first, then kv heads), processed by one warp.  A lane owns pair
// slice j of every row it touches: dims [8j, 8j+8) and [D/2+8j, D/2+8j+8),
// two 16-byte vectors, so both members of each of its rotary pairs are in
// its own registers.  A row spans D/16 lanes (the RMSNorm sum of squares is
// a shuffle reduction over them) and a warp step covers 512/D rows.  The
// token's position and slot, the lane's cos/sin values and its slices of
// both norm weights are loaded once per unit; the unit's rows (and, for kv
// rows, the v rows) are loaded before any is finished.  Arithmetic on pairs
// of floats uses the f32x2 forms.
#ifndef PKV_ROPE_STEPS
#define PKV_ROPE_STEPS 2
#endif
#ifndef PKV_ROPE_MINBLOCKS
#define PKV_ROPE_MINBLOCKS 2
#endif
constexpr int kRopeSteps = PKV_ROPE_STEPS;
constexpr int kRopeBlocksPerSm = PKV_ROPE_MINBLOCKS;

namespace {
// the 4 bf16 pairs of a 16-byte vector as 4 float pairs
__device__ __forceinline__ void unpack_pairs(const uint4 v, uint64_t (&p)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k)
    p[k] = f2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
}
__device__ __forceinline__ uint4 pack_pairs(const uint64_t (&p)[4]) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float lo, hi;
    f2_split(p[k], lo, hi);
    w[k] = pack_bf16(lo, hi);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
}  // namespace

template <int D>
__global__ void __launch_bounds__(256, kRopeBlocksPerSm) kv_append_rope_kernel(
    const RopeAppendArgs a) {
  constexpr int LPR = D / 16;     // lanes per row
  constexpr int RPS = 32 / LPR;   // rows per warp step
  constexpr int U = kRopeSteps;   // steps per unit
  constexpr int R = U * RPS;      // rows per unit
  constexpr int VR = D / 8;       // 16-byte vectors per row
  constexpr int HV = D / 16;      // ... per half row
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int j = lane & (LPR - 1);  // the lane's pair slice
  const int sub = lane / LPR;      // the lane's row within a step
  const int32_t Hq = a.q != nullptr ? a.H_q : 0;
  const int32_t rows = Hq + a.H_kv;
  const int32_t units_per_tok = (rows + R - 1) / R;
  const int32_t units = a.T * units_per_tok;  // host-checked to fit
  const int32_t nwarps = (int32_t)((gridDim.x * blockDim.x) >> 5);
  uint4* q = static_cast<uint4*>(a.q);
  const uint4* k_new = static_cast<const uint4*>(a.k_new);
  const uint4* v_new = static_cast<const uint4*>(a.v_new);
  uint4* k_cache = static_cast<uint4*>(a.k_cache);
  uint4* v_cache = static_cast<uint4*>(a.v_cache);
  // the lane's slices of the two norm weights, kept packed (bf16)
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  const uint4* qwp = static_cast<const uint4*>(a.q_w);
  const uint4* kwp = static_cast<const uint4*>(a.k_w);
  const uint4 qwl = qwp ? __ldg(qwp + j) : z, qwh = qwp ? __ldg(qwp + HV + j) : z;
  const uint4 kwl = kwp ? __ldg(kwp + j) : z, kwh = kwp ? __ldg(kwp + HV + j) : z;

  for (int32_t unit = (int32_t)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); unit < units;
       unit += nwarps) {  // warp-uniform
    const int32_t t = unit / units_per_tok;
    const int32_t row0 = (unit - t * units_per_tok) * R;
    const int32_t pos = __ldg(a.positions + t);
    const bool live = pos >= 0 && pos < a.max_pos;
    // the rows: loads first
    uint4 xl[U], xh[U], vl[U], vh[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int32_t hr = row0 + u * RPS + sub;
      xl[u] = xh[u] = vl[u] = vh[u] = z;
      if (live && hr < rows) {
        if (hr < Hq) {
          const int64_t b = ((int64_t)t * Hq + hr) * VR + j;
          xl[u] = q[b];
          xh[u] = q[b + HV];
        } else {
          const int64_t b = ((int64_t)t * a.H_kv + (hr - Hq)) * VR + j;
          xl[u] = __ldg(k_new + b);
          xh[u] = __ldg(k_new + b + HV);
          vl[u] = __ldg(v_new + b);
          vh[u] = __ldg(v_new + b + HV);
        }
      }
    }
    if (!live) {  // warp-uniform: the whole unit belongs to token t
      if (row0 == 0 && lane == 0) raise_err(a.err, PKV_DEVERR_POS);
      continue;
    }
    uint64_t c[4], sp[4], sn[4];  // cos, sin and -sin of the lane's 8 pairs
    {
      const float4* cs = reinterpret_cast<const float4*>(a.cos_sin + (int64_t)pos * D);
      const float4 c0 = __ldg(cs + 2 * j), c1 = __ldg(cs + 2 * j + 1);
      const float4 s0 = __ldg(cs + D / 8 + 2 * j), s1 = __ldg(cs + D / 8 + 2 * j + 1);
      c[0] = f2(c0.x, c0.y); c[1] = f2(c0.z, c0.w); c[2] = f2(c1.x, c1.y); c[3] = f2(c1.z, c1.w);
      sp[0] = f2(s0.x, s0.y); sp[1] = f2(s0.z, s0.w); sp[2] = f2(s1.x, s1.y); sp[3] = f2(s1.z, s1.w);
      sn[0] = f2(-s0.x, -s0.y); sn[1] = f2(-s0.z, -s0.w);
      sn[2] = f2(-s1.x, -s1.y); sn[3] = f2(-s1.z, -s1.w);
    }
    const bool has_kv = row0 + R > Hq;
    int64_t slot = -1;
    if (has_kv) slot = __ldg(a.slot_mapping + t);
    if (has_kv && slot >= a.num_slots && lane == 0 && row0 <= Hq)
      raise_err(a.err, PKV_DEVERR_SLOT);
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
      uint64_t fl[4], fh[4];
      unpack_pairs(xl[u], fl);
      unpack_pairs(xh[u], fh);
      // per-head RMSNorm: sum of squares over the row's LPR lanes
      uint64_t acc = f2_mul(fl[0], fl[0]);
#pragma unroll
      for (int k = 1; k < 4; ++k) acc = f2_fma(fl[k], fl[k], acc);
#pragma unroll
      for (int k = 0; k < 4; ++k) acc = f2_fma(fh[k], fh[k], acc);
      float s0, s1;
      f2_split(acc, s0, s1);
      float ss = s0 + s1;
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
      if (isq ? qwp != nullptr : kwp != nullptr) {
        const float rn = rsqrtf(ss * (1.f / (float)D) + a.eps);
        const uint64_t rn2 = f2(rn, rn);
        uint64_t wl[4], wh[4];
        unpack_pairs(isq ? qwl : kwl, wl);
        unpack_pairs(isq ? qwh : kwh, wh);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          fl[k] = f2_mul(fl[k], f2_mul(rn2, wl[k]));
          fh[k] = f2_mul(fh[k], f2_mul(rn2, wh[k]));
        }
      }
      // rotary: (lo, hi) -> (lo c - hi s, hi c + lo s)
      uint64_t ol[4], oh[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        ol[k] = f2_fma(fl[k], c[k], f2_mul(fh[k], sn[k]));
        oh[k] = f2_fma(fh[k], c[k], f2_mul(fl[k], sp[k]));
      }
      if (hr >= rows) continue;
      if (isq) {
        const int64_t b = ((int64_t)t * Hq + hr) * VR + j;
        q[b] = pack_pairs(ol);
        q[b + HV] = pack_pairs(oh);
      } else if (store_kv) {
        const int64_t b = ((page * a.H_kv + (hr - Hq)) * a.P + prow) * VR + j;
        k_cache[b] = pack_pairs(ol);
        k_cache[b + HV] = pack_pairs(oh);
        v_cache[b] = vl[u];
        v_cache[b + HV] = vh[u];
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
  const int64_t R = (int64_t)kRopeSteps * (512 / D);
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
