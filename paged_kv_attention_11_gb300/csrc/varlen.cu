// paged_attn_varlen: the tcgen05 prefill kernel (its body, varlen_cta, is in
// varlen_body.cuh) and its host-side launch.
#include "varlen_body.cuh"

namespace pkv {

template <int D, int NQ, int BN, int NS, int NKS, int NVS, int DV>
__global__ void __launch_bounds__(varlen_threads<NQ>(), 1)
    varlen_fwd_kernel(const VarlenArgs a, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  varlen_cta<D, NQ, BN, NS, NKS, NVS, false, DV>(a, tmQ, tmK, tmV, smem, blockIdx.x, gridDim.x);
}

// --------------------------------------------------------------- host side
template <int D, int NQ, int BN, int NS, int NKS, int NVS, int DV = D>
static cudaError_t launch_varlen_t(const VarlenArgs& a, const VarlenMaps& maps,
                                   cudaStream_t stream, int num_sms) {
  using S_ = VarlenSmem<D, NQ, BN, NS, NKS, NVS, DV>;
  auto kern = varlen_fwd_kernel<D, NQ, BN, NS, NKS, NVS, DV>;
  const size_t smem = S_::bytes(a.batch, a.pairs_max);
  if (smem > 227 * 1024) {
    // the deep rings do not fit next to this batch's schedule: fewer slots
    if (NKS > 2)
      return launch_varlen_t<D, NQ, BN, NS, (NKS > 2 ? NKS - 1 : 2), NVS, DV>(a, maps, stream,
                                                                              num_sms);
    if (NVS > 2)
      return launch_varlen_t<D, NQ, BN, NS, NKS, (NVS > 2 ? NVS - 1 : 2), DV>(a, maps, stream,
                                                                              num_sms);
    return cudaErrorNotSupported;
  }
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < (int)smem) {
    if (NQ == 2) {
      // the softmax warps raise their registers to 200 with what the other
      // warpgroup gives back (down to 104): that needs the launch to hold
      // 168 per thread, else the raise would never be granted
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs * varlen_threads<NQ>() < 8 * 32 * 200 + 4 * 32 * 104)
        return cudaErrorNotSupported;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = (int)smem;
  }
  // persistent grid: one CTA per SM, never more CTAs than work items
  const int64_t items_max = (int64_t)a.batch * a.H_kv * a.R * (D / DV);
  const int64_t grid = items_max < num_sms ? items_max : num_sms;
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(varlen_threads<NQ>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, maps.q, maps.k, maps.v);
}

int varlen_kv_tile(int head_dim) {
  return head_dim == 512 ? 32 : (head_dim == 256 ? 64 : 128);
}

// head_dim 512: one Q tile (128 x 512 bf16, 128 KB) fills half of shared
// memory and its fp32 O would fill all 512 TMEM columns, so a work item
// computes one 256-column half of O (S = Q K^T over all 512 dims, twice per
// Q tile) over 32-key tiles.
int varlen_v_cols(int head_dim) { return head_dim == 512 ? 256 : head_dim; }

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
  const int BN = varlen_kv_tile(D);
  a.P = P;
  a.box_rows = P < BN ? P : BN;
  a.num_pages = num_pages;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = causal;
  a.window = window;
  a.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31) == 0 ? 1 : 0;
  a.err = err;
  if (max_seqlen_q <= 0) return cudaSuccess;
  switch (D) {
    case 64:
      a.R = (max_seqlen_q + 2 * QP - 1) / (2 * QP);
      a.pairs_max = batch * a.R;
      return launch_varlen_t<64, 2, 128, 1, 4, 4>(a, maps, stream, num_sms);
    case 128:
      a.R = (max_seqlen_q + 2 * QP - 1) / (2 * QP);
      a.pairs_max = batch * a.R;
      return launch_varlen_t<128, 2, 128, 1, 3, 2>(a, maps, stream, num_sms);
    case 256:
      a.R = (max_seqlen_q + QP - 1) / QP;
      a.pairs_max = batch * a.R;
      return launch_varlen_t<256, 1, 64, 2, 2, 2>(a, maps, stream, num_sms);
    case 512:
      a.R = (max_seqlen_q + QP - 1) / QP;
      a.pairs_max = batch * a.R;
      return launch_varlen_t<512, 1, 32, 2, 2, 2, 256>(a, maps, stream, num_sms);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace pkv
