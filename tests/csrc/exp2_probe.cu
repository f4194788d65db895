// Test probe: evaluates the softmax's polynomial 2^x (poly_exp2x2) on the
// GPU for a host-chosen set of inputs, so that a test can check its stated
// error bound.  Built by the test itself; not part of libpkv.so.
#include "../../paged_kv_attention_11_gb300/csrc/exp2_math.cuh"

namespace {

__global__ void poly_exp2_probe_kernel(const float* x, float* y, int n_pairs) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_pairs) return;
  float y0, y1;
  pkv::f2_split(pkv::poly_exp2x2(pkv::f2(x[2 * i], x[2 * i + 1])), y0, y1);
  y[2 * i] = y0;
  y[2 * i + 1] = y1;
}

}  // namespace

// x, y: device arrays of 2 * n_pairs floats.  Returns a cudaError_t value.
extern "C" int poly_exp2_probe(const float* x, float* y, int n_pairs, void* stream) {
  if (n_pairs <= 0) return 0;
  poly_exp2_probe_kernel<<<(n_pairs + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, y, n_pairs);
  return static_cast<int>(cudaGetLastError());
}
