// Prefill-side helper kernels: small gathers and bookkeeping.  The projection
// GEMMs (whose epilogues also carry the RMSNorm of the prefill rows) are in
// gemm_tcgen05.cu and the causal attention in attn_prefill_tcgen05.cu.
#include "internal.cuh"

#include <math.h>

namespace ladder {

// ---------------------------------------------------------------------------
// out[b, :] = x[rows[b], :]
// ---------------------------------------------------------------------------
__global__ void gather_rows_kernel(const float* __restrict__ x, int d, const int* __restrict__ rows,
                                   float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const float* src = x + (size_t)rows[b] * d;
  for (int i = threadIdx.x * 4; i < d; i += blockDim.x * 4)
    *reinterpret_cast<float4*>(out + (size_t)b * d + i) = *reinterpret_cast<const float4*>(src + i);
}

cudaError_t launch_gather_rows(const float* x, int d, const int* rows, int B, float* out, cudaStream_t s, bool pdl) {
  return launch_k(gather_rows_kernel, dim3(B), dim3(256), 0, s, pdl, x, d, rows, out);
}

__global__ void set_lens_kernel(const int* lens, int B, int* seq_lens) {
  pdl_trigger();
  pdl_wait();
  const int b = threadIdx.x;
  if (b < B) seq_lens[b] = lens[b];
}

cudaError_t launch_set_lens(const int* lens, int B, int* seq_lens, cudaStream_t s, bool pdl) {
  return launch_k(set_lens_kernel, dim3(1), dim3(64), 0, s, pdl, lens, B, seq_lens);
}

}  // namespace ladder
