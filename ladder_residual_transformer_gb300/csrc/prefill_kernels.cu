// Prefill-side helper kernels: RMSNorm of the stream rows into the 16-bit
// operand of the next tensor-core GEMM, and small gathers.  The projection
// GEMMs are in gemm_tcgen05.cu and the causal attention in attn_prefill_tcgen05.cu.
#include "internal.cuh"

#include <math.h>

namespace ladder {

// ---------------------------------------------------------------------------
// out[m, :] = x[m, :] * rsqrt(mean(x[m, :]^2) + eps) * g, rounded to the
// operand type (bf16 or fp16).  One CTA per row, fixed reduction order.  With
// lo_off > 0 the rounding remainder of every value, u - float(round(u)), is
// rounded too and written to the lo plane at out + lo_off, so that the pair
// (hi, lo) carries u to about twice the 16-bit precision.
// ---------------------------------------------------------------------------
template <typename WT>
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const float* __restrict__ x, int d,
                                                            const WT* __restrict__ g, float eps,
                                                            WT* __restrict__ out, size_t lo_off) {
  using C = W16<WT>;
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, tid = threadIdx.x;
  const float* xr = x + (size_t)m * d;
  float ss = 0.f;
  for (int i = tid * 4; i < d; i += 1024) {
    const float4 v = *reinterpret_cast<const float4*>(xr + i);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  __shared__ float red[8];
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += red[w];
  const float r = rsqrtf(t / (float)d + eps);
  WT* o = out + (size_t)m * d;
  for (int i = tid * 4; i < d; i += 1024) {
    const float4 v = *reinterpret_cast<const float4*>(xr + i);
    const uint2 graw = *reinterpret_cast<const uint2*>(g + i);
    const float u0 = v.x * r * C::lo(graw.x), u1 = v.y * r * C::hi(graw.x);
    const float u2 = v.z * r * C::lo(graw.y), u3 = v.w * r * C::hi(graw.y);
    uint2 pk;
    pk.x = C::pack(u0, u1);
    pk.y = C::pack(u2, u3);
    *reinterpret_cast<uint2*>(o + i) = pk;
    if (lo_off) {
      uint2 pl;
      pl.x = C::pack(u0 - C::lo(pk.x), u1 - C::hi(pk.x));
      pl.y = C::pack(u2 - C::lo(pk.y), u3 - C::hi(pk.y));
      *reinterpret_cast<uint2*>(o + lo_off + i) = pl;
    }
  }
}

cudaError_t launch_rmsnorm_rows(const float* x, int M, int d, const void* g, float eps, void* out, size_t lo_off,
                                int wdt, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (wdt == WDT_F16)
    return launch_k(rmsnorm_rows_kernel<f16>, dim3(M), dim3(256), 0, s, pdl, x, d, static_cast<const f16*>(g), eps,
                    static_cast<f16*>(out), lo_off);
  return launch_k(rmsnorm_rows_kernel<bf16>, dim3(M), dim3(256), 0, s, pdl, x, d, static_cast<const bf16*>(g), eps,
                  static_cast<bf16*>(out), lo_off);
}

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
