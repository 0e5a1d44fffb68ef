// Prefill-side kernels: RMSNorm to bf16 GEMM operands, the projection GEMMs
// with fused epilogues (RoPE + KV-cache scatter, SwiGLU, residual add), causal
// attention over the paged cache, and small gathers.
#include "internal.cuh"

#include <math.h>

namespace ladder {

// ---------------------------------------------------------------------------
// out[m, :] = bf16(x[m, :] * rsqrt(mean(x[m, :]^2) + eps) * g)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const float* __restrict__ x, int d,
                                                            const bf16* __restrict__ g, float eps,
                                                            bf16* __restrict__ out) {
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
  bf16* o = out + (size_t)m * d;
  for (int i = tid * 4; i < d; i += 1024) {
    const float4 v = *reinterpret_cast<const float4*>(xr + i);
    const uint2 graw = *reinterpret_cast<const uint2*>(g + i);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * r * bf_lo(graw.x), v.y * r * bf_hi(graw.x));
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * r * bf_lo(graw.y), v.w * r * bf_hi(graw.y));
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(o + i) = pk;
  }
}

cudaError_t launch_rmsnorm_rows(const float* x, int M, int d, const bf16* g, float eps, bf16* out,
                                cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  rmsnorm_rows_kernel<<<M, 256, 0, s>>>(x, d, g, eps, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Shared epilogue of the projection GEMMs for output element pair (m, n), (m, n+1),
// n even.  QKV: rotate q/k pairs, store q (bf16) or scatter k/v into the cache;
// GATEUP: act = silu(gate) * up (bf16); RESID: x_out = x_res + acc (fp32).
// ---------------------------------------------------------------------------
template <int MODE>
__device__ __forceinline__ void gemm_store_pair(const GemmParams& p, int m, int n, float a0, float a1,
                                                float u0, float u1) {
  if (MODE == GEMM_QKV) {
    const int hd = p.kv.head_dim;
    int local, kind;
    if (n < p.nq_hd) { local = n; kind = 0; }
    else if (n < p.nq_hd + p.nkv_hd) { local = n - p.nq_hd; kind = 1; }
    else { local = n - p.nq_hd - p.nkv_hd; kind = 2; }
    const int pos = p.row_pos[m];
    float r0 = a0, r1 = a1;
    if (kind < 2) {
      const int j = (local % hd) >> 1;
      const float c = p.rope_cos[(size_t)pos * (hd >> 1) + j];
      const float s = p.rope_sin[(size_t)pos * (hd >> 1) + j];
      r0 = a0 * c - a1 * s;
      r1 = a0 * s + a1 * c;
    }
    __nv_bfloat162 v = __floats2bfloat162_rn(r0, r1);
    if (kind == 0) {
      *reinterpret_cast<__nv_bfloat162*>(p.out_bf + (size_t)m * p.ldo + local) = v;
    } else {
      const int b = p.row_b[m];
      const int head = local / hd, dim = local % hd;
      *reinterpret_cast<__nv_bfloat162*>(p.kv.base + p.kv.slot(b, pos, kind - 1, head) + dim) = v;
    }
  } else if (MODE == GEMM_GATEUP) {
    __nv_bfloat162 v = __floats2bfloat162_rn(silu_f(a0) * u0, silu_f(a1) * u1);
    *reinterpret_cast<__nv_bfloat162*>(p.out_bf + (size_t)m * p.ldo + n) = v;
  } else {
    const float2 r = *reinterpret_cast<const float2*>(p.x_res + (size_t)m * p.ldo + n);
    *reinterpret_cast<float2*>(p.out_f + (size_t)m * p.ldo + n) = make_float2(r.x + a0, r.y + a1);
  }
}

// ---------------------------------------------------------------------------
// Plain tiled GEMM on the CUDA cores: C[m, n] = sum_k A[m, k] W[n, k].
// 64 x 64 tile, k-step 32, each of 256 threads owns a 4 x 4 block.
// ---------------------------------------------------------------------------
template <int MODE>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const GemmParams p) {
  constexpr int BM = 64, BN = 64, BK = 32;
  constexpr bool TWO = MODE == GEMM_GATEUP;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float Us[TWO ? BK : 1][TWO ? BN + 4 : 1];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int K = p.K;

  const bf16* W = p.w0;
  int nrow0 = n0;  // first row of the tile inside W
  int nlim = p.N;  // rows of W
  if (MODE == GEMM_QKV) {
    if (n0 < p.nq_hd) { W = p.w0; nrow0 = n0; nlim = p.nq_hd; }
    else if (n0 < p.nq_hd + p.nkv_hd) { W = p.w1; nrow0 = n0 - p.nq_hd; nlim = p.nkv_hd; }
    else { W = p.w2; nrow0 = n0 - p.nq_hd - p.nkv_hd; nlim = p.nkv_hd; }
  }

  float acc[4][4], accu[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = accu[i][j] = 0.f;

  const int lr = tid >> 2, lk = (tid & 3) * 8;
  for (int k0 = 0; k0 < K; k0 += BK) {
    {
      uint4 a = make_uint4(0, 0, 0, 0), w = make_uint4(0, 0, 0, 0), uu = make_uint4(0, 0, 0, 0);
      if (m0 + lr < p.M) a = *reinterpret_cast<const uint4*>(p.A + (size_t)(m0 + lr) * K + k0 + lk);
      if (nrow0 + lr < nlim) {
        w = *reinterpret_cast<const uint4*>(W + (size_t)(nrow0 + lr) * K + k0 + lk);
        if (TWO) uu = *reinterpret_cast<const uint4*>(p.w1 + (size_t)(nrow0 + lr) * K + k0 + lk);
      }
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, wv[4] = {w.x, w.y, w.z, w.w};
      const uint32_t uv[4] = {uu.x, uu.y, uu.z, uu.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        As[lk + 2 * i][lr] = bf_lo(av[i]);
        As[lk + 2 * i + 1][lr] = bf_hi(av[i]);
        Bs[lk + 2 * i][lr] = bf_lo(wv[i]);
        Bs[lk + 2 * i + 1][lr] = bf_hi(wv[i]);
        if (TWO) {
          Us[lk + 2 * i][lr] = bf_lo(uv[i]);
          Us[lk + 2 * i + 1][lr] = bf_hi(uv[i]);
        }
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4], u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
        if (TWO) u[i] = Us[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (TWO) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const int n = n0 + tx * 4 + j;
      if (n >= p.N) continue;
      gemm_store_pair<MODE>(p, m, n, acc[i][j], acc[i][j + 1], accu[i][j], accu[i][j + 1]);
    }
  }
}

cudaError_t launch_gemm(const GemmParams& p, int mode, cudaStream_t s) {
  if (p.M <= 0) return cudaSuccess;
  dim3 grid((p.N + 63) / 64, (p.M + 63) / 64);
  switch (mode) {
    case GEMM_QKV: gemm_simt_kernel<GEMM_QKV><<<grid, 256, 0, s>>>(p); break;
    case GEMM_GATEUP: gemm_simt_kernel<GEMM_GATEUP><<<grid, 256, 0, s>>>(p); break;
    default: gemm_simt_kernel<GEMM_RESID><<<grid, 256, 0, s>>>(p); break;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Causal attention for packed prefill rows: one warp per (row, query head),
// keys 0..pos of the row's sequence read from the paged cache, online softmax
// over blocks of 32 keys (lane j scores key j of the block).
// ---------------------------------------------------------------------------
template <int HD>
__global__ void __launch_bounds__(256) attn_prefill_simt_kernel(const AttnPrefillParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 8 + warp;
  __shared__ float q_s[8][HD];
  if (item >= p.M * p.n_q) return;
  const int m = item / p.n_q, h = item % p.n_q;
  const int b = p.row_b[m], pos = p.row_pos[m];
  const int G = p.n_q / p.kv.n_kv, kvh = h / G;
  const bf16* qr = p.q + (size_t)m * p.n_q * HD + (size_t)h * HD;
  for (int d = lane; d < HD; d += 32) q_s[warp][d] = __bfloat162float(qr[d]);
  __syncwarp();

  constexpr int NV = HD / 32;
  float o[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) o[i] = 0.f;
  float mrun = -INFINITY, lrun = 0.f;
  for (int kb = 0; kb <= pos; kb += 32) {
    const int key = kb + lane;
    const bool valid = key <= pos;
    float sc = -INFINITY;
    if (valid) {
      const bf16* kr = p.kv.base + p.kv.slot(b, key, 0, kvh);
      float dot = 0.f;
#pragma unroll 4
      for (int d = 0; d < HD; d += 8) {
        const uint4 kw = *reinterpret_cast<const uint4*>(kr + d);
        const float* qq = &q_s[warp][d];
        dot += qq[0] * bf_lo(kw.x) + qq[1] * bf_hi(kw.x) + qq[2] * bf_lo(kw.y) + qq[3] * bf_hi(kw.y) +
               qq[4] * bf_lo(kw.z) + qq[5] * bf_hi(kw.z) + qq[6] * bf_lo(kw.w) + qq[7] * bf_hi(kw.w);
      }
      sc = dot * p.scale;
    }
    const float mnew = fmaxf(mrun, warp_max(sc));
    const float e = valid ? expf(sc - mnew) : 0.f;
    const float corr = expf(mrun - mnew);
    lrun = lrun * corr + warp_sum(e);
#pragma unroll
    for (int i = 0; i < NV; ++i) o[i] *= corr;
    const int nv = min(32, pos + 1 - kb);
    for (int j = 0; j < nv; ++j) {
      const float pj = __shfl_sync(0xffffffffu, e, j);
      const bf16* vr = p.kv.base + p.kv.slot(b, kb + j, 1, kvh);
#pragma unroll
      for (int i = 0; i < NV; ++i) o[i] += pj * __bfloat162float(vr[lane + 32 * i]);
    }
    mrun = mnew;
  }
  bf16* orow = p.out + (size_t)m * p.n_q * HD + (size_t)h * HD;
#pragma unroll
  for (int i = 0; i < NV; ++i) orow[lane + 32 * i] = __float2bfloat16_rn(o[i] / lrun);
}

cudaError_t launch_attn_prefill(const AttnPrefillParams& p, int hd, cudaStream_t s) {
  if (p.M <= 0) return cudaSuccess;
  const long long items = (long long)p.M * p.n_q;
  const unsigned grid = (unsigned)((items + 7) / 8);
  if (hd == 64) attn_prefill_simt_kernel<64><<<grid, 256, 0, s>>>(p);
  else attn_prefill_simt_kernel<128><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// out[b, :] = x[rows[b], :]
// ---------------------------------------------------------------------------
__global__ void gather_rows_kernel(const float* __restrict__ x, int d, const int* __restrict__ rows,
                                   float* __restrict__ out) {
  const int b = blockIdx.x;
  const float* src = x + (size_t)rows[b] * d;
  for (int i = threadIdx.x * 4; i < d; i += blockDim.x * 4)
    *reinterpret_cast<float4*>(out + (size_t)b * d + i) = *reinterpret_cast<const float4*>(src + i);
}

cudaError_t launch_gather_rows(const float* x, int d, const int* rows, int B, float* out, cudaStream_t s) {
  gather_rows_kernel<<<B, 256, 0, s>>>(x, d, rows, out);
  return cudaGetLastError();
}

__global__ void set_lens_kernel(const int* lens, int B, int* seq_lens) {
  const int b = threadIdx.x;
  if (b < B) seq_lens[b] = lens[b];
}

cudaError_t launch_set_lens(const int* lens, int B, int* seq_lens, cudaStream_t s) {
  set_lens_kernel<<<1, 64, 0, s>>>(lens, B, seq_lens);
  return cudaGetLastError();
}

}  // namespace ladder
