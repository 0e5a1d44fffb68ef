// Decode-side kernels of the Ladder Transformer forward pass (one new token per
// sequence, B <= 64 sequences): embedding gather, paged split-context
// attention and its combine step, greedy argmax, and small bookkeeping
// kernels.  The weight-streaming GEMVs are in gemv_stream.cu.
#include "internal.cuh"

#include <math.h>

namespace ladder {


// ---------------------------------------------------------------------------
// Embedding gather: x[m, :] = float(E[tok[m], :]).  Out-of-range ids write a
// zero row and set bit 0 of the error word.
// ---------------------------------------------------------------------------
template <typename WT>
__global__ void embed_kernel(const int* __restrict__ tok, const WT* __restrict__ E, int d, int vocab,
                             float* __restrict__ x, int* err) {
  using C = W16<WT>;
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  const int t = tok[m];
  const bool ok = (unsigned)t < (unsigned)vocab;
  if (!ok && threadIdx.x == 0) atomicOr(err, 1);
  const WT* row = E + (size_t)(ok ? t : 0) * d;
  float* out = x + (size_t)m * d;
  for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
    uint4 v = ok ? *reinterpret_cast<const uint4*>(row + i) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<float4*>(out + i) = make_float4(C::lo(v.x), C::hi(v.x), C::lo(v.y), C::hi(v.y));
    *reinterpret_cast<float4*>(out + i + 4) = make_float4(C::lo(v.z), C::hi(v.z), C::lo(v.w), C::hi(v.w));
  }
}

cudaError_t launch_embed(const int* tok, int M, const void* E, int wdt, int d, int vocab, float* x, int* err,
                         cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (wdt == WDT_F16)
    return launch_k(embed_kernel<f16>, dim3(M), dim3(128), 0, s, pdl, tok, static_cast<const f16*>(E), d, vocab, x, err);
  return launch_k(embed_kernel<bf16>, dim3(M), dim3(128), 0, s, pdl, tok, static_cast<const bf16*>(E), d, vocab, x, err);
}

// ---------------------------------------------------------------------------
// Decode attention over the paged cache, split along the context.
// CTA (split, kv head, sequence): the G = n_q / n_kv query heads of the group
// against keys [split * split_len, ...) of the sequence.  The CTA first issues
// every K and V load of its split at once (16-byte cp.async, coalesced along
// each page's contiguous [page_size][head_dim] slab) into padded shared memory,
// so the whole split is a single memory round trip.  Thread t then scores key t
// for all G heads; each warp normalises heads w, w+4 with warp-shuffle max/sum
// reductions; threads (dim pair, key group) accumulate P V.  Partial (max, sum,
// o) per split are merged by attn_combine_kernel.
// ---------------------------------------------------------------------------
constexpr int ATT_THREADS = 128;
constexpr int ATT_MAXG = 8;
constexpr int ATT_SPLIT = 128;  // keys per split (= ATT_THREADS)

__device__ __forceinline__ void att_cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

template <int HD>
__global__ void __launch_bounds__(ATT_THREADS) attn_decode_kernel(const AttnDecodeParams p) {
  constexpr int LD = HD + 8;                 // padded bf16 row: conflict-free 16-byte reads
  constexpr int KG = ATT_THREADS / (HD / 2);  // key groups in the P V phase
  extern __shared__ uint4 att_dyn[];
  bf16* sK = reinterpret_cast<bf16*>(att_dyn);  // [ATT_SPLIT][LD]
  bf16* sV = sK + ATT_SPLIT * LD;              // [ATT_SPLIT][LD]
  __shared__ __align__(16) float q_s[ATT_MAXG][HD];
  __shared__ float p_s[ATT_MAXG][ATT_SPLIT];
  __shared__ float m_s[ATT_MAXG], l_s[ATT_MAXG];
  __shared__ float2 o_red[KG > 1 ? KG - 1 : 1][ATT_MAXG][HD / 2];

  pdl_trigger();
  pdl_wait();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.n_q / p.kv.n_kv;
  const int ctx = p.seq_lens[b] + 1;
  const int s0 = split * p.split_len;
  const int s1 = min(ctx, s0 + p.split_len);
  if (s0 >= s1) return;  // the combine step reads only splits below ctx
  const int n = s1 - s0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // 1. all K/V loads of the split in flight at once
  for (int c = tid; c < n * (HD / 8); c += ATT_THREADS) {
    const int r = c / (HD / 8), d8 = (c % (HD / 8)) * 8;
    const size_t kofs = p.kv.slot(b, s0 + r, 0, kvh) + d8;
    const size_t vofs = kofs + (size_t)p.kv.n_kv * p.kv.page_size * HD;  // V slab follows the K slab of the page
    att_cp16(sK + r * LD + d8, p.kv.base + kofs);
    att_cp16(sV + r * LD + d8, p.kv.base + vofs);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  const float* qg = p.q + (size_t)b * p.n_q * HD + (size_t)kvh * G * HD;
  for (int i = tid; i < G * HD; i += ATT_THREADS) q_s[i / HD][i % HD] = qg[i];
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // 2. scores: thread t <-> key s0 + t
  float acc[ATT_MAXG];
#pragma unroll
  for (int h = 0; h < ATT_MAXG; ++h) acc[h] = 0.f;
  if (tid < n) {
    const bf16* krow = sK + tid * LD;
#pragma unroll 4
    for (int d = 0; d < HD; d += 8) {
      const uint4 kw = *reinterpret_cast<const uint4*>(krow + d);
      const float k0 = bf_lo(kw.x), k1 = bf_hi(kw.x), k2 = bf_lo(kw.y), k3 = bf_hi(kw.y);
      const float k4 = bf_lo(kw.z), k5 = bf_hi(kw.z), k6 = bf_lo(kw.w), k7 = bf_hi(kw.w);
#pragma unroll
      for (int h = 0; h < ATT_MAXG; ++h) {
        if (h < G) {
          const float4 qa = *reinterpret_cast<const float4*>(&q_s[h][d]);
          const float4 qb = *reinterpret_cast<const float4*>(&q_s[h][d + 4]);
          acc[h] += qa.x * k0 + qa.y * k1 + qa.z * k2 + qa.w * k3 + qb.x * k4 + qb.y * k5 + qb.z * k6 + qb.w * k7;
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < ATT_MAXG; ++h)
    if (h < G) p_s[h][tid] = tid < n ? acc[h] * p.scale : -INFINITY;
  __syncthreads();

  // 3. softmax statistics per head (warp w: heads w, w + 4)
  for (int h = warp; h < G; h += ATT_THREADS / 32) {
    float v[4];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = p_s[h][lane + 32 * i];
      m = fmaxf(m, v[i]);
    }
    m = warp_max(m);
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float e = (v[i] == -INFINITY) ? 0.f : __expf(v[i] - m);
      p_s[h][lane + 32 * i] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) {
      m_s[h] = m;
      l_s[h] = l;
    }
  }
  __syncthreads();

  // 4. P V: thread (dim pair dp, key group kg) over keys kg, kg + KG, ...
  const int dp = tid % (HD / 2), kg = tid / (HD / 2);
  float2 o[ATT_MAXG];
#pragma unroll
  for (int h = 0; h < ATT_MAXG; ++h) o[h] = make_float2(0.f, 0.f);
  for (int t = kg; t < n; t += KG) {
    const uint32_t vv = *reinterpret_cast<const uint32_t*>(sV + t * LD + 2 * dp);
    const float v0 = bf_lo(vv), v1 = bf_hi(vv);
#pragma unroll
    for (int h = 0; h < ATT_MAXG; ++h) {
      if (h < G) {
        const float pw = p_s[h][t];
        o[h].x += pw * v0;
        o[h].y += pw * v1;
      }
    }
  }
  if (KG > 1) {
    if (kg > 0) {
#pragma unroll
      for (int h = 0; h < ATT_MAXG; ++h)
        if (h < G) o_red[kg - 1][h][dp] = o[h];
    }
    __syncthreads();
    if (kg != 0) return;
    for (int g2 = 0; g2 < KG - 1; ++g2) {
#pragma unroll
      for (int h = 0; h < ATT_MAXG; ++h) {
        if (h < G) {
          o[h].x += o_red[g2][h][dp].x;
          o[h].y += o_red[g2][h][dp].y;
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < ATT_MAXG; ++h) {
    if (h >= G) continue;
    const size_t idx = ((size_t)b * p.n_q + (size_t)kvh * G + h) * p.nsplit + split;
    *reinterpret_cast<float2*>(p.part_o + idx * HD + 2 * dp) = o[h];
    if (dp == 0) {
      p.part_ml[idx * 2] = m_s[h];
      p.part_ml[idx * 2 + 1] = l_s[h];
    }
  }
}

template <int HD>
__global__ void __launch_bounds__(HD) attn_combine_kernel(const AttnDecodeParams p) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int ctx = p.seq_lens[b] + 1;
  int ns = (ctx + p.split_len - 1) / p.split_len;
  if (ns > p.nsplit) ns = p.nsplit;
  const size_t base = ((size_t)b * p.n_q + h) * p.nsplit;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, p.part_ml[(base + s) * 2]);
  float L = 0.f, acc = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float m = p.part_ml[(base + s) * 2];
    const float w = __expf(m - M);
    L += w * p.part_ml[(base + s) * 2 + 1];
    acc += w * p.part_o[(base + s) * HD + d];
  }
  p.out[(size_t)b * p.n_q * HD + (size_t)h * HD + d] = acc / L;
}

static constexpr size_t att_dyn_smem(int hd) { return (size_t)2 * ATT_SPLIT * (hd + 8) * sizeof(bf16); }

// The K/V tiles need more than the default 48 KB of shared memory for head_dim
// 128: raise the limit once per device before the first launch there.
static cudaError_t attn_configure_current_device() {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && configured[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(attn_decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)att_dyn_smem(64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)att_dyn_smem(128));
  if (e == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = 1;
  return e;
}

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int B, int n_kv, int hd, cudaStream_t s, bool pdl) {
  if (p.split_len != ATT_SPLIT) return cudaErrorInvalidValue;
  cudaError_t e = attn_configure_current_device();
  if (e != cudaSuccess) return e;
  const dim3 grid(p.nsplit, n_kv, B);
  if (hd == 64) {
    e = launch_k(attn_decode_kernel<64>, grid, dim3(ATT_THREADS), att_dyn_smem(64), s, pdl, p);
    if (e == cudaSuccess) e = launch_k(attn_combine_kernel<64>, dim3(p.n_q, B), dim3(64), 0, s, pdl, p);
  } else {
    e = launch_k(attn_decode_kernel<128>, grid, dim3(ATT_THREADS), att_dyn_smem(128), s, pdl, p);
    if (e == cudaSuccess) e = launch_k(attn_combine_kernel<128>, dim3(p.n_q, B), dim3(128), 0, s, pdl, p);
  }
  return e;
}

// ---------------------------------------------------------------------------
// Greedy token: argmax over the vocabulary, lowest index on ties, NaN ignored.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__global__ void __launch_bounds__(256) argmax_partial_kernel(const float* __restrict__ logits, int V,
                                                             float* pv, int* pi, int nblk) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y, blk = blockIdx.x;
  const int chunk = (V + nblk - 1) / nblk;
  const int lo = blk * chunk, hi = min(V, lo + chunk);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) better(bv, bi, logits[(size_t)b * V + i], i);
  __shared__ float sv[32];
  __shared__ int si[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) better(bv, bi, sv[w], si[w]);
    pv[b * nblk + blk] = bv;
    pi[b * nblk + blk] = bi;
  }
}

__global__ void argmax_final_kernel(const float* pv, const int* pi, int nblk, int* out) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, lane = threadIdx.x;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = lane; i < nblk; i += 32) better(bv, bi, pv[b * nblk + i], pi[b * nblk + i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  if (lane == 0) out[b] = bi == 0x7fffffff ? 0 : bi;
}

cudaError_t launch_argmax(const float* logits, int B, int V, float* part_v, int* part_i, int nblk,
                          int* out, cudaStream_t s, bool pdl) {
  cudaError_t e = launch_k(argmax_partial_kernel, dim3(nblk, B), dim3(256), 0, s, pdl, logits, V, part_v, part_i, nblk);
  if (e == cudaSuccess) e = launch_k(argmax_final_kernel, dim3(B), dim3(32), 0, s, pdl, (const float*)part_v,
                                     (const int*)part_i, nblk, out);
  return e;
}

// ---------------------------------------------------------------------------
// Small bookkeeping kernels
// ---------------------------------------------------------------------------
__global__ void advance_kernel(int* seq_lens, int B) {
  pdl_trigger();
  pdl_wait();
  const int b = threadIdx.x;
  if (b < B) seq_lens[b] += 1;
}

cudaError_t launch_advance(int* seq_lens, int B, cudaStream_t s, bool pdl) {
  return launch_k(advance_kernel, dim3(1), dim3(64), 0, s, pdl, seq_lens, B);
}

// cos/sin of p * theta^(-2j/hd), formed in double precision and rounded once.
__global__ void rope_table_kernel(float* c, float* sn, int max_seq, int hd, double theta) {
  const int half = hd / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)max_seq * half) return;
  const int p = (int)(idx / half), j = (int)(idx % half);
  const double inv = pow(theta, -2.0 * (double)j / (double)hd);
  const double a = (double)p * inv;
  c[idx] = (float)cos(a);
  sn[idx] = (float)sin(a);
}

cudaError_t launch_rope_tables(float* cos_t, float* sin_t, int max_seq, int hd, float theta,
                               cudaStream_t s) {
  const long long n = (long long)max_seq * (hd / 2);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(cos_t, sin_t, max_seq, hd, (double)theta);
  return cudaGetLastError();
}

}  // namespace ladder
