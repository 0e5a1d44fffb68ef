// Decode-side kernels of the Ladder Transformer forward pass (one new token per
// sequence, B <= 64 sequences): embedding gather (with the prefill variant that
// also leaves the RMSNorm inputs of the first modules), paged split-context
// attention and its combine step, greedy argmax, and small bookkeeping kernels.
// The decode projections are in gemv.cu.
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

// Prefill embedding with the RMSNorm outputs of the modules that read x_0 (see
// NormOut): thread t holds 8 consecutive columns, so a 128-column entry of the
// sums of squares is sixteen neighbouring lanes, whose partial sums meet by four
// shuffles (in a fixed order); d is a multiple of 256, so every warp's lanes are
// all in or all out of each pass.
template <typename WT>
__global__ void embed_norm_kernel(const int* __restrict__ tok, const WT* __restrict__ E, int d, int vocab,
                                  float* __restrict__ x, const NormOut no, int* err) {
  using C = W16<WT>;
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  const int t = tok[m];
  const bool ok = (unsigned)t < (unsigned)vocab;
  if (!ok && threadIdx.x == 0) atomicOr(err, ERR_TOKEN);
  const WT* row = E + (size_t)(ok ? t : 0) * d;
  float* out = x + (size_t)m * d;
  for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
    const uint4 v = ok ? *reinterpret_cast<const uint4*>(row + i) : make_uint4(0, 0, 0, 0);
    const float f[8] = {C::lo(v.x), C::hi(v.x), C::lo(v.y), C::hi(v.y), C::lo(v.z), C::hi(v.z), C::lo(v.w), C::hi(v.w)};
    *reinterpret_cast<float4*>(out + i) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(out + i + 4) = make_float4(f[4], f[5], f[6], f[7]);
    if (!no.ss) continue;
    float sq = ((f[0] * f[0] + f[1] * f[1]) + (f[2] * f[2] + f[3] * f[3])) +
               ((f[4] * f[4] + f[5] * f[5]) + (f[6] * f[6] + f[7] * f[7]));
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sq += __shfl_xor_sync(0xffffffffu, sq, 4);
    sq += __shfl_xor_sync(0xffffffffu, sq, 8);
    if ((threadIdx.x & 15) == 0) no.ss[(size_t)(i >> 7) * no.ld_ss + m] = sq;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (!no.u[k]) continue;
      const uint4 gr = *reinterpret_cast<const uint4*>(static_cast<const WT*>(no.g[k]) + i);
      const float g[8] = {C::lo(gr.x), C::hi(gr.x), C::lo(gr.y), C::hi(gr.y),
                          C::lo(gr.z), C::hi(gr.z), C::lo(gr.w), C::hi(gr.w)};
      float u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) u[j] = f[j] * g[j];
      uint4 hi;
      hi.x = C::pack(u[0], u[1]);
      hi.y = C::pack(u[2], u[3]);
      hi.z = C::pack(u[4], u[5]);
      hi.w = C::pack(u[6], u[7]);
      WT* dst = static_cast<WT*>(no.u[k]) + (size_t)m * d + i;
      *reinterpret_cast<uint4*>(dst) = hi;
      if (no.u_lo) {
        uint4 lo;
        lo.x = C::pack(u[0] - C::lo(hi.x), u[1] - C::hi(hi.x));
        lo.y = C::pack(u[2] - C::lo(hi.y), u[3] - C::hi(hi.y));
        lo.z = C::pack(u[4] - C::lo(hi.z), u[5] - C::hi(hi.z));
        lo.w = C::pack(u[6] - C::lo(hi.w), u[7] - C::hi(hi.w));
        *reinterpret_cast<uint4*>(dst + no.u_lo) = lo;
      }
    }
  }
}

cudaError_t launch_embed_norm(const int* tok, int M, const void* E, int wdt, int d, int vocab, float* x,
                              const NormOut& no, int* err, cudaStream_t s, bool pdl) {
  if (M <= 0) return cudaSuccess;
  if (wdt == WDT_F16)
    return launch_k(embed_norm_kernel<f16>, dim3(M), dim3(128), 0, s, pdl, tok, static_cast<const f16*>(E), d, vocab,
                    x, no, err);
  return launch_k(embed_norm_kernel<bf16>, dim3(M), dim3(128), 0, s, pdl, tok, static_cast<const bf16*>(E), d, vocab,
                  x, no, err);
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

template <typename KT, int HD>
__global__ void __launch_bounds__(ATT_THREADS) attn_decode_kernel(const AttnDecodeParams p) {
  using C = W16<KT>;
  constexpr int LD = HD + 8;                 // padded 16-bit row: conflict-free 16-byte reads
  constexpr int KG = ATT_THREADS / (HD / 2);  // key groups in the P V phase
  extern __shared__ uint4 att_dyn[];
  KT* sK = reinterpret_cast<KT*>(att_dyn);  // [ATT_SPLIT][LD]
  KT* sV = sK + ATT_SPLIT * LD;            // [ATT_SPLIT][LD]
  const KT* kvbase = static_cast<const KT*>(p.kv.base);
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
    att_cp16(sK + r * LD + d8, kvbase + kofs);
    att_cp16(sV + r * LD + d8, kvbase + vofs);
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
    const KT* krow = sK + tid * LD;
#pragma unroll 4
    for (int d = 0; d < HD; d += 8) {
      const uint4 kw = *reinterpret_cast<const uint4*>(krow + d);
      const float k0 = C::lo(kw.x), k1 = C::hi(kw.x), k2 = C::lo(kw.y), k3 = C::hi(kw.y);
      const float k4 = C::lo(kw.z), k5 = C::hi(kw.z), k6 = C::lo(kw.w), k7 = C::hi(kw.w);
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
    const float v0 = C::lo(vv), v1 = C::hi(vv);
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
  const size_t base = ((size_t)b * p.n_q + h) * p.nsplit;
  constexpr int CB = 16;
  if (p.nsplit <= CB) {
    // Every partial is requested at once, together with the length (one memory
    // round trip); splits past the context are masked by selection, and the
    // arithmetic is that of the loop below, in the same order.
    float m[CB], l[CB], o[CB];
#pragma unroll
    for (int s = 0; s < CB; ++s) {
      if (s < p.nsplit) {
        m[s] = p.part_ml[(base + s) * 2];
        l[s] = p.part_ml[(base + s) * 2 + 1];
        o[s] = p.part_o[(base + s) * HD + d];
      }
    }
    const int ctx = p.seq_lens[b] + 1;
    int ns = (ctx + p.split_len - 1) / p.split_len;
    if (ns > p.nsplit) ns = p.nsplit;
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < CB; ++s)
      if (s < ns) M = fmaxf(M, m[s]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int s = 0; s < CB; ++s) {
      if (s < ns) {
        const float w = __expf(m[s] - M);
        L += w * l[s];
        acc += w * o[s];
      }
    }
    p.out[(size_t)b * p.n_q * HD + (size_t)h * HD + d] = acc / L;
    return;
  }
  const int ctx = p.seq_lens[b] + 1;
  int ns = (ctx + p.split_len - 1) / p.split_len;
  if (ns > p.nsplit) ns = p.nsplit;
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
  e = cudaFuncSetAttribute(attn_decode_kernel<bf16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)att_dyn_smem(64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<bf16, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)att_dyn_smem(128));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<f16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)att_dyn_smem(64));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<f16, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)att_dyn_smem(128));
  if (e == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = 1;
  return e;
}

template <typename KT, int HD>
static cudaError_t attn_decode_go(const AttnDecodeParams& p, int B, int n_kv, cudaStream_t s, bool pdl) {
  const dim3 grid(p.nsplit, n_kv, B);
  cudaError_t e = launch_k(attn_decode_kernel<KT, HD>, grid, dim3(ATT_THREADS), att_dyn_smem(HD), s, pdl, p);
  if (e == cudaSuccess) e = launch_k(attn_combine_kernel<HD>, dim3(p.n_q, B), dim3(HD), 0, s, pdl, p);
  return e;
}

cudaError_t launch_attn_combine(const AttnDecodeParams& p, int B, int hd, cudaStream_t s, bool pdl) {
  if (hd == 64) return launch_k(attn_combine_kernel<64>, dim3(p.n_q, B), dim3(64), 0, s, pdl, p);
  return launch_k(attn_combine_kernel<128>, dim3(p.n_q, B), dim3(128), 0, s, pdl, p);
}

cudaError_t launch_attn_decode(const AttnDecodeParams& p, int B, int n_kv, int hd, int kv_dtype, cudaStream_t s,
                               bool pdl) {
  if (p.split_len != ATT_SPLIT) return cudaErrorInvalidValue;
  cudaError_t e = attn_configure_current_device();
  if (e != cudaSuccess) return e;
  if (kv_dtype == WDT_F16)
    return hd == 64 ? attn_decode_go<f16, 64>(p, B, n_kv, s, pdl) : attn_decode_go<f16, 128>(p, B, n_kv, s, pdl);
  return hd == 64 ? attn_decode_go<bf16, 64>(p, B, n_kv, s, pdl) : attn_decode_go<bf16, 128>(p, B, n_kv, s, pdl);
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

// x_out[b, n] = x_res[b, n] + sum_s part[b][s][n] (fixed order): the on-device
// stand-in for the all-reduce of tensor parallelism in shard mode.
__global__ void shard_reduce_kernel(const float* __restrict__ part, int k, int d, const float* __restrict__ x_res,
                                    float* __restrict__ x_out) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.y;
  const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (n >= d) return;
  float4 acc = *reinterpret_cast<const float4*>(x_res + (size_t)b * d + n);
  const float* pb = part + (size_t)b * k * d + n;
  for (int s = 0; s < k; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(pb + (size_t)s * d);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  *reinterpret_cast<float4*>(x_out + (size_t)b * d + n) = acc;
}

cudaError_t launch_shard_reduce(const float* part, int k, int B, int d, const float* x_res, float* x_out,
                                cudaStream_t s, bool pdl) {
  const int threads = 128;
  return launch_k(shard_reduce_kernel, dim3((d / 4 + threads - 1) / threads, B), dim3(threads), 0, s, pdl, part, k,
                  d, x_res, x_out);
}

cudaError_t launch_advance(int* seq_lens, int B, cudaStream_t s, bool pdl) {
  return launch_k(advance_kernel, dim3(1), dim3(64), 0, s, pdl, seq_lens, B);
}

// cos/sin of p * theta^(-2j/hd), formed in double precision and rounded once.
__global__ void rope_table_kernel(float* c, float* sn, int max_seq, int hd, double theta, RopeScaling sc) {
  const int half = hd / 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)max_seq * half) return;
  const int p = (int)(idx / half), j = (int)(idx % half);
  double inv = pow(theta, -2.0 * (double)j / (double)hd);
  if (sc.factor > 1.0) {  // Llama-3.1 frequency scaling by wavelength band
    const double w = 2.0 * 3.14159265358979323846 / inv, L = sc.original_max_pos;
    if (w > L / sc.low_freq_factor) {
      inv = inv / sc.factor;
    } else if (w >= L / sc.high_freq_factor) {
      const double s = (L / w - sc.low_freq_factor) / (sc.high_freq_factor - sc.low_freq_factor);
      inv = (1.0 - s) * inv / sc.factor + s * inv;
    }
  }
  const double a = (double)p * inv;
  c[idx] = (float)cos(a);
  sn[idx] = (float)sin(a);
}

cudaError_t launch_rope_tables(float* cos_t, float* sin_t, int max_seq, int hd, float theta, RopeScaling sc,
                               cudaStream_t s) {
  const long long n = (long long)max_seq * (hd / 2);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(cos_t, sin_t, max_seq, hd, (double)theta, sc);
  return cudaGetLastError();
}

}  // namespace ladder
