// Next-token sampling with temperature and top-k.
//
// The generation loop of the Ladder Residual paper's benchmark code
// (logits_to_probs / multinomial_sample_one_no_sync / sample, named in the
// paper's codewithpapers record) scales the logits by 1/T, keeps those at or
// above the k-th largest, normalises them to probabilities p and returns
// argmax_i p_i / q_i with q_i ~ Exp(1): an "exponential race", which is a
// sample of p.  Written in the log domain it is an argmax,
//     token = argmax_{i : l_i >= pivot} l_i / T - ln(q_i),   q_i = -ln(u_i),
// so the sampler is a selection (the pivot) followed by one argmax pass, with
// no softmax and no sort.
//
// The uniforms u_i come from SplitMix64 counters (Steele, Lea and Flood,
// "Fast splittable pseudorandom number generators", OOPSLA 2014), keyed by the
// seed, the batch row and the position of the token being sampled:
//     key = mix(mix(seed + G (row + 1)) + G (pos + 1)),
//     u_i = (top 23 bits of mix(key + G (i + 1)) + 1/2) / 2^23,
// G = 0x9E3779B97F4A7C15, mix = the SplitMix64 output function.  Every u_i lies
// in (0, 1) and is exact in fp32.
//
// One CTA of 1024 threads per batch row (the logits row, 0.5 MB for a 128k
// vocabulary, is L2-resident after the lm_head GEMV):
//   1. radix select of the k-th largest logit on order-preserving 32-bit keys,
//      8 bits per pass, most significant first (4 passes over the row); each
//      warp keeps its own 256-bin histogram and adds the lanes that share a
//      bin with one shared-memory atomic (__match_any_sync);
//   2. one pass that scores the candidates (key >= pivot key) and keeps the
//      largest score, the lowest index on ties.
// Histogram counts are integers and the argmax is order-independent, so the
// result does not depend on scheduling.
#include "internal.cuh"

namespace ladder {

namespace {

constexpr int SAMPLE_THREADS = 1024;
constexpr int SAMPLE_WARPS = SAMPLE_THREADS / 32;
constexpr uint64_t SM64_GAMMA = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Order-preserving map of an fp32 value to an unsigned key (a > b <=> key(a) > key(b)).
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(SAMPLE_THREADS) sample_kernel(const float* __restrict__ logits, int V,
                                                                float inv_t, int top_k, uint64_t seed,
                                                                const int* __restrict__ pos, int pos_off,
                                                                int* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned hist[SAMPLE_WARPS][256];
  __shared__ float s_best[SAMPLE_WARPS];
  __shared__ int s_best_i[SAMPLE_WARPS];
  __shared__ uint32_t s_sel[2];  // chosen prefix, remaining rank
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* l = logits + (size_t)b * V;

  // 1. pivot key = key of the k-th largest logit (0: every logit is a candidate)
  uint32_t prefix = 0;
  if (top_k > 0 && top_k < V) {
    uint32_t mask = 0, remaining = (uint32_t)top_k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int j = lane; j < 256; j += 32) hist[warp][j] = 0u;
      __syncwarp();
      for (int base = warp * 32; base < V; base += SAMPLE_THREADS) {
        const int i = base + lane;
        const uint32_t key = i < V ? order_key(l[i]) : 0u;
        const bool in = i < V && (key & mask) == prefix;
        const uint32_t bin = (key >> shift) & 255u;
        const unsigned act = __ballot_sync(0xffffffffu, in);
        if (in) {
          const unsigned peers = __match_any_sync(act, bin);
          if (lane == __ffs(peers) - 1) atomicAdd(&hist[warp][bin], (unsigned)__popc(peers));
        }
      }
      __syncthreads();
      // bin totals (thread j owns bin j)
      if (tid < 256) {
        unsigned t = 0;
        for (int w = 0; w < SAMPLE_WARPS; ++w) t += hist[w][tid];
        hist[0][tid] = t;
      }
      __syncthreads();
      // the largest bin j with count(bins >= j) >= remaining; lane L scans bins 8L..8L+7
      if (warp == 0) {
        unsigned own[8], s = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          own[q] = hist[0][8 * lane + q];
          s += own[q];
        }
        unsigned suffix = s;  // inclusive suffix sum over lanes >= this lane
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const unsigned t = __shfl_down_sync(0xffffffffu, suffix, off);
          if (lane + off < 32) suffix += t;
        }
        unsigned above = suffix - s;  // candidates in higher lanes' bins
        int found = -1;
        unsigned rem_out = 0;
#pragma unroll
        for (int q = 7; q >= 0; --q) {
          if (found < 0) {
            const unsigned c = above + own[q];
            if (c >= remaining) {
              found = 8 * lane + q;
              rem_out = remaining - above;
            }
            above = c;
          }
        }
        const unsigned has = __ballot_sync(0xffffffffu, found >= 0);
        const int src = 31 - __clz((int)has);  // the highest lane holding a satisfying bin
        const int fb = __shfl_sync(0xffffffffu, found, src);
        const unsigned fr = __shfl_sync(0xffffffffu, rem_out, src);
        if (lane == 0) {
          s_sel[0] = (uint32_t)(has ? fb : 0);
          s_sel[1] = has ? fr : 1u;
        }
      }
      __syncthreads();
      prefix |= s_sel[0] << shift;
      mask |= 255u << shift;
      remaining = s_sel[1];
      __syncthreads();  // s_sel and hist are reused by the next pass
    }
  }
  const uint32_t pivot = prefix;

  // 2. argmax of l_i / T - ln(-ln u_i) over the candidates
  const uint64_t k1 = sm64_mix(seed + SM64_GAMMA * (uint64_t)(b + 1));
  const uint64_t key = sm64_mix(k1 + SM64_GAMMA * (uint64_t)(pos[b] + pos_off + 1));
  float best = -INFINITY;
  int best_i = 0x7fffffff;
  for (int i = tid; i < V; i += SAMPLE_THREADS) {
    const float x = l[i];
    if (order_key(x) >= pivot) {
      const uint64_t h = sm64_mix(key + SM64_GAMMA * (uint64_t)(i + 1));
      const float u = ((float)(uint32_t)(h >> 41) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
      const float sc = x * inv_t - logf(-logf(u));
      if (sc > best || (sc == best && i < best_i)) {
        best = sc;
        best_i = i;
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, off);
    const int oi = __shfl_xor_sync(0xffffffffu, best_i, off);
    if (ob > best || (ob == best && oi < best_i)) {
      best = ob;
      best_i = oi;
    }
  }
  if (lane == 0) {
    s_best[warp] = best;
    s_best_i[warp] = best_i;
  }
  __syncthreads();
  if (tid == 0) {
    float bv = s_best[0];
    int bi = s_best_i[0];
    for (int w = 1; w < SAMPLE_WARPS; ++w)
      if (s_best[w] > bv || (s_best[w] == bv && s_best_i[w] < bi)) {
        bv = s_best[w];
        bi = s_best_i[w];
      }
    out[b] = bi;
  }
}

}  // namespace

cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k, uint64_t seed,
                          const int* pos, int pos_off, int* out, cudaStream_t s, bool pdl) {
  if (B <= 0) return cudaSuccess;
  if (!(temperature > 0.f) || V <= 0) return cudaErrorInvalidValue;
  const float t = temperature < 1e-5f ? 1e-5f : temperature;
  return launch_k(sample_kernel, dim3(B), dim3(SAMPLE_THREADS), 0, s, pdl, logits, V, 1.0f / t, top_k, seed, pos,
                  pos_off, out);
}

}  // namespace ladder
