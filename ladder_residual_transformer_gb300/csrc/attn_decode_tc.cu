// Decode attention (one new query per sequence) over the paged KV cache, on
// the tensor cores, split along the context like attn_decode_kernel.
//
// CTA = (128-key split, KV head, sequence), 4 warps.  One thread issues the
// TMA copies of the split's K and V pages (3-D map of the pool, 128-byte
// swizzle: [64-dim block][key][64 dims]); the G = n_q / n_kv query heads of the
// group, pre-scaled by scale * log2(e), sit as rows 0..G-1 of a 16-row 16-bit
// tile, and their rounding remainders (also 16-bit) as rows 8..8+G-1: the MMA's
// idle padding rows carry the lo half of a hi/lo pair, so S = Q_hi K^T + Q_lo
// K^T is a sum of two accumulator rows that one thread already holds (about 22
// significant bits of q at no extra tensor-core work; G <= 8).  Warp w computes
// S = Q K^T for keys 32w..32w+31 with mma.sync m16n8k16 (K fragments by
// ldmatrix from the swizzled tile), the row maxima and sums are combined across
// the warps through shared memory, P is written to shared memory as the same
// hi/lo row pair, and warp w computes O = P V for a quarter of the head
// dimensions (V fragments by ldmatrix.trans), adding the two rows of each pair.
// Keys past the context are masked in S and their V rows zeroed.  The per-split partials (unnormalised O, max in
// natural-log units, sum) feed the same combine kernel as attn_decode_kernel.
// Every wait is bounded (bit 1 of the error word on expiry).
#include "internal.cuh"
#include "tcgen05.cuh"

#include <math.h>
#include <string.h>

namespace ladder {

constexpr int AD_KEYS = 128;     // keys per split
constexpr int AD_THREADS = 128;  // 4 warps
constexpr int AD_BLK = 128 * 128; // one [128 keys][64 dims] 16-bit block, bytes
constexpr long long AD_WAIT_LIMIT = 2000000000LL;

template <int HD>
struct AdCfg {
  static constexpr int NB = HD / 64;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = NB * AD_BLK;
  static constexpr int LDQ = HD + 8;           // padded 16-bit rows: conflict-free ldmatrix
  static constexpr int Q_OFF = 2 * NB * AD_BLK;
  static constexpr int LDP = AD_KEYS + 8;
  static constexpr int P_OFF = Q_OFF + 16 * LDQ * 2;
  static constexpr int RED_OFF = P_OFF + 16 * LDP * 2;  // [2][4 warps][8 rows] floats
  static constexpr int BAR_OFF = RED_OFF + 2 * 4 * 8 * 4;
  static constexpr int SMEM = BAR_OFF + 16 + 1024;      // + alignment slack
};

__device__ __forceinline__ void ad_ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ad_ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
__device__ __forceinline__ void ad_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  if constexpr (W16<T>::umma_fmt == 1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Byte offset of (key, dim) in a swizzled [64-dim block][128 keys][64 dims] tile.
__device__ __forceinline__ uint32_t ad_swz(int key, int dim) {
  return (uint32_t)((dim >> 6) * AD_BLK + key * 128 + ((((dim & 63) >> 3) ^ (key & 7)) << 4) + ((dim & 7) << 1));
}

template <typename T, int HD>
__global__ void __launch_bounds__(AD_THREADS) attn_decode_tc_kernel(const __grid_constant__ CUtensorMap kv_map,
                                                                   const AttnDecodeParams p, int* err) {
  using C = W16<T>;
  using L = AdCfg<HD>;
  constexpr int NB = L::NB;
  extern __shared__ uint8_t ad_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ad_smem_raw) + 1023) & ~uintptr_t(1023));
  T* sQ = reinterpret_cast<T*>(smem + L::Q_OFF);
  T* sP = reinterpret_cast<T*>(smem + L::P_OFF);
  float* red_m = reinterpret_cast<float*>(smem + L::RED_OFF);  // [4][8]
  float* red_l = red_m + 32;                                   // [4][8]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);

  pdl_trigger();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  const int G = p.n_q / p.kv.n_kv;
  const int ctx = p.seq_lens[b] + 1;
  const int s0 = split * AD_KEYS;
  if (s0 >= ctx) return;  // the combine step reads only splits below ctx (uniform over the CTA)
  const int n = min(AD_KEYS, ctx - s0);
  __syncthreads();  // barrier initialised

  // 1. K and V pages of the split: one TMA box per (page, kv, 64-dim block).
  const int ps = p.kv.page_size;
  const int nch = (n + ps - 1) / ps;
  if (tid == 0) {
    mbar_expect_tx(bar, (uint32_t)(nch * ps * 128 * NB * 2));
    const int* btr = p.kv.block_table + (size_t)b * p.kv.max_pages + s0 / ps;
    for (int c = 0; c < nch; ++c) {
      const int page = btr[c];
      const int zk = (page * 2) * p.kv.n_kv + kvh, zv = zk + p.kv.n_kv;
      for (int blk = 0; blk < NB; ++blk) {
        tma_load_3d(smem + L::K_OFF + blk * AD_BLK + c * ps * 128, &kv_map, blk * 64, 0, zk, bar);
        tma_load_3d(smem + L::V_OFF + blk * AD_BLK + c * ps * 128, &kv_map, blk * 64, 0, zv, bar);
      }
    }
  }
  // 2. Queries of the group, pre-scaled for exp2: rows 0..G-1 the 16-bit values
  //    (hi), rows 8..8+G-1 their rounding remainders (lo), other rows zero.
  const float qs = p.scale * 1.4426950408889634f;
  const float* qg = p.q + (size_t)b * p.n_q * HD + (size_t)kvh * G * HD;
  for (int i = tid; i < 8 * (HD / 2); i += AD_THREADS) {
    const int r = i / (HD / 2), d2 = (i % (HD / 2)) * 2;
    float2 v = make_float2(0.f, 0.f);
    if (r < G) v = *reinterpret_cast<const float2*>(qg + r * HD + d2);
    const float a = v.x * qs, c = v.y * qs;
    const uint32_t hi = C::pack(a, c);
    *reinterpret_cast<uint32_t*>(sQ + r * L::LDQ + d2) = hi;
    *reinterpret_cast<uint32_t*>(sQ + (r + 8) * L::LDQ + d2) = C::pack(a - C::lo(hi), c - C::hi(hi));
  }
  const bool ok = mbar_wait(bar, 0, AD_WAIT_LIMIT);
  // keys past the context: zero their V rows (they meet P = 0)
  for (int i = tid; i < (AD_KEYS - n) * NB * 8; i += AD_THREADS) {
    const int key = n + i / (NB * 8), c16 = i % (NB * 8);
    *reinterpret_cast<uint4*>(smem + L::V_OFF + (c16 >> 3) * AD_BLK + key * 128 + (c16 & 7) * 16) =
        make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (!__syncthreads_and(ok)) {
    if (tid == 0) atomicOr(err, 2);
    return;
  }
  const uint32_t kbase = smem_u32(smem + L::K_OFF), vbase = smem_u32(smem + L::V_OFF);
  const uint32_t qbase = smem_u32(sQ), pbase = smem_u32(sP);
  const int q8 = lane >> 3, r8 = lane & 7;
  const int g = lane >> 2, t4 = lane & 3;

  // 3. S = Q K^T for keys 32w .. 32w + 31 (four 8-key n tiles).
  float s[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
  for (int kt = 0; kt < HD / 16; ++kt) {
    uint32_t a0, a1, a2, a3;
    ad_ldsm_x4(a0, a1, a2, a3, qbase + (uint32_t)(((q8 & 1) * 8 + r8) * L::LDQ + kt * 16 + (q8 >> 1) * 8) * 2);
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const int key = warp * 32 + (j + (q8 >> 1)) * 8 + r8;
      uint32_t b0, b1, b2, b3;
      ad_ldsm_x4(b0, b1, b2, b3, kbase + ad_swz(key, kt * 16 + (q8 & 1) * 8));
      ad_mma<T>(s[j], a0, a1, a2, a3, b0, b1);
      ad_mma<T>(s[j + 1], a0, a1, a2, a3, b2, b3);
    }
  }
  // row g of S (thread holds keys warp*32 + j*8 + 2 t4 + {0,1}) = accumulator
  // row g (q hi) + row g + 8 (q lo)
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = warp * 32 + j * 8 + 2 * t4 + e;
      s[j][e] += s[j][e + 2];
      if (key >= n) s[j][e] = -INFINITY;
      mx = fmaxf(mx, s[j][e]);
    }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  if (t4 == 0 && g < 8) red_m[warp * 8 + g] = mx;
  __syncthreads();
  const float m = fmaxf(fmaxf(red_m[g], red_m[8 + g]), fmaxf(red_m[16 + g], red_m[24 + g]));
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float p0 = exp2f(s[j][0] - m), p1 = exp2f(s[j][1] - m);
    sum += p0 + p1;
    // row g: P rounded to 16 bits (hi); row g + 8: the rounding remainders (lo)
    const uint32_t hi = C::pack(p0, p1);
    *reinterpret_cast<uint32_t*>(sP + g * L::LDP + warp * 32 + j * 8 + 2 * t4) = hi;
    *reinterpret_cast<uint32_t*>(sP + (g + 8) * L::LDP + warp * 32 + j * 8 + 2 * t4) =
        C::pack(p0 - C::lo(hi), p1 - C::hi(hi));
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  if (t4 == 0 && g < 8) red_l[warp * 8 + g] = sum;
  __syncthreads();

  // 4. O = P V for dims warp * HD/4 .. + HD/4 (HD/32 n tiles of 8).
  constexpr int NT = HD / 32;
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  const int d0 = warp * (HD / 4);
#pragma unroll
  for (int kt = 0; kt < AD_KEYS / 16; ++kt) {
    uint32_t a0, a1, a2, a3;
    ad_ldsm_x4(a0, a1, a2, a3, pbase + (uint32_t)(((q8 & 1) * 8 + r8) * L::LDP + kt * 16 + (q8 >> 1) * 8) * 2);
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      uint32_t b0, b1, b2, b3;
      ad_ldsm_x4_t(b0, b1, b2, b3, vbase + ad_swz(kt * 16 + (q8 & 1) * 8 + r8, d0 + (j + (q8 >> 1)) * 8));
      ad_mma<T>(o[j], a0, a1, a2, a3, b0, b1);
      ad_mma<T>(o[j + 1], a0, a1, a2, a3, b2, b3);
    }
  }
  // 5. Partials of rows g < G: o unnormalised, m in natural-log units, l.
  if (g < G) {
    const size_t idx = ((size_t)b * p.n_q + (size_t)kvh * G + g) * p.nsplit + split;
#pragma unroll
    for (int j = 0; j < NT; ++j)  // row g (P hi) + row g + 8 (P lo)
      *reinterpret_cast<float2*>(p.part_o + idx * HD + d0 + j * 8 + 2 * t4) =
          make_float2(o[j][0] + o[j][2], o[j][1] + o[j][3]);
    if (warp == 0 && t4 == 0) {
      p.part_ml[idx * 2] = m * 0.6931471805599453f;
      p.part_ml[idx * 2 + 1] = red_l[g] + red_l[8 + g] + red_l[16 + g] + red_l[24 + g];
    }
  }
}

size_t attn_decode_tc_smem(int hd) { return hd == 64 ? AdCfg<64>::SMEM : AdCfg<128>::SMEM; }

template <typename T>
static cudaError_t ad_configure_t() {
  cudaError_t e = cudaFuncSetAttribute(attn_decode_tc_kernel<T, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       AdCfg<64>::SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_decode_tc_kernel<T, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              AdCfg<128>::SMEM);
}

cudaError_t attn_decode_tc_configure() {
  cudaError_t e = ad_configure_t<bf16>();
  return e != cudaSuccess ? e : ad_configure_t<f16>();
}

cudaError_t launch_attn_decode_tc(const void* kv_map, const AttnDecodeParams& p, int B, int n_kv, int hd, int wdt,
                                  int* err, cudaStream_t s, bool pdl, bool pdl_combine) {
  if (p.split_len != AD_KEYS || (hd != 64 && hd != 128) || p.n_q / n_kv > 8) return cudaErrorInvalidValue;
  CUtensorMap map;
  memcpy(&map, kv_map, sizeof(map));
  const dim3 grid(p.nsplit, n_kv, B);
  cudaError_t e;
  if (wdt == WDT_F16)
    e = hd == 64 ? launch_k(attn_decode_tc_kernel<f16, 64>, grid, dim3(AD_THREADS), (size_t)AdCfg<64>::SMEM, s, pdl, map, p, err)
                 : launch_k(attn_decode_tc_kernel<f16, 128>, grid, dim3(AD_THREADS), (size_t)AdCfg<128>::SMEM, s, pdl, map, p, err);
  else
    e = hd == 64 ? launch_k(attn_decode_tc_kernel<bf16, 64>, grid, dim3(AD_THREADS), (size_t)AdCfg<64>::SMEM, s, pdl, map, p, err)
                 : launch_k(attn_decode_tc_kernel<bf16, 128>, grid, dim3(AD_THREADS), (size_t)AdCfg<128>::SMEM, s, pdl, map, p, err);
  if (e != cudaSuccess) return e;
  return launch_attn_combine(p, B, hd, s, pdl_combine);
}

}  // namespace ladder
