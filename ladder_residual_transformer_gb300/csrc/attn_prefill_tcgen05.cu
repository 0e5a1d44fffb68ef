// Causal grouped-query attention for prefill on the 5th-generation tensor
// cores (tcgen05 + TMA + TMEM).
//
// CTA = (128-query block, query head, sequence).  Keys are visited in tiles of
// 128 up to the diagonal; for key tile j
//   S_j  = Q K_j^T                        tcgen05.mma, M=128, N=128, K=head_dim -> TMEM
//   P_j  = exp2(S_j * scale * log2(e) - m) softmax warps, written to shared memory
//   O   += P_j V_j                         tcgen05.mma, M=128, N=head_dim, K=128 -> TMEM
// with the online-softmax reference m kept per query row.  m is raised (and O
// and the row sum rescaled) only when a tile's row maximum exceeds it by more
// than 8 in log2 units, so P stays below 2^8 and most tiles skip the rescale;
// the result is the same softmax because O and the row sum always share one
// reference.
//
// Warp roles (192 threads):
//   warps 0-3  softmax + epilogue, thread r owns query row r (TMEM lane r);
//   warp 4     issues the TMA copies: the Q tile once, then K and V tiles
//              page by page from the paged KV cache into a ring of stages
//              (3-D tensor map over [page*2*n_kv + kv*n_kv + head][slot][dim]),
//              one lane per page of the tile;
//   warp 5     allocates TMEM (S double buffer + O) and one thread issues the
//              MMAs: S_{j+1} is issued before PV_j so that the tensor cores
//              compute the next scores while the softmax warps work on P_j.
// Operands sit in shared memory in the 128-byte-swizzled layout TMA writes:
// Q, K and P are K-major; V is read as an MN-major operand straight from its
// [key][dim] rows, so no transpose is needed.
//
// Keys past the sequence end inside the last tile are masked out of S, and the
// softmax warps zero their V rows, so stale cache contents never reach O.
// Every wait is bounded: on expiry the kernel sets bit 1 of the error word and
// winds down without touching further memory.
#include "internal.cuh"
#include "tcgen05.cuh"

#include <math.h>
#include <string.h>

namespace ladder {

constexpr int FT_BM = 128;        // query rows per CTA = TMEM lanes
constexpr int FT_BN = 128;        // keys per tile
constexpr int FT_THREADS = 192;
constexpr int FT_BLK = 128 * 128; // one 128-row x 64-element swizzled block, bytes
constexpr long long FT_WAIT_LIMIT = 4000000000LL;

template <int HD>
struct FtCfg {
  static constexpr int NB = HD / 64;              // 64-element column blocks of a row
  static constexpr int STAGES = HD == 64 ? 3 : 2; // K/V ring depth
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = NB * FT_BLK;
  static constexpr int STAGE_BYTES = 2 * NB * FT_BLK;  // K then V
  static constexpr int P_OFF = KV_OFF + STAGES * STAGE_BYTES;
  static constexpr int P_BYTES = 2 * FT_BLK;            // 128 rows x 128 keys
  static constexpr int BAR_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;     // + barriers + alignment slack
};

struct FtMaps {
  CUtensorMap q;   // [rows][n_q * hd], box 64 x 128
  CUtensorMap kv;  // [pages * 2 * n_kv][page_size][hd], box 64 x page_size x 1
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T, int HD>
__global__ void __launch_bounds__(FT_THREADS, 1)
    attn_prefill_tcgen05_kernel(const __grid_constant__ FtMaps maps, const AttnPrefillParams p, int nqb, int B,
                                int* err) {
  using C = W16<T>;
  using L = FtCfg<HD>;
  constexpr int NB = L::NB, ST = L::STAGES;
  extern __shared__ uint8_t ft_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ft_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;        // [ST]
  uint64_t* kv_empty = kv_full + ST;   // [ST]
  uint64_t* s_full = kv_empty + ST;    // [2]
  uint64_t* s_empty = s_full + 2;      // [2]
  uint64_t* p_full = s_empty + 2;      // [2]
  uint64_t* pv_done = p_full + 2;      // [2]
  uint64_t* mma_done = pv_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* bail = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // Heaviest query blocks (most key tiles) first.
  const int per_qb = p.n_q * B;
  const int qb = nqb - 1 - (int)(blockIdx.x / per_qb);
  const int rem = (int)(blockIdx.x % per_qb);
  const int h = rem % p.n_q, b = rem / p.n_q;
  const int Tn = p.seq_len[b];
  if (qb * FT_BM >= Tn) return;
  const int start = p.seq_start[b];
  const int kvh = h / (p.n_q / p.kv.n_kv);
  const int n_kb = qb + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(mma_done, 1);
    *bail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + 256;
  // Launched early (programmatic dependent launch), the prologue above overlaps
  // the previous kernel; no thread touches global memory before it completes.
  pdl_wait();

  if (warp == 4) {
    // Lane c < nch issues the K and V boxes of page chunk c of the tile; the
    // page ids of tile j + 1 are read while tile j's stage is awaited, so the
    // block-table latency stays off the copy path.
    const int ps = p.kv.page_size, cpt = FT_BN / ps;
    const int npg = (Tn + ps - 1) / ps;  // pages holding the sequence
    const int* btr = p.kv.block_table + (size_t)b * p.kv.max_pages;
    if (lane == 0) {
      mbar_expect_tx(q_full, NB * FT_BLK);
      for (int c = 0; c < NB; ++c)
        tma_load_2d(smem + L::Q_OFF + c * FT_BLK, &maps.q, h * HD + c * 64, start + qb * FT_BM, q_full);
    }
    int pg = lane < cpt && lane < npg ? btr[lane] : 0;
    int j = 0;
    for (; j < n_kb; ++j) {
      const int s = j % ST;
      const int nidx = (j + 1) * cpt + lane;
      const int pg_next = j + 1 < n_kb && lane < cpt && nidx < npg ? btr[nidx] : 0;
      bool ok = j < ST || mbar_wait(&kv_empty[s], ((j / ST) - 1) & 1, FT_WAIT_LIMIT);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) {
        atomicOr(err, 2);
        *bail = 1;
      }
      if (__shfl_sync(0xffffffffu, (int)(!ok || *bail), 0)) break;
      const int key0 = j * FT_BN;
      int nch = (Tn - key0 + ps - 1) / ps;
      if (nch > cpt) nch = cpt;
      if (lane == 0) mbar_expect_tx(&kv_full[s], (uint32_t)(nch * ps * 128 * NB * 2));
      __syncwarp();
      if (lane < nch) {
        uint8_t* kdst = smem + L::KV_OFF + s * L::STAGE_BYTES + lane * ps * 128;
        uint8_t* vdst = kdst + NB * FT_BLK;
        const int zk = (pg * 2) * p.kv.n_kv + kvh, zv = zk + p.kv.n_kv;
        for (int blk = 0; blk < NB; ++blk) {
          tma_load_3d(kdst + blk * FT_BLK, &maps.kv, blk * 64, 0, zk, &kv_full[s]);
          tma_load_3d(vdst + blk * FT_BLK, &maps.kv, blk * 64, 0, zv, &kv_full[s]);
        }
      }
      pg = pg_next;
    }
    // No copy into this CTA's shared memory may be in flight at exit.
    if (lane == 0) {
      mbar_wait(q_full, 0, FT_WAIT_LIMIT);
      for (int k = j - ST < 0 ? 0 : j - ST; k < j; ++k) mbar_wait(&kv_full[k % ST], (k / ST) & 1, FT_WAIT_LIMIT);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc(FT_BM, FT_BN, C::umma_fmt);
      constexpr uint32_t idesc_o = umma_idesc(FT_BM, HD, C::umma_fmt, 1);
      const uint32_t q_base = smem_u32(smem + L::Q_OFF);
      bool ok = mbar_wait(q_full, 0, FT_WAIT_LIMIT);
      for (int j = 0; ok && j <= n_kb; ++j) {
        if (j < n_kb) {
          const int s = j % ST, sb = j & 1;
          if (!mbar_wait(&kv_full[s], (j / ST) & 1, FT_WAIT_LIMIT) ||
              (j >= 2 && !mbar_wait(&s_empty[sb], ((j >> 1) - 1) & 1, FT_WAIT_LIMIT)) || *bail) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_base = smem_u32(smem + L::KV_OFF + s * L::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * FT_BLK + (kk & 3) * 32;
            umma_f16(tmem + sb * FT_BN, umma_desc_sw128(q_base + off, 16, 1024),
                     umma_desc_sw128(k_base + off, 16, 1024), idesc_s, kk != 0);
          }
          umma_commit(&s_full[sb]);
        }
        if (j >= 1) {
          const int i = j - 1, pb = i & 1, s = i % ST;
          if (!mbar_wait(&p_full[pb], (i >> 1) & 1, FT_WAIT_LIMIT) || *bail) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t p_base = smem_u32(smem + L::P_OFF + pb * L::P_BYTES);
          const uint32_t v_base = smem_u32(smem + L::KV_OFF + s * L::STAGE_BYTES + NB * FT_BLK);
#pragma unroll
          for (int t = 0; t < FT_BN / 16; ++t) {
            umma_f16(tmem_o, umma_desc_sw128(p_base + (t >> 2) * FT_BLK + (t & 3) * 32, 16, 1024),
                     umma_desc_sw128(v_base + t * 2048, FT_BLK, 1024), idesc_o, (i | t) != 0);
          }
          umma_commit(&pv_done[pb]);
          umma_commit(&kv_empty[s]);
        }
      }
      if (!ok) {
        atomicOr(err, 2);
        *bail = 1;
      }
      // every MMA issued above has completed before TMEM is released
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, FT_WAIT_LIMIT);
    }
  } else {
    // softmax warps: thread r owns query row r
    const int r = threadIdx.x;
    const int q = qb * FT_BM + r;
    const int lim = q < Tn - 1 ? q : Tn - 1;  // last key this row may attend to
    const float sl2 = p.scale * 1.4426950408889634f;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m_ref = 0.f, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kb; ++j) {
      const int sb = j & 1, pb = j & 1;
      ok = mbar_wait(&s_full[sb], (j >> 1) & 1, FT_WAIT_LIMIT);
      ok = __all_sync(0xffffffffu, ok) && !*bail;
      if (!ok) break;
      tc_fence_after();
      float sv[FT_BN];
      tmem_ld128(tmem + lane_base + sb * FT_BN, sv);
      // S buffer sb may be overwritten by S_{j+2}
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[sb]);

      const int key0 = j * FT_BN;
      if (j == n_kb - 1) {
#pragma unroll
        for (int e = 0; e < FT_BN; ++e)
          if (key0 + e > lim) sv[e] = -INFINITY;
      }
      // row maximum: eight independent chains, then a tree
      float m8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) m8[e] = sv[e];
#pragma unroll
      for (int e = 8; e < FT_BN; ++e) m8[e & 7] = fmaxf(m8[e & 7], sv[e]);
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mt = mx * sl2;
      bool rescale = false;
      float corr = 1.f;
      if (j == 0) {
        m_ref = mt;
      } else if (mt > m_ref + 8.f) {
        corr = ex2_approx(m_ref - mt);
        l_sum *= corr;
        m_ref = mt;
        rescale = true;
      }
      // P buffer pb was last read by PV_{j-2}
      if (j >= 2) {
        ok = mbar_wait(&pv_done[pb], ((j >> 1) - 1) & 1, FT_WAIT_LIMIT);
        ok = __all_sync(0xffffffffu, ok) && !*bail;
        if (!ok) break;
      }
      uint8_t* prow = smem + L::P_OFF + pb * L::P_BYTES + r * 128;
      float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c8 = 0; c8 < FT_BN / 8; ++c8) {
        float pv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          pv[e] = ex2_approx(fmaf(sv[c8 * 8 + e], sl2, -m_ref));
          r8[e] += pv[e];
        }
        uint4 pk;
        pk.x = C::pack(pv[0], pv[1]);
        pk.y = C::pack(pv[2], pv[3]);
        pk.z = C::pack(pv[4], pv[5]);
        pk.w = C::pack(pv[6], pv[7]);
        const int blk = c8 >> 3, chunk = c8 & 7;
        *reinterpret_cast<uint4*>(prow + blk * FT_BLK + ((chunk ^ (r & 7)) << 4)) = pk;
      }
      const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
      l_sum += rs;
      // keys past the sequence end: zero their V rows (the MMA multiplies them by P = 0)
      if (j == n_kb - 1 && Tn - key0 < FT_BN) {
        const int s = j % ST;
        ok = mbar_wait(&kv_full[s], (j / ST) & 1, FT_WAIT_LIMIT);
        ok = __all_sync(0xffffffffu, ok) && !*bail;
        if (!ok) break;
        if (key0 + r >= Tn) {
          uint8_t* vrow = smem + L::KV_OFF + s * L::STAGE_BYTES + NB * FT_BLK + r * 128;
#pragma unroll
          for (int blk = 0; blk < NB; ++blk)
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + blk * FT_BLK + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold PV_{j-1} before it is rescaled
        const int i = j - 1;
        ok = mbar_wait(&pv_done[i & 1], (i >> 1) & 1, FT_WAIT_LIMIT);
        ok = __all_sync(0xffffffffu, ok) && !*bail;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          float o[32];
          tmem_ld32(tmem_o + lane_base + c * 32, o);
          if (rescale) {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= corr;
          }
          tmem_st32(tmem_o + lane_base + c * 32, o);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    if (ok) {
      const int i = n_kb - 1;
      ok = mbar_wait(&pv_done[i & 1], (i >> 1) & 1, FT_WAIT_LIMIT);
      ok = __all_sync(0xffffffffu, ok) && !*bail;
    }
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l_sum;
      T* dst = static_cast<T*>(p.out) + (size_t)(start + q) * ((size_t)p.n_q * HD) + (size_t)h * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        float o[32];
        tmem_ld32(tmem_o + lane_base + c * 32, o);
        if (q < Tn) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = o[e + i] * inv;
            uint4 pk;
            pk.x = C::pack(v[0], v[1]);
            pk.y = C::pack(v[2], v[3]);
            pk.z = C::pack(v[4], v[5]);
            pk.w = C::pack(v[6], v[7]);
            *reinterpret_cast<uint4*>(dst + c * 32 + e) = pk;
            if (p.lo_off) {  // rounding remainders into the lo plane (hi/lo operand of the O projection)
              uint4 pl;
              pl.x = C::pack(v[0] - C::lo(pk.x), v[1] - C::hi(pk.x));
              pl.y = C::pack(v[2] - C::lo(pk.y), v[3] - C::hi(pk.y));
              pl.z = C::pack(v[4] - C::lo(pk.z), v[5] - C::hi(pk.z));
              pl.w = C::pack(v[6] - C::lo(pk.w), v[7] - C::hi(pk.w));
              *reinterpret_cast<uint4*>(dst + p.lo_off + c * 32 + e) = pl;
            }
          }
        }
      }
    } else if (lane == 0) {
      atomicOr(err, 2);
      *bail = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t attn_prefill_tcgen05_smem(int hd) { return hd == 64 ? FtCfg<64>::SMEM : FtCfg<128>::SMEM; }

template <typename T>
static cudaError_t ft_configure_t() {
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_tcgen05_kernel<T, 64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, FtCfg<64>::SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_prefill_tcgen05_kernel<T, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FtCfg<128>::SMEM);
}

cudaError_t attn_prefill_tcgen05_configure() {
  cudaError_t e = ft_configure_t<bf16>();
  return e != cudaSuccess ? e : ft_configure_t<f16>();
}

template <typename T>
static cudaError_t ft_dispatch(const FtMaps& maps, const AttnPrefillParams& p, int hd, int nqb, int B, int* err,
                               cudaStream_t s, bool pdl) {
  const unsigned grid = (unsigned)nqb * p.n_q * B;
  if (hd == 64)
    return launch_k(attn_prefill_tcgen05_kernel<T, 64>, dim3(grid), dim3(FT_THREADS), (size_t)FtCfg<64>::SMEM, s, pdl,
                    maps, p, nqb, B, err);
  return launch_k(attn_prefill_tcgen05_kernel<T, 128>, dim3(grid), dim3(FT_THREADS), (size_t)FtCfg<128>::SMEM, s, pdl,
                  maps, p, nqb, B, err);
}

cudaError_t launch_attn_prefill_tcgen05(const void* q_map, const void* kv_map, const AttnPrefillParams& p, int hd,
                                        int wdt, int B, int max_len, int* err, cudaStream_t s, bool pdl) {
  if (max_len <= 0) return cudaSuccess;
  if (hd != 64 && hd != 128) return cudaErrorInvalidValue;
  FtMaps maps;
  memcpy(&maps.q, q_map, sizeof(CUtensorMap));
  memcpy(&maps.kv, kv_map, sizeof(CUtensorMap));
  const int nqb = (max_len + FT_BM - 1) / FT_BM;
  return wdt == WDT_F16 ? ft_dispatch<f16>(maps, p, hd, nqb, B, err, s, pdl)
                        : ft_dispatch<bf16>(maps, p, hd, nqb, B, err, s, pdl);
}

}  // namespace ladder
