// Causal grouped-query attention for prefill, on the tensor cores.
//
// CTA = (64-query block, query head, sequence); four warps of 16 query rows.
// Keys and values of the sequence are read from the paged KV cache (the QKV
// GEMM epilogue has just written them) in 64-key tiles, double-buffered with
// cp.async.  S = Q K^T and O += P V use mma.sync m16n8k16 (16-bit in, fp32
// accumulate); the softmax is the online (running max / running sum) form in
// fp32 registers, with the row reductions done by quad shuffles.  Only key
// tiles at or below the diagonal are visited; the diagonal tile is masked.
//
// This contraction is a few percent of prefill FLOPs; the projection GEMMs,
// which dominate, run on tcgen05 (gemm_tcgen05.cu).
#include "internal.cuh"

#include <math.h>

namespace ladder {

constexpr int FA_BM = 64;       // query rows per CTA
constexpr int FA_BN = 64;       // keys per tile
constexpr int FA_THREADS = 128;

__device__ __forceinline__ uint32_t fa_smem(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the destination is zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(fa_smem(dst)), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(fa_smem(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(fa_smem(p)));
}

// D += A B for one m16n8k16 tile, 16-bit A and B of type T, fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
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

// T: 16-bit type of q, K, V, P and the output (the weight dtype).
template <typename T, int HD>
__global__ void __launch_bounds__(FA_THREADS) attn_prefill_kernel(const AttnPrefillParams p) {
  using C = W16<T>;
  constexpr int LD = HD + 8;  // padded row (elements): conflict-free ldmatrix
  constexpr int KT = HD / 16; // k-steps over the head dimension
  constexpr int NT = HD / 8;  // n-tiles of the output
  extern __shared__ uint4 fa_smem_raw[];
  T* sQ = reinterpret_cast<T*>(fa_smem_raw);
  T* sK = sQ + FA_BM * LD;        // [2][FA_BN][LD]
  T* sV = sK + 2 * FA_BN * LD;    // [2][FA_BN][LD]
  const T* qsrc = static_cast<const T*>(p.q);
  const T* kvbase = static_cast<const T*>(p.kv.base);

  // The heaviest (last) query blocks of the causal triangle are scheduled first.
  const int qb = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int Tn = p.seq_len[b];
  if (qb * FA_BM >= Tn) return;
  const int start = p.seq_start[b];
  const int G = p.n_q / p.kv.n_kv, kvh = h / G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t ldq = (size_t)p.n_q * HD;

  // Q tile -> shared memory (rows beyond T are zero).
  for (int c = tid; c < FA_BM * HD / 8; c += FA_THREADS) {
    const int r = c / (HD / 8), d8 = (c % (HD / 8)) * 8;
    const int pos = qb * FA_BM + r;
    const T* src = qsrc + (size_t)(start + (pos < Tn ? pos : 0)) * ldq + (size_t)h * HD + d8;
    cp_async16(sQ + r * LD + d8, src, pos < Tn);
  }
  auto load_kv = [&](int kb, int buf) {
    T* dk = sK + buf * FA_BN * LD;
    T* dv = sV + buf * FA_BN * LD;
    for (int c = tid; c < FA_BN * HD / 8; c += FA_THREADS) {
      const int r = c / (HD / 8), d8 = (c % (HD / 8)) * 8;
      const int key = kb * FA_BN + r;
      const bool ok = key < Tn;
      const int kk = ok ? key : 0;
      cp_async16(dk + r * LD + d8, kvbase + p.kv.slot(b, kk, 0, kvh) + d8, ok);
      cp_async16(dv + r * LD + d8, kvbase + p.kv.slot(b, kk, 1, kvh) + d8, ok);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  const int n_kb = qb + 1;  // causal: key tiles 0..qb
  const float sl2 = p.scale * 1.4426950408889634f;  // softmax in base 2
  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  uint32_t qf[KT][4];
  const int row0 = warp * 16;  // this warp's first row in the tile
  const int qpos0 = qb * FA_BM + row0 + (lane >> 2);  // positions of this thread's two rows: qpos0, qpos0 + 8

  for (int kb = 0; kb < n_kb; ++kb) {
    if (kb + 1 < n_kb) load_kv(kb + 1, (kb + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        const int q = lane >> 3;
        const T* a = sQ + (row0 + (q & 1) * 8 + (lane & 7)) * LD + kt * 16 + (q >> 1) * 8;
        ldsm_x4(qf[kt][0], qf[kt][1], qf[kt][2], qf[kt][3], a);
      }
    }
    const T* K = sK + (kb & 1) * FA_BN * LD;
    const T* V = sV + (kb & 1) * FA_BN * LD;

    // S = Q K^T for 16 rows x 64 keys (8 n-tiles of 8 keys)
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const int q = lane >> 3;
        const T* bp = K + ((j + (q >> 1)) * 8 + (lane & 7)) * LD + kt * 16 + (q & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, bp);
        mma16816<T>(s[j], qf[kt][0], qf[kt][1], qf[kt][2], qf[kt][3], b0, b1);
        mma16816<T>(s[j + 1], qf[kt][0], qf[kt][1], qf[kt][2], qf[kt][3], b2, b3);
      }
    }
    // causal mask on the diagonal tile, then the online softmax update
    float mx[2] = {m_r[0], m_r[1]};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kb * FA_BN + j * 8 + 2 * (lane & 3) + (e & 1);
        const int qp = qpos0 + (e >> 1) * 8;
        float v = s[j][e] * sl2;
        if (kb == qb && key > qp) v = -INFINITY;
        s[j][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float corr[2], rs[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) corr[r] = exp2f(m_r[r] - mx[r]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = exp2f(s[j][e] - mx[e >> 1]);
        s[j][e] = pv;
        rs[e >> 1] += pv;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
      rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
      l_r[r] = l_r[r] * corr[r] + rs[r];
      m_r[r] = mx[r];
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }
    // O += P V: keys in 4 k-steps of 16, output dims in NT n-tiles
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t a0 = C::pack(s[2 * t][0], s[2 * t][1]);
      const uint32_t a1 = C::pack(s[2 * t][2], s[2 * t][3]);
      const uint32_t a2 = C::pack(s[2 * t + 1][0], s[2 * t + 1][1]);
      const uint32_t a3 = C::pack(s[2 * t + 1][2], s[2 * t + 1][3]);
#pragma unroll
      for (int j = 0; j < NT; j += 2) {
        const int q = lane >> 3;
        const T* vp = V + (t * 16 + (q & 1) * 8 + (lane & 7)) * LD + (j + (q >> 1)) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, vp);
        mma16816<T>(o[j], a0, a1, a2, a3, b0, b1);
        mma16816<T>(o[j + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();  // the buffer just read is refilled two tiles later
  }

  // normalise and store (rows beyond T are skipped)
  const float inv0 = 1.f / l_r[0], inv1 = 1.f / l_r[1];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int pos = qpos0 + r * 8;
    if (pos >= Tn) continue;
    T* dst = static_cast<T*>(p.out) + (size_t)(start + pos) * ldq + (size_t)h * HD + 2 * (lane & 3);
    const float inv = r ? inv1 : inv0;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      *reinterpret_cast<uint32_t*>(dst + j * 8) = C::pack(o[j][2 * r] * inv, o[j][2 * r + 1] * inv);
    }
  }
}

size_t attn_prefill_smem(int hd) { return (size_t)(FA_BM + 4 * FA_BN) * (hd + 8) * sizeof(bf16); }

template <typename OT>
static cudaError_t attn_prefill_configure_t() {
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<OT, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)attn_prefill_smem(64));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_prefill_kernel<OT, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)attn_prefill_smem(128));
}

cudaError_t attn_prefill_configure() {
  cudaError_t e = attn_prefill_configure_t<bf16>();
  return e != cudaSuccess ? e : attn_prefill_configure_t<f16>();
}

template <typename OT>
static void attn_prefill_dispatch(const AttnPrefillParams& p, int hd, dim3 grid, cudaStream_t s) {
  if (hd == 64) attn_prefill_kernel<OT, 64><<<grid, FA_THREADS, attn_prefill_smem(64), s>>>(p);
  else attn_prefill_kernel<OT, 128><<<grid, FA_THREADS, attn_prefill_smem(128), s>>>(p);
}

cudaError_t launch_attn_prefill_tc(const AttnPrefillParams& p, int hd, int wdt, int B, int max_len, cudaStream_t s) {
  if (max_len <= 0) return cudaSuccess;
  dim3 grid((max_len + FA_BM - 1) / FA_BM, p.n_q, B);
  if (wdt == WDT_F16) attn_prefill_dispatch<f16>(p, hd, grid, s);
  else attn_prefill_dispatch<bf16>(p, hd, grid, s);
  return cudaGetLastError();
}

}  // namespace ladder
