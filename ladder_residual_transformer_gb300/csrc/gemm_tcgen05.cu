// Prefill projection GEMM on the 5th-generation tensor cores (sm_103a):
//   C[m, n] = sum_k A[m, k] * W[n, k],  A = bf16 activations [M, K],
//   W = bf16 weights [N, K] (both K-major), fp32 accumulation in TMEM.
//
// Persistent CTAs (one per SM) loop over 128 x BN tiles (BN = 256, or 128 for
// narrow matrices) with tcgen05.mma (cta_group::1, kind::f16, M = 128, N = BN,
// K = 16 per instruction).  Warp roles:
//   warp 4: one elected thread issues the TMA loads of A (128 x 64) and of the
//           two 128-row halves of B (each half may come from a different
//           weight matrix: q/k/v rows, or the gate and up rows of SwiGLU);
//   warp 5: allocates 2 x BN TMEM columns (two accumulator buffers) and one
//           elected thread issues the MMAs, releasing each shared-memory stage
//           with tcgen05.commit and each finished accumulator to the epilogue;
//   warps 0-3: epilogue, reading the accumulator with tcgen05.ld (warp w owns
//           TMEM lanes 32w..32w+31, i.e. tile rows) and applying the fused
//           RoPE + KV scatter, SwiGLU, or residual add, then handing the
//           accumulator buffer back, so the epilogue of one tile overlaps the
//           main loop of the next.
// Operands sit in shared memory in the 128-byte-swizzled K-major layout that
// TMA writes and the MMA descriptors describe.  Every mbarrier wait is bounded
// by a clock limit: on expiry the kernel sets bit 1 of the error word, stops
// issuing work, and still frees its TMEM before returning.
#include "internal.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <string.h>

namespace ladder {

constexpr int TC_BM = 128, TC_BK = 64;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;   // 16 KB
constexpr int TC_BH_BYTES = 128 * TC_BK * 2;    // one 128-row half of B, 16 KB
// Shared memory for the stage ring: 7 stages of 32 KB at BN = 128, 4 of 48 KB at BN = 256.
constexpr int TC_SMEM = 7 * (TC_A_BYTES + TC_BH_BYTES) + 1024 + 256;
constexpr int TC_THREADS = 192;
constexpr long long TC_WAIT_LIMIT = 4000000000LL;  // cycles (about 2 s)

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait(bar, parity, TC_WAIT_LIMIT);
}

// K-major operand tile in the 128-byte-swizzled layout that TMA writes: 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) { return umma_desc_sw128(saddr, 16, 1024); }

// ---------------------------------------------------------------------------
// B-operand half selection: (tensor map index, first row) of 128-row half h of
// N-tile `tile_n` (tiles are BN wide; GATEUP tiles are 128 outputs = gate half
// + up half).  Returns false when the half lies beyond N and must be ignored.
// ---------------------------------------------------------------------------
template <int MODE, int BN>
__device__ __forceinline__ bool b_half(const GemmParams& p, int tile_n, int h, int& map, int& row) {
  if (MODE == GEMM_GATEUP) {
    map = h;
    row = tile_n * 128;
    return true;
  }
  const int c = tile_n * BN + h * 128;
  if (MODE == GEMM_RESID) {
    map = 0;
    row = c;
    return c < p.N;
  }
  if (c < p.nq_hd) { map = 0; row = c; return true; }
  if (c < p.nq_hd + p.nkv_hd) { map = 1; row = c - p.nq_hd; return true; }
  if (c < p.N) { map = 2; row = c - p.nq_hd - p.nkv_hd; return true; }
  map = 0;
  row = 0;
  return false;
}

struct TcMaps {
  CUtensorMap a;
  CUtensorMap b[3];
};

// Persistent CTA: tiles t = blockIdx.x + i * gridDim.x, tile t -> (m = t % m_tiles,
// n = t / m_tiles) so that CTAs running together share the weight tile in L2.
// The accumulator is double-buffered in TMEM (2 x BN columns): the MMA warp
// fills buffer i & 1 while the epilogue warps drain the other one.
template <typename WT, int MODE, int BN>
__global__ void __launch_bounds__(TC_THREADS, 1) gemm_tc_kernel(const __grid_constant__ TcMaps maps,
                                                                const GemmParams p, int m_tiles, int n_tiles,
                                                                int* err) {
  using C = W16<WT>;
  constexpr int HALVES = BN / 128;
  constexpr int STAGE = TC_A_BYTES + HALVES * TC_BH_BYTES;
  constexpr int NST = (TC_SMEM - 1024 - 256) / STAGE;
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * STAGE);
  uint64_t* empty = full + NST;
  uint64_t* tfull = empty + NST;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;    // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* bail = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = p.K / TC_BK;
  const int total = m_tiles * n_tiles;
  const int my_tiles = blockIdx.x < total ? (total - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
    }
    *bail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      int it = 0;  // running k-block index across tiles
      bool ok = true;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int t = blockIdx.x + i * gridDim.x;
        const int m0 = (t % m_tiles) * TC_BM, tn = t / m_tiles;
        int map0, row0, map1 = 0, row1 = 0;
        b_half<MODE, BN>(p, tn, 0, map0, row0);
        if (HALVES == 2 && !b_half<MODE, BN>(p, tn, 1, map1, row1)) { map1 = map0; row1 = row0; }
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (it >= NST && !mbar_wait(&empty[s], ph ^ 1)) {
            atomicOr(err, 2);
            *reinterpret_cast<volatile int*>(bail) = 1;
            ok = false;
            break;
          }
          if (*reinterpret_cast<volatile int*>(bail)) { ok = false; break; }
          uint8_t* st = smem + s * STAGE;
          mbar_expect_tx(&full[s], STAGE);
          tma_load_2d(st, &maps.a, kb * TC_BK, m0, &full[s]);
          tma_load_2d(st + TC_A_BYTES, &maps.b[map0], kb * TC_BK, row0, &full[s]);
          if (HALVES == 2) tma_load_2d(st + TC_A_BYTES + TC_BH_BYTES, &maps.b[map1], kb * TC_BK, row1, &full[s]);
        }
      }
      // Make sure no copy into this CTA's shared memory is still in flight.
      for (int k = it - NST < 0 ? 0 : it - NST; k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc(TC_BM, BN, C::umma_fmt);
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int acc = i & 1;
        if (i >= 2 && !mbar_wait(&tempty[acc], ((i >> 1) - 1) & 1)) {
          atomicOr(err, 2);
          *reinterpret_cast<volatile int*>(bail) = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % NST;
          const uint32_t ph = (it / NST) & 1;
          if (!mbar_wait(&full[s], ph)) {
            atomicOr(err, 2);
            *reinterpret_cast<volatile int*>(bail) = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * STAGE);
          const uint32_t b_base = a_base + TC_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            umma_f16(d, umma_desc(a_base + kk * 32), umma_desc(b_base + kk * 32), idesc, (kb | kk) != 0);
          umma_commit(&empty[s]);
        }
        umma_commit(&tfull[acc]);  // also after a bail, so that the MMAs in flight finish first
      }
    }
  } else {
    const int hd = p.kv.head_dim;
    for (int i = 0; i < my_tiles; ++i) {
      const int acc = i & 1;
      const int t = blockIdx.x + i * gridDim.x;
      const int m = (t % m_tiles) * TC_BM + warp * 32 + lane, tile_n = t / m_tiles;
      const bool ok = mbar_wait(&tfull[acc], (i >> 1) & 1);
      tc_fence_after();
      if (!ok) {
        if (lane == 0) atomicOr(err, 2);
        break;
      }
      if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(bail), 0)) break;
      const uint32_t trow = tmem + acc * BN + ((uint32_t)(warp * 32) << 16);
      if (MODE == GEMM_GATEUP) {
        for (int c = 0; c < 4; ++c) {
          float g[32], u[32];
          tmem_ld32(trow + c * 32, g);
          tmem_ld32(trow + 128 + c * 32, u);
          if (m < p.M) {
            WT* dst = static_cast<WT*>(p.out_h) + (size_t)m * p.ldo + tile_n * 128 + c * 32;
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 pk;
              pk.x = C::pack(silu_f(g[j]) * u[j], silu_f(g[j + 1]) * u[j + 1]);
              pk.y = C::pack(silu_f(g[j + 2]) * u[j + 2], silu_f(g[j + 3]) * u[j + 3]);
              pk.z = C::pack(silu_f(g[j + 4]) * u[j + 4], silu_f(g[j + 5]) * u[j + 5]);
              pk.w = C::pack(silu_f(g[j + 6]) * u[j + 6], silu_f(g[j + 7]) * u[j + 7]);
              *reinterpret_cast<uint4*>(dst + j) = pk;
            }
          }
        }
      } else if (MODE == GEMM_RESID) {
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(trow + c * 32, v);
          const int n0 = tile_n * BN + c * 32;
          if (m < p.M && n0 < p.N) {
            const size_t off = (size_t)m * p.ldo + n0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 r = *reinterpret_cast<const float4*>(p.x_res + off + j);
              *reinterpret_cast<float4*>(p.out_f + off + j) =
                  make_float4(r.x + v[j], r.y + v[j + 1], r.z + v[j + 2], r.w + v[j + 3]);
            }
          }
        }
      } else {  // GEMM_QKV
        const int pos = m < p.M ? p.row_pos[m] : 0;
        const int b = m < p.M ? p.row_b[m] : 0;
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(trow + c * 32, v);
          int map, row;
          if (!b_half<GEMM_QKV, BN>(p, tile_n, c >> 2, map, row) || m >= p.M) continue;
          const int local = row + (c & 3) * 32;  // first column of the chunk inside its matrix
          const int head = local / hd, dim0 = local % hd;
          if (map < 2) {
            const float* cs = p.rope_cos + (size_t)pos * (hd >> 1) + (dim0 >> 1);
            const float* sn = p.rope_sin + (size_t)pos * (hd >> 1) + (dim0 >> 1);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float cj = cs[j >> 1], sj = sn[j >> 1];
              const float a0 = v[j], a1 = v[j + 1];
              v[j] = a0 * cj - a1 * sj;
              v[j + 1] = a0 * sj + a1 * cj;
            }
          }
          // q, K and V are stored in the weight dtype (the attention operands)
          WT* dst = map == 0 ? static_cast<WT*>(p.out_h) + (size_t)m * p.ldo + local
                             : static_cast<WT*>(p.kv.base) + p.kv.slot(b, pos, map - 1, head) + dim0;
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 pk;
            pk.x = C::pack(v[j], v[j + 1]);
            pk.y = C::pack(v[j + 2], v[j + 3]);
            pk.z = C::pack(v[j + 4], v[j + 5]);
            pk.w = C::pack(v[j + 6], v[j + 7]);
            *reinterpret_cast<uint4*>(dst + j) = pk;
          }
        }
      }
      // hand the accumulator buffer back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty[acc])) : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BN) : "memory");
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Row-major 16-bit [rows, cols] matrix, box of 128 rows x 64 columns, 128-byte swizzle.
bool make_tma_map(void* map_out, const void* base, uint64_t rows, uint64_t cols, int wdt) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows % 128 || cols % 64 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {TC_BK, 128};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = wdt == WDT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(map_out), dt, 2, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One layer of the paged KV pool viewed as [pages * 2 * n_kv][page_size][hd]
// 16-bit elements; box = 64 elements x page_size slots x 1, 128-byte swizzle.
bool make_kv_tma_map(void* map_out, const void* base, uint64_t num_pages, int n_kv, int page_size, int hd, int wdt) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || hd % 64 || page_size < 8 || page_size > 256 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)page_size, num_pages * 2 * (cuuint64_t)n_kv};
  cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)page_size * hd * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)page_size, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = wdt == WDT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(map_out), dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename WT>
static cudaError_t gemm_tc_configure_t() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_QKV, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_QKV, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_GATEUP, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_RESID, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  return cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_RESID, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
}

cudaError_t gemm_tc_configure() {
  cudaError_t e = gemm_tc_configure_t<bf16>();
  return e != cudaSuccess ? e : gemm_tc_configure_t<f16>();
}

template <typename WT, int MODE, int BN>
static cudaError_t gemm_tc_go(const TcMaps& maps, const GemmParams& p, int mt, int nt, int num_sms, int* err,
                              cudaStream_t s) {
  const int total = mt * nt;
  const int grid = total < num_sms ? total : num_sms;
  gemm_tc_kernel<WT, MODE, BN><<<grid, TC_THREADS, TC_SMEM, s>>>(maps, p, mt, nt, err);
  return cudaGetLastError();
}

// 256-wide tiles unless that leaves most SMs idle (narrow N at small M).
template <typename WT>
static cudaError_t gemm_tc_dispatch(const TcMaps& maps, const GemmParams& p, int mode, int mt, int num_sms, int* err,
                                    cudaStream_t s) {
  if (mode == GEMM_GATEUP) return gemm_tc_go<WT, GEMM_GATEUP, 256>(maps, p, mt, p.N / 128, num_sms, err, s);
  const int nt256 = (p.N + 255) / 256;
  const bool narrow = (long long)mt * nt256 * 4 < (long long)num_sms * 3;
  if (mode == GEMM_RESID) {
    if (narrow) return gemm_tc_go<WT, GEMM_RESID, 128>(maps, p, mt, (p.N + 127) / 128, num_sms, err, s);
    return gemm_tc_go<WT, GEMM_RESID, 256>(maps, p, mt, nt256, num_sms, err, s);
  }
  if (narrow) return gemm_tc_go<WT, GEMM_QKV, 128>(maps, p, mt, (p.N + 127) / 128, num_sms, err, s);
  return gemm_tc_go<WT, GEMM_QKV, 256>(maps, p, mt, nt256, num_sms, err, s);
}

cudaError_t launch_gemm_tc(const void* a_map, const void* b0, const void* b1, const void* b2, const GemmParams& p,
                           int mode, int wdt, int num_sms, int* err, cudaStream_t s) {
  if (p.M <= 0) return cudaSuccess;
  TcMaps maps;
  memcpy(&maps.a, a_map, sizeof(CUtensorMap));
  memcpy(&maps.b[0], b0, sizeof(CUtensorMap));
  memcpy(&maps.b[1], b1 ? b1 : b0, sizeof(CUtensorMap));
  memcpy(&maps.b[2], b2 ? b2 : b0, sizeof(CUtensorMap));
  const int mt = (p.M + TC_BM - 1) / TC_BM;
  return wdt == WDT_F16 ? gemm_tc_dispatch<f16>(maps, p, mode, mt, num_sms, err, s)
                        : gemm_tc_dispatch<bf16>(maps, p, mode, mt, num_sms, err, s);
}

}  // namespace ladder
