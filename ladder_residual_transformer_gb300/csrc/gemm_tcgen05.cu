// Prefill projection GEMM on the 5th-generation tensor cores (sm_103a):
//   C[m, n] = sum_k A[m, k] * W[n, k],  A = bf16 activations [M, K],
//   W = bf16 weights [N, K] (both K-major), fp32 accumulation in TMEM.
//
// One CTA computes a 128 x 256 tile with tcgen05.mma (cta_group::1, kind::f16,
// M = 128, N = 256, K = 16 per instruction).  Warp roles:
//   warp 4: one elected thread issues the TMA loads of A (128 x 64) and of the
//           two 128-row halves of B (each half may come from a different
//           weight matrix: q/k/v rows, or the gate and up rows of SwiGLU);
//   warp 5: allocates 256 TMEM columns and one elected thread issues the MMAs,
//           releasing each shared-memory stage with tcgen05.commit;
//   warps 0-3: epilogue, reading the accumulator with tcgen05.ld (warp w owns
//           TMEM lanes 32w..32w+31, i.e. tile rows) and applying the fused
//           RoPE + KV scatter, SwiGLU, or residual add.
// Operands sit in shared memory in the 128-byte-swizzled K-major layout that
// TMA writes and the MMA descriptors describe.  Every mbarrier wait is bounded
// by a clock limit: on expiry the kernel sets bit 1 of the error word, stops
// issuing work, and still frees its TMEM before returning.
#include "internal.cuh"

#include <cuda.h>
#include <string.h>

namespace ladder {

constexpr int TC_BM = 128, TC_BN = 256, TC_BK = 64, TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;   // 16 KB
constexpr int TC_BH_BYTES = 128 * TC_BK * 2;    // one 128-row half of B, 16 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + 2 * TC_BH_BYTES;
constexpr int TC_SMEM = TC_STAGES * TC_STAGE_BYTES + 1024 + 256;
constexpr int TC_THREADS = 192;
constexpr long long TC_WAIT_LIMIT = 4000000000LL;  // cycles (about 2 s)

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Wait for the phase of parity `parity` to complete; false after the clock limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  const long long start = clock64();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if (clock64() - start > TC_WAIT_LIMIT) return false;
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c_inner, int c_row,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c_inner), "r"(c_row), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
  d |= (uint64_t)1 << 46;            // version
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: A and B of format `fmt` (0 = f16, 1 = bf16),
// fp32 D, both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, uint32_t fmt) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// B-operand half selection: (tensor map index, first row) of tile half h.
// Returns false when the half lies beyond N (QKV only) and must be ignored.
// ---------------------------------------------------------------------------
template <int MODE>
__device__ __forceinline__ bool b_half(const GemmParams& p, int tile_n, int h, int& map, int& row) {
  if (MODE == GEMM_GATEUP) {
    map = h;
    row = tile_n * 128;
    return true;
  }
  const int c = tile_n * TC_BN + h * 128;
  if (MODE == GEMM_RESID) {
    map = 0;
    row = c;
    return true;
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

template <typename WT, int MODE>
__global__ void __launch_bounds__(TC_THREADS, 1) gemm_tc_kernel(const __grid_constant__ TcMaps maps,
                                                                const GemmParams p, int* err) {
  using C = W16<WT>;
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TC_STAGES * TC_STAGE_BYTES);
  uint64_t* empty = full + TC_STAGES;
  uint64_t* accum = empty + TC_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  int* bail = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_n = blockIdx.x, m0 = blockIdx.y * TC_BM;
  const int nkb = p.K / TC_BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *bail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TC_BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0) {
      int map0, row0, map1, row1;
      b_half<MODE>(p, tile_n, 0, map0, row0);
      if (!b_half<MODE>(p, tile_n, 1, map1, row1)) { map1 = map0; row1 = row0; }
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % TC_STAGES;
        const uint32_t ph = (kb / TC_STAGES) & 1;
        if (kb >= TC_STAGES && !mbar_wait(&empty[s], ph ^ 1)) {
          atomicOr(err, 2);
          *reinterpret_cast<volatile int*>(bail) = 1;
          break;
        }
        if (*reinterpret_cast<volatile int*>(bail)) break;
        uint8_t* st = smem + s * TC_STAGE_BYTES;
        mbar_expect_tx(&full[s], TC_STAGE_BYTES);
        tma_load_2d(st, &maps.a, kb * TC_BK, m0, &full[s]);
        tma_load_2d(st + TC_A_BYTES, &maps.b[map0], kb * TC_BK, row0, &full[s]);
        tma_load_2d(st + TC_A_BYTES + TC_BH_BYTES, &maps.b[map1], kb * TC_BK, row1, &full[s]);
        ++issued;
      }
      // Make sure no copy into this CTA's shared memory is still in flight.
      for (int kb = issued - TC_STAGES < 0 ? 0 : issued - TC_STAGES; kb < issued; ++kb)
        mbar_wait(&full[kb % TC_STAGES], (kb / TC_STAGES) & 1);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc(TC_BM, TC_BN, C::umma_fmt);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % TC_STAGES;
        const uint32_t ph = (kb / TC_STAGES) & 1;
        if (!mbar_wait(&full[s], ph)) {
          atomicOr(err, 2);
          *reinterpret_cast<volatile int*>(bail) = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + s * TC_STAGE_BYTES);
        const uint32_t b_base = a_base + TC_A_BYTES;
#pragma unroll
        for (int kk = 0; kk < TC_BK / 16; ++kk)
          umma_bf16(tmem, umma_desc(a_base + kk * 32), umma_desc(b_base + kk * 32), idesc, (kb | kk) != 0);
        umma_commit(&empty[s]);
      }
      umma_commit(accum);  // also issued after a bail, so that the MMAs in flight finish first
    }
  } else {
    const bool ok = mbar_wait(accum, 0);
    tc_fence_after();
    if (!ok) {
      if (lane == 0) atomicOr(err, 2);
    } else if (!__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(bail), 0)) {
      const int m = m0 + warp * 32 + lane;
      const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
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
        for (int c = 0; c < TC_BN / 32; ++c) {
          float v[32];
          tmem_ld32(trow + c * 32, v);
          if (m < p.M) {
            const size_t off = (size_t)m * p.ldo + (size_t)tile_n * TC_BN + c * 32;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 r = *reinterpret_cast<const float4*>(p.x_res + off + j);
              *reinterpret_cast<float4*>(p.out_f + off + j) =
                  make_float4(r.x + v[j], r.y + v[j + 1], r.z + v[j + 2], r.w + v[j + 3]);
            }
          }
        }
      } else {  // GEMM_QKV
        const int hd = p.kv.head_dim;
        const int pos = m < p.M ? p.row_pos[m] : 0;
        const int b = m < p.M ? p.row_b[m] : 0;
        for (int c = 0; c < TC_BN / 32; ++c) {
          float v[32];
          tmem_ld32(trow + c * 32, v);
          int map, row;
          if (!b_half<GEMM_QKV>(p, tile_n, c >> 2, map, row) || m >= p.M) continue;
          // q and the KV cache are bf16 whatever the weight type (the attention kernels read bf16)
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
          bf16* dst = map == 0 ? static_cast<bf16*>(p.out_h) + (size_t)m * p.ldo + local
                               : p.kv.base + p.kv.slot(b, pos, map - 1, head) + dim0;
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 pk;
            __nv_bfloat162 t0 = __floats2bfloat162_rn(v[j], v[j + 1]);
            __nv_bfloat162 t1 = __floats2bfloat162_rn(v[j + 2], v[j + 3]);
            __nv_bfloat162 t2 = __floats2bfloat162_rn(v[j + 4], v[j + 5]);
            __nv_bfloat162 t3 = __floats2bfloat162_rn(v[j + 6], v[j + 7]);
            pk.x = *reinterpret_cast<uint32_t*>(&t0);
            pk.y = *reinterpret_cast<uint32_t*>(&t1);
            pk.z = *reinterpret_cast<uint32_t*>(&t2);
            pk.w = *reinterpret_cast<uint32_t*>(&t3);
            *reinterpret_cast<uint4*>(dst + j) = pk;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_BN) : "memory");
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

template <typename WT>
static cudaError_t gemm_tc_configure_t() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_QKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  return cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_RESID>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
}

cudaError_t gemm_tc_configure() {
  cudaError_t e = gemm_tc_configure_t<bf16>();
  return e != cudaSuccess ? e : gemm_tc_configure_t<f16>();
}

template <typename WT>
static void gemm_tc_dispatch(const TcMaps& maps, const GemmParams& p, int mode, int mt, int* err, cudaStream_t s) {
  if (mode == GEMM_GATEUP) {
    gemm_tc_kernel<WT, GEMM_GATEUP><<<dim3(p.N / 128, mt), TC_THREADS, TC_SMEM, s>>>(maps, p, err);
  } else if (mode == GEMM_RESID) {
    gemm_tc_kernel<WT, GEMM_RESID><<<dim3(p.N / TC_BN, mt), TC_THREADS, TC_SMEM, s>>>(maps, p, err);
  } else {
    gemm_tc_kernel<WT, GEMM_QKV><<<dim3((p.N + TC_BN - 1) / TC_BN, mt), TC_THREADS, TC_SMEM, s>>>(maps, p, err);
  }
}

cudaError_t launch_gemm_tc(const void* a_map, const void* b0, const void* b1, const void* b2, const GemmParams& p,
                           int mode, int wdt, int* err, cudaStream_t s) {
  if (p.M <= 0) return cudaSuccess;
  TcMaps maps;
  memcpy(&maps.a, a_map, sizeof(CUtensorMap));
  memcpy(&maps.b[0], b0, sizeof(CUtensorMap));
  memcpy(&maps.b[1], b1 ? b1 : b0, sizeof(CUtensorMap));
  memcpy(&maps.b[2], b2 ? b2 : b0, sizeof(CUtensorMap));
  const int mt = (p.M + TC_BM - 1) / TC_BM;
  if (wdt == WDT_F16) gemm_tc_dispatch<f16>(maps, p, mode, mt, err, s);
  else gemm_tc_dispatch<bf16>(maps, p, mode, mt, err, s);
  return cudaGetLastError();
}

}  // namespace ladder
