// Decode GEMV: out[b, n] = sum_k W[n, k] * u[b, k] for B <= 4 rows, with the
// RMSNorm prologue (u = x * rsqrt(mean(x^2) + eps) * g) and the per-module
// epilogues (RoPE + KV-cache write, SwiGLU, residual add, logits) fused.
//
// Decode is bound by HBM bandwidth: every step streams all weights once.  Each
// CTA is persistent over a contiguous range of tasks (a task is two weight
// rows: a RoPE pair, the matching gate and up rows, or two consecutive rows)
// and splits its work between
//   - one producer warp, whose elected lane streams the tasks' weight rows,
//     chunk by chunk, into a ring of shared-memory stages with cp.async.bulk
//     (completion counted on an mbarrier per stage), and
//   - four consumer warps that stage the normalised input rows once, then take
//     whole tasks round-robin, wait for each chunk's stage, accumulate the two
//     dot products in fp32 (lane l owns elements 8l + 256i of a chunk) and
//     release the stage.
// The ring is split into one sub-ring per consumer warp: every stage is filled
// and drained by the same warp, in order, so a warp never waits on a stage
// whose previous use belongs to another warp (an mbarrier parity wait only
// distinguishes consecutive phases).
// Weights depend on no earlier kernel, so the producer starts streaming at
// launch; with programmatic dependent launch this overlaps the previous
// kernel's tail.  Only the consumers wait (griddepcontrol.wait) before they
// read the stream.  The ring is sized to keep a CTA near 100 KB of shared
// memory so that CTAs of two consecutive kernels can share an SM.
// Every mbarrier wait is bounded by a clock limit; on expiry the kernel sets
// bit 2 of the error word and stops.
#include "internal.cuh"

namespace ladder {

constexpr int SG_CONSUMERS = 4;
constexpr int SG_THREADS = (SG_CONSUMERS + 1) * 32;
constexpr int SG_MAX_STAGES = 16;
constexpr int SG_RING_BYTES = 64 * 1024;
constexpr int SG_MAX_CHUNK = 2048;  // elements of K per stage and row
constexpr int SG_SMEM_LIMIT = 226 * 1024;  // dynamic shared memory cap (leaves room for the static part)
constexpr long long SG_WAIT_LIMIT = 4000000000LL;  // cycles (about 2 s)

__device__ __forceinline__ uint32_t sg_smem(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool sg_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = sg_smem(bar);
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
    if (clock64() - start > SG_WAIT_LIMIT) return false;
  }
}

template <typename WT, int BT>
__device__ __forceinline__ void sg_fma(const uint4& w, const float* __restrict__ u, int half, int k,
                                       float (&acc)[BT], int ustride) {
  using C = W16<WT>;
  const float w0 = C::lo(w.x), w1 = C::hi(w.x), w2 = C::lo(w.y), w3 = C::hi(w.y);
  const float w4 = C::lo(w.z), w5 = C::hi(w.z), w6 = C::lo(w.w), w7 = C::hi(w.w);
  const int q = (k >> 3) << 2;
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    const float4 a = *reinterpret_cast<const float4*>(u + b * ustride + q);
    const float4 c = *reinterpret_cast<const float4*>(u + b * ustride + half + q);
    float s = acc[b];
    s = fmaf(w0, a.x, s);
    s = fmaf(w1, a.y, s);
    s = fmaf(w2, a.z, s);
    s = fmaf(w3, a.w, s);
    s = fmaf(w4, c.x, s);
    s = fmaf(w5, c.y, s);
    s = fmaf(w6, c.z, s);
    s = fmaf(w7, c.w, s);
    acc[b] = s;
  }
}

// Rows of task t: (row0, row1) and, for QKV, the matrix (kind 0 q, 1 k, 2 v) and
// the first row's index inside it.
template <typename WT, int MODE>
__device__ __forceinline__ void sg_rows(const GemvParams& p, int t, const WT*& r0, const WT*& r1, int& kind,
                                        int& local) {
  const WT* W0 = static_cast<const WT*>(p.w0);
  const int K = p.K;
  kind = 0;
  local = 0;
  if (MODE == GEMV_QKV) {
    const int q0 = 2 * t;
    if (q0 < p.nq_hd) {
      local = q0; kind = 0; r0 = W0 + (size_t)local * K;
    } else if (q0 < p.nq_hd + p.nkv_hd) {
      local = q0 - p.nq_hd; kind = 1; r0 = static_cast<const WT*>(p.w1) + (size_t)local * K;
    } else {
      local = q0 - p.nq_hd - p.nkv_hd; kind = 2; r0 = static_cast<const WT*>(p.w2) + (size_t)local * K;
    }
    r1 = r0 + K;
  } else if (MODE == GEMV_GATEUP) {
    r0 = W0 + (size_t)t * K;
    r1 = static_cast<const WT*>(p.w1) + (size_t)t * K;
  } else {
    r0 = W0 + (size_t)(2 * t) * K;
    r1 = r0 + K;
  }
}

template <int MODE>
__device__ __forceinline__ void sg_epilogue(const GemvParams& p, int b, int task, int kind, int local, float v0,
                                            float v1) {
  if (MODE == GEMV_QKV) {
    const int hd = p.kv.head_dim;
    const int pos = p.pos[b];
    float r0 = v0, r1 = v1;
    if (kind < 2) {
      const int j = (local % hd) >> 1;
      const float c = p.rope_cos[(size_t)pos * (hd >> 1) + j];
      const float s = p.rope_sin[(size_t)pos * (hd >> 1) + j];
      r0 = v0 * c - v1 * s;
      r1 = v0 * s + v1 * c;
    }
    if (kind == 0) {
      *reinterpret_cast<float2*>(p.out + (size_t)b * p.ldo + local) = make_float2(r0, r1);
    } else {
      const int head = local / hd, dim = local % hd;
      *reinterpret_cast<__nv_bfloat162*>(p.kv.base + p.kv.slot(b, pos, kind - 1, head) + dim) =
          __floats2bfloat162_rn(r0, r1);
    }
  } else if (MODE == GEMV_GATEUP) {
    p.out[(size_t)b * p.ldo + task] = silu_f(v0) * v1;
  } else if (MODE == GEMV_RESID) {
    const size_t n = 2 * (size_t)task;
    const float2 r = *reinterpret_cast<const float2*>(p.x_res + (size_t)b * p.ldr + n);
    *reinterpret_cast<float2*>(p.out + (size_t)b * p.ldo + n) = make_float2(r.x + v0, r.y + v1);
  } else {
    *reinterpret_cast<float2*>(p.out + (size_t)b * p.ldo + 2 * (size_t)task) = make_float2(v0, v1);
  }
}

template <typename WT, int BT, int MODE>
__global__ void __launch_bounds__(SG_THREADS, 1) sgemv_kernel(const GemvParams p) {
  using C = W16<WT>;
  extern __shared__ __align__(128) uint8_t sg_raw[];
  const int K = p.K, kch = p.kc, nch = K / kch, nst = p.nst;
  const int stage_bytes = 4 * kch;  // two rows of kch 16-bit elements
  uint8_t* ring = sg_raw;
  float* u = reinterpret_cast<float*>(sg_raw + (size_t)nst * stage_bytes);  // [BT][K], two planes per row
  uint64_t* full = reinterpret_cast<uint64_t*>(u + (size_t)BT * K);
  uint64_t* empty = full + SG_MAX_STAGES;
  __shared__ float s_red[SG_CONSUMERS][BT];
  __shared__ float s_rms[BT];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (p.n_tasks + gridDim.x - 1) / gridDim.x;
  const int t0 = blockIdx.x * per;
  const int t1 = min(p.n_tasks, t0 + per);
  const int n_items = t1 > t0 ? (t1 - t0) * nch : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sg_smem(&full[s])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sg_smem(&empty[s])) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();

  if (warp == SG_CONSUMERS) {
    // ---------------- producer: stream weight chunks into the sub-rings ----------------
    if (lane == 0) {
      const int spw = nst / SG_CONSUMERS;  // stages per consumer warp
      int cnt[SG_CONSUMERS] = {0, 0, 0, 0};  // chunks issued to each warp's sub-ring
      bool ok = true;
      for (int ti = 0; ok && ti < t1 - t0; ++ti) {
        const int w = ti % SG_CONSUMERS;
        const WT *r0, *r1;
        int kind, local;
        sg_rows<WT, MODE>(p, t0 + ti, r0, r1, kind, local);
        for (int c = 0; c < nch; ++c) {
          const int j = cnt[w];
          const int s = w * spw + j % spw;
          if (j >= spw && !sg_wait(&empty[s], ((j / spw) - 1) & 1)) {
            atomicOr(p.err, 4);
            ok = false;
            break;
          }
          uint8_t* dst = ring + (size_t)s * stage_bytes;
          const uint32_t bar = sg_smem(&full[s]);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(stage_bytes)
                       : "memory");
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                       ::"r"(sg_smem(dst)), "l"(r0 + (size_t)c * kch), "r"(2 * kch), "r"(bar)
                       : "memory");
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                       ::"r"(sg_smem(dst + 2 * kch)), "l"(r1 + (size_t)c * kch), "r"(2 * kch), "r"(bar)
                       : "memory");
          cnt[w] = j + 1;
        }
      }
      // no copy into this CTA's shared memory may be in flight when it exits
      for (int w = 0; w < SG_CONSUMERS; ++w)
        for (int j = cnt[w] - spw < 0 ? 0 : cnt[w] - spw; j < cnt[w]; ++j)
          sg_wait(&full[w * spw + j % spw], (j / spw) & 1);
    }
    return;
  }

  // ---------------- consumers ----------------
  pdl_wait();
  const int ctid = threadIdx.x;  // 0 .. 127
  if (p.g != nullptr) {
    float ss[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) ss[b] = 0.f;
    for (int i = ctid * 4; i < K; i += SG_CONSUMERS * 128) {
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        if (b < p.B) {
          const float4 v = *reinterpret_cast<const float4*>(p.x + (size_t)b * p.ldx + i);
          ss[b] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const float t = warp_sum(ss[b]);
      if (lane == 0) s_red[warp][b] = t;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(SG_CONSUMERS * 32) : "memory");
    if (ctid < BT) {
      float t = 0.f;
      for (int w = 0; w < SG_CONSUMERS; ++w) t += s_red[w][ctid];
      s_rms[ctid] = rsqrtf(t / (float)K + p.eps);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(SG_CONSUMERS * 32) : "memory");
  }
  const WT* g = static_cast<const WT*>(p.g);
  for (int i = ctid * 4; i < K; i += SG_CONSUMERS * 128) {
    float4 gv = make_float4(1.f, 1.f, 1.f, 1.f);
    if (g != nullptr) {
      const uint2 graw = *reinterpret_cast<const uint2*>(g + i);
      gv = make_float4(C::lo(graw.x), C::hi(graw.x), C::lo(graw.y), C::hi(graw.y));
    }
    const int dst = ((i & 4) ? (K >> 1) : 0) + ((i >> 3) << 2);
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (b < p.B) {
        v = *reinterpret_cast<const float4*>(p.x + (size_t)b * p.ldx + i);
        const float sc = (g != nullptr) ? s_rms[b] : 1.f;
        v.x *= sc * gv.x; v.y *= sc * gv.y; v.z *= sc * gv.z; v.w *= sc * gv.w;
      }
      *reinterpret_cast<float4*>(u + b * K + dst) = v;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(SG_CONSUMERS * 32) : "memory");

  bool ok = true;
  const int spw = nst / SG_CONSUMERS;
  int j = 0;  // chunks consumed from this warp's sub-ring
  for (int t = t0 + warp; t < t1 && ok; t += SG_CONSUMERS) {
    float a0[BT], a1[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) a0[b] = a1[b] = 0.f;
    for (int c = 0; c < nch; ++c, ++j) {
      const int s = warp * spw + j % spw;
      if (!sg_wait(&full[s], (j / spw) & 1)) {
        if (lane == 0) atomicOr(p.err, 4);
        ok = false;
        break;
      }
      const WT* w0 = reinterpret_cast<const WT*>(ring + (size_t)s * stage_bytes);
      const WT* w1 = w0 + kch;
      const int kbase = c * kch;
#pragma unroll 4
      for (int e = lane * 8; e < kch; e += 256) {
        const uint4 va = *reinterpret_cast<const uint4*>(w0 + e);
        const uint4 vb = *reinterpret_cast<const uint4*>(w1 + e);
        sg_fma<WT, BT>(va, u, K >> 1, kbase + e, a0, K);
        sg_fma<WT, BT>(vb, u, K >> 1, kbase + e, a1, K);
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sg_smem(&empty[s])) : "memory");
    }
    if (!ok) break;
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      a0[b] = warp_sum(a0[b]);
      a1[b] = warp_sum(a1[b]);
    }
    const WT *r0, *r1;
    int kind, local;
    sg_rows<WT, MODE>(p, t, r0, r1, kind, local);
#pragma unroll
    for (int b = 0; b < BT; ++b)
      if (lane == b && b < p.B) sg_epilogue<MODE>(p, b, t, kind, local, a0[b], a1[b]);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct SgPlan {
  int bt, kch, nst;
  size_t smem;
};

// Batch tile, chunk and ring depth for a GEMV of depth K and B rows.
static SgPlan sg_plan(int B, int K) {
  SgPlan pl;
  int nch = (K + SG_MAX_CHUNK - 1) / SG_MAX_CHUNK;
  while (K % nch || (K / nch) % 256) ++nch;
  pl.kch = K / nch;
  const int stage = 4 * pl.kch;
  pl.nst = SG_RING_BYTES / stage;
  if (pl.nst > SG_MAX_STAGES) pl.nst = SG_MAX_STAGES;
  pl.nst -= pl.nst % SG_CONSUMERS;             // whole sub-rings
  if (pl.nst < 2 * SG_CONSUMERS) pl.nst = 2 * SG_CONSUMERS;  // two stages per warp at least
  // the staged input rows must fit next to the ring
  pl.bt = B <= 1 ? 1 : (B <= 2 ? 2 : 4);
  while (pl.bt > 1 && (size_t)pl.nst * stage + (size_t)pl.bt * K * 4 + 2 * SG_MAX_STAGES * 8 > (size_t)SG_SMEM_LIMIT)
    pl.bt >>= 1;
  pl.smem = (size_t)pl.nst * stage + (size_t)pl.bt * K * 4 + 2 * SG_MAX_STAGES * 8;
  return pl;
}

int gemv_chunk(int B, int K) { return sg_plan(B, K).kch; }

template <typename WT, int BT>
static cudaError_t set_sg_attrs() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(sgemv_kernel<WT, BT, GEMV_QKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, SG_SMEM_LIMIT))) return e;
  if ((e = cudaFuncSetAttribute(sgemv_kernel<WT, BT, GEMV_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, SG_SMEM_LIMIT))) return e;
  if ((e = cudaFuncSetAttribute(sgemv_kernel<WT, BT, GEMV_RESID>, cudaFuncAttributeMaxDynamicSharedMemorySize, SG_SMEM_LIMIT))) return e;
  return cudaFuncSetAttribute(sgemv_kernel<WT, BT, GEMV_LOGITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, SG_SMEM_LIMIT);
}

cudaError_t gemv_configure() {
  cudaError_t e;
  if ((e = set_sg_attrs<bf16, 1>())) return e;
  if ((e = set_sg_attrs<bf16, 2>())) return e;
  if ((e = set_sg_attrs<bf16, 4>())) return e;
  if ((e = set_sg_attrs<f16, 1>())) return e;
  if ((e = set_sg_attrs<f16, 2>())) return e;
  return set_sg_attrs<f16, 4>();
}

template <typename WT, int BT>
static cudaError_t sg_dispatch(const GemvParams& p, int mode, int grid, size_t smem, cudaStream_t s, bool pdl) {
  const dim3 g(grid), b(SG_THREADS);
  switch (mode) {
    case GEMV_QKV: return launch_k(sgemv_kernel<WT, BT, GEMV_QKV>, g, b, smem, s, pdl, p);
    case GEMV_GATEUP: return launch_k(sgemv_kernel<WT, BT, GEMV_GATEUP>, g, b, smem, s, pdl, p);
    case GEMV_RESID: return launch_k(sgemv_kernel<WT, BT, GEMV_RESID>, g, b, smem, s, pdl, p);
    default: return launch_k(sgemv_kernel<WT, BT, GEMV_LOGITS>, g, b, smem, s, pdl, p);
  }
}

template <typename WT>
static cudaError_t sg_dispatch_bt(const GemvParams& p, int bt, int mode, int grid, size_t smem, cudaStream_t s,
                                  bool pdl) {
  if (bt == 1) return sg_dispatch<WT, 1>(p, mode, grid, smem, s, pdl);
  if (bt == 2) return sg_dispatch<WT, 2>(p, mode, grid, smem, s, pdl);
  return sg_dispatch<WT, 4>(p, mode, grid, smem, s, pdl);
}

// Batches larger than the batch tile run as consecutive launches over row chunks.
cudaError_t launch_gemv(const GemvParams& p0, int mode, int wdt, int num_sms, cudaStream_t s, bool pdl) {
  const SgPlan pl = sg_plan(p0.B, p0.K);
  for (int b0 = 0; b0 < p0.B; b0 += pl.bt) {
    GemvParams p = p0;
    p.B = p0.B - b0 < pl.bt ? p0.B - b0 : pl.bt;
    p.x = p0.x + (size_t)b0 * p0.ldx;
    p.out = p0.out + (size_t)b0 * p0.ldo;
    if (p0.x_res) p.x_res = p0.x_res + (size_t)b0 * p0.ldr;
    if (p0.pos) p.pos = p0.pos + b0;
    if (p0.kv.block_table) p.kv.block_table = p0.kv.block_table + (size_t)b0 * p0.kv.max_pages;
    p.kc = pl.kch;
    p.nst = pl.nst;
    const int grid = p.n_tasks < num_sms ? p.n_tasks : num_sms;
    cudaError_t e = wdt == WDT_F16 ? sg_dispatch_bt<f16>(p, pl.bt, mode, grid, pl.smem, s, pdl)
                                   : sg_dispatch_bt<bf16>(p, pl.bt, mode, grid, pl.smem, s, pdl);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int gemv_launch_count(int B, int K) {
  const int bt = sg_plan(B, K).bt;
  return (B + bt - 1) / bt;
}

}  // namespace ladder
