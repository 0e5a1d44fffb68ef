// Decode projections: the weight-streaming GEMV for one or two rows (CUDA cores,
// fused RMSNorm prologue and RoPE / KV-write, SwiGLU, residual, logits and
// shard-partial epilogues) and the split-K projection for 3..16 rows on
// mma.sync, with the launcher that picks between them.
#include "internal.cuh"

#include <math.h>

namespace ladder {

constexpr int GEMV_WARPS = 8;
constexpr int GEMV_THREADS = GEMV_WARPS * 32;
constexpr int GEMV_SMEM_FLOATS = 16384;  // 64 KB staged input per CTA
constexpr int GEMV_PF_HEAD = 1024;       // columns of the first task prefetched by multi-round launches

// ---------------------------------------------------------------------------
// GEMV: out[b, n] = sum_k W[n, k] * u[b, k] for B <= BT rows, fused prologue and
// epilogue by mode.  u = x * rsqrt(mean(x^2) + eps) * g when a gain is given.
//
// Work unit ("task") = two weight rows computed together by one warp: a RoPE
// pair (2j, 2j+1) for QKV, the matching gate and up rows for SwiGLU, or two
// consecutive rows otherwise.  Lane l reads 16 bytes (8 bf16) at k = 8l + 256i.
// Staged input layout per batch row: two planes [kc/8][4] holding elements
// k%8 < 4 and k%8 >= 4, so that each lane's 16-byte shared-memory reads are
// contiguous across the warp (no bank conflicts).
// ---------------------------------------------------------------------------
template <typename WT, int BT>
__device__ __forceinline__ void gemv_fma(const uint4& w, const float* __restrict__ u, int kc, int k,
                                         float (&acc)[BT]) {
  using C = W16<WT>;
  const float w0 = C::lo(w.x), w1 = C::hi(w.x), w2 = C::lo(w.y), w3 = C::hi(w.y);
  const float w4 = C::lo(w.z), w5 = C::hi(w.z), w6 = C::lo(w.w), w7 = C::hi(w.w);
  const int q = (k >> 3) << 2;
#pragma unroll
  for (int b = 0; b < BT; ++b) {
    const float4 a = *reinterpret_cast<const float4*>(u + b * kc + q);
    const float4 c = *reinterpret_cast<const float4*>(u + b * kc + (kc >> 1) + q);
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

// The two weight rows of GEMV task `task` (see the task definition above); for
// QKV also which matrix (kind 0 = q, 1 = k, 2 = v) and the first row inside it.
template <typename WT, int MODE>
__device__ __forceinline__ void gemv_task_rows(const GemvParams& p, int task, const WT*& row0, const WT*& row1,
                                               int& kind, int& local, int& koff) {
  const WT* W0 = static_cast<const WT*>(p.w0);
  const WT* W1 = static_cast<const WT*>(p.w1);
  const WT* W2 = static_cast<const WT*>(p.w2);
  const int K = p.K;
  kind = 0;
  local = 0;
  koff = 0;
  if (MODE == GEMV_QKV) {
    const int r0 = 2 * task;
    if (r0 < p.nq_hd) {
      local = r0; kind = 0; row0 = W0 + (size_t)local * K;
    } else if (r0 < p.nq_hd + p.nkv_hd) {
      local = r0 - p.nq_hd; kind = 1; row0 = W1 + (size_t)local * K;
    } else {
      local = r0 - p.nq_hd - p.nkv_hd; kind = 2; row0 = W2 + (size_t)local * K;
    }
    row1 = row0 + K;
  } else if (MODE == GEMV_GATEUP) {
    row0 = W0 + (size_t)task * K;
    row1 = W1 + (size_t)task * K;
  } else if (MODE == GEMV_PARTIAL) {
    koff = (task / p.shard_tasks) * K;
    row0 = W0 + (size_t)(2 * (task % p.shard_tasks)) * p.ldw + koff;
    row1 = row0 + p.ldw;
  } else {
    row0 = W0 + (size_t)(2 * task) * K;
    row1 = row0 + K;
  }
}

// Epilogue of task `task` for batch row b: (v0, v1) are the dot products of its
// two weight rows.
template <typename WT, int MODE>
__device__ __forceinline__ void gemv_store(const GemvParams& p, int task, int b, int kind, int local, float v0,
                                           float v1) {
  using C = W16<WT>;
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
      float* q = p.out + (size_t)b * p.ldo + local;
      q[0] = r0;
      q[1] = r1;
    } else {
      const int head = local / hd, dim = local % hd;
      WT* dst = static_cast<WT*>(p.kv.base) + p.kv.slot(b, pos, kind - 1, head) + dim;
      const uint32_t pk = C::pack(r0, r1);
      *reinterpret_cast<uint32_t*>(dst) = pk;
      if (C::bad(pk) && p.err != nullptr) atomicOr(p.err, ERR_NONFINITE);  // beyond the 16-bit range
    }
  } else if (MODE == GEMV_GATEUP) {
    p.out[(size_t)b * p.ldo + task] = silu_f(v0) * v1;
  } else if (MODE == GEMV_RESID) {
    const size_t n = 2 * (size_t)task;
    p.out[(size_t)b * p.ldo + n] = p.x_res[(size_t)b * p.ldr + n] + v0;
    p.out[(size_t)b * p.ldo + n + 1] = p.x_res[(size_t)b * p.ldr + n + 1] + v1;
  } else if (MODE == GEMV_PARTIAL) {
    // out is [B][k][d]: shard s writes its partial sums at s * (2 * shard_tasks)
    const size_t n = (size_t)(task / p.shard_tasks) * (2 * p.shard_tasks) + 2 * (size_t)(task % p.shard_tasks);
    p.out[(size_t)b * p.ldo + n] = v0;
    p.out[(size_t)b * p.ldo + n + 1] = v1;
  } else {
    const size_t n = 2 * (size_t)task;
    p.out[(size_t)b * p.ldo + n] = v0;
    p.out[(size_t)b * p.ldo + n + 1] = v1;
  }
}

template <typename WT, int BT, int MODE>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_kernel(const GemvParams p) {
  using C = W16<WT>;
  const WT* g = static_cast<const WT*>(p.g);
  const WT* W0 = static_cast<const WT*>(p.w0);
  const WT* W1 = static_cast<const WT*>(p.w1);
  const WT* W2 = static_cast<const WT*>(p.w2);
  extern __shared__ float4 gemv_smem4[];
  float* u = reinterpret_cast<float*>(gemv_smem4);
  __shared__ float s_red[GEMV_WARPS][BT];
  __shared__ float s_rms[BT];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = p.K;
  pdl_trigger();

  // Weights depend on no earlier kernel: before the RMSNorm prologue and before
  // waiting for the previous kernel, each warp asks L2 for its first task's
  // weight rows -- the whole range when every task of this CTA fits in one
  // round of a single chunk, else the first GEMV_PF_HEAD columns (a whole round
  // of a large matrix would not stay in L2) -- so that the DRAM traffic
  // overlaps both and the launch boundary (no registers are held for it).
  // Measured on the graph decode step: 8B hybrid 3245 -> 3178 us, 70B
  // 23.99 -> 23.71 ms; 2048 columns were no better, 4096 slower.
  {
    const int ks_ = p.ks;
    const int task0 = blockIdx.x * (GEMV_WARPS / ks_) + warp / ks_;
    const bool one_round =
        (MODE == GEMV_PARTIAL || p.kc >= p.kfull) && (long long)gridDim.x * (GEMV_WARPS / ks_) >= p.n_tasks;
    if (task0 < p.n_tasks) {
      const WT* r0;
      const WT* r1;
      if (MODE == GEMV_QKV) {
        const int q0 = 2 * task0;
        r0 = q0 < p.nq_hd ? W0 + (size_t)q0 * K
                          : (q0 < p.nq_hd + p.nkv_hd ? W1 + (size_t)(q0 - p.nq_hd) * K
                                                     : W2 + (size_t)(q0 - p.nq_hd - p.nkv_hd) * K);
        r1 = r0 + K;
      } else if (MODE == GEMV_GATEUP) {
        r0 = W0 + (size_t)task0 * K;
        r1 = W1 + (size_t)task0 * K;
      } else if (MODE == GEMV_PARTIAL) {
        r0 = W0 + (size_t)(2 * (task0 % p.shard_tasks)) * p.ldw + (size_t)(task0 / p.shard_tasks) * K;
        r1 = r0 + p.ldw;
      } else {
        r0 = W0 + (size_t)(2 * task0) * K;
        r1 = r0 + K;
      }
      const int span0 = (p.kc >= p.kfull ? K : p.kc) / ks_;  // the warp's slice of the first staged chunk
      const int kb = ks_ > 1 ? (warp % ks_) * span0 : 0;
      const int ke_all = ks_ > 1 ? kb + span0 : K;
      const int ke = one_round ? ke_all : min(ke_all, kb + GEMV_PF_HEAD);
      // one 128-byte line (64 elements) per lane per step
      for (int k = kb + lane * 64; k < ke; k += 32 * 64) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(r0 + k));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(r1 + k));
      }
    }
  }
  pdl_wait();

  // RMSNorm statistics of each input row, in a fixed order (identical in every CTA).
  if (p.g != nullptr) {
    float ss[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) ss[b] = 0.f;
    for (int i = tid * 4; i < K; i += GEMV_THREADS * 4) {
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
    __syncthreads();
    if (tid < BT) {
      float t = 0.f;
      for (int w = 0; w < GEMV_WARPS; ++w) t += s_red[w][tid];
      s_rms[tid] = rsqrtf(t / (float)K + p.eps);
    }
    __syncthreads();
  }

  // Warp w works on task slot w / ks of this CTA and on K slice w % ks.
  const int ks = p.ks;
  const int tpc = GEMV_WARPS / ks;  // tasks per CTA per round
  const int slot = warp / ks, kslice = warp % ks;
  const int total_slots = gridDim.x * tpc;
  const int rounds = (p.n_tasks + total_slots - 1) / total_slots;
  // Length of the staged input rows: the whole row, or for shard partials the
  // K-slice of one shard (a CTA's tasks in one round share a shard: its tasks
  // per round divide the shard's task count).
  const int KF = MODE == GEMV_PARTIAL ? K : p.kfull;
  const bool single_chunk = p.kc >= KF;
  const int kspan = K / ks;  // the warp's slice of a single staged chunk
  __shared__ float s_part[GEMV_WARPS][2][BT];

  for (int r = 0; r < rounds; ++r) {
    const int task = r * total_slots + blockIdx.x * tpc + slot;
    const bool active = task < p.n_tasks;

    // Which two weight rows this task reads.
    const WT* row0 = W0;
    const WT* row1 = W0;
    int local = 0, kind = 0;  // QKV: kind 0 = q, 1 = k, 2 = v; local = row inside its matrix
    int koff = 0;             // PARTIAL: first input element of the task's shard
    if (active) gemv_task_rows<WT, MODE>(p, task, row0, row1, kind, local, koff);
    // PARTIAL: the shard whose slice this round stages (every CTA stages one,
    // active or not, so that all threads reach the barriers)
    int xoff = 0;
    if (MODE == GEMV_PARTIAL) xoff = (min(r * total_slots + blockIdx.x * tpc, p.n_tasks - 1) / p.shard_tasks) * K;

    float a0[BT], a1[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) a0[b] = a1[b] = 0.f;

    for (int k0 = 0; k0 < KF; k0 += p.kc) {
      const int kc = min(p.kc, KF - k0);
      if (!single_chunk || r == 0 || MODE == GEMV_PARTIAL) {
        __syncthreads();
        // Stage the (normalised) input chunk in the two-plane layout.
        for (int i = tid * 4; i < kc; i += GEMV_THREADS * 4) {
          float4 gv = make_float4(1.f, 1.f, 1.f, 1.f);
          if (g != nullptr) {
            const uint2 graw = *reinterpret_cast<const uint2*>(g + xoff + k0 + i);
            gv = make_float4(C::lo(graw.x), C::hi(graw.x), C::lo(graw.y), C::hi(graw.y));
          }
          const int dst = ((i & 4) ? (kc >> 1) : 0) + ((i >> 3) << 2);
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (b < p.B) {
              v = *reinterpret_cast<const float4*>(p.x + (size_t)b * p.ldx + xoff + k0 + i);
              const float sc = (p.g != nullptr) ? s_rms[b] : 1.f;
              v.x *= sc * gv.x; v.y *= sc * gv.y; v.z *= sc * gv.z; v.w *= sc * gv.w;
            }
            *reinterpret_cast<float4*>(u + b * kc + dst) = v;
          }
        }
        __syncthreads();
      }
      if (active) {
        // Weights: row + k0 + k (a shard's rows start at its slice); staged
        // input: element k of the chunk (of the shard's slice).
        const WT* p0 = row0 + k0;
        const WT* p1 = row1 + k0;
        const int ksl = single_chunk ? kspan : kc / ks;  // rows staged in chunks: a slice of each chunk
        const int kb = ks > 1 ? kslice * ksl : 0;
        const int ke = ks > 1 ? kb + ksl : kc;
        int k = kb + lane * 8;
        for (; k + 768 < ke; k += 1024) {
          uint4 wa[4], wb[4];
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            wa[s] = ld_stream_u4(p0 + k + 256 * s);
            wb[s] = ld_stream_u4(p1 + k + 256 * s);
          }
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            gemv_fma<WT, BT>(wa[s], u, kc, k + 256 * s, a0);
            gemv_fma<WT, BT>(wb[s], u, kc, k + 256 * s, a1);
          }
        }
        for (; k < ke; k += 256) {
          const uint4 wa = ld_stream_u4(p0 + k);
          const uint4 wb = ld_stream_u4(p1 + k);
          gemv_fma<WT, BT>(wa, u, kc, k, a0);
          gemv_fma<WT, BT>(wb, u, kc, k, a1);
        }
      }
    }

#pragma unroll
    for (int b = 0; b < BT; ++b) {
      a0[b] = warp_sum(a0[b]);
      a1[b] = warp_sum(a1[b]);
    }
    if (ks > 1) {
      // combine the K slices of each task in a fixed order
      if (lane == 0) {
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          s_part[warp][0][b] = a0[b];
          s_part[warp][1][b] = a1[b];
        }
      }
      __syncthreads();
      if (kslice == 0) {
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          float t0 = 0.f, t1 = 0.f;
          for (int i = 0; i < ks; ++i) {
            t0 += s_part[warp + i][0][b];
            t1 += s_part[warp + i][1][b];
          }
          a0[b] = t0;
          a1[b] = t1;
        }
      }
      __syncthreads();
      if (kslice != 0) continue;
    }
    if (!active) continue;

    // Epilogue: lane b handles batch row b.
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      if (lane != b || b >= p.B) continue;
      gemv_store<WT, MODE>(p, task, b, kind, local, a0[b], a1[b]);
    }
  }
}

// ---------------------------------------------------------------------------
// Batched decode projection, 3..16 rows, on the tensor cores.  The GEMV above
// streams every weight byte once per 4 rows; here mma.sync m16n8k16 takes the
// weights as the M = 16 operand and the batch as N (two 8-wide tiles), so each
// weight byte is streamed once for all 16 rows.
//
// Warp task = 8 GEMV tasks (row pairs): MMA row g < 8 is the first row of pair g,
// row g + 8 its second, so lane (g, t) ends up holding both values of pair g for
// batch rows 2t, 2t+1 (+8) and the GEMV epilogue applies unchanged.
// K is permuted inside each 32-element block so that lane (g, t) reads the 16
// contiguous bytes k = 8t..8t+7 of its two weight rows and of each staged
// input row: element 8t + 4c + {0,1,2,3} plays logical column {2t, 2t+1, 2t+8,
// 2t+9} of MMA k-block c.  A permutation of K applied to both operands leaves
// every dot product unchanged.
//
// Split K across CTAs: CTA (group, slice) stages only its K slice of the 16
// input rows (x * g as 16-bit values, rows padded by 16 bytes for
// conflict-free reads) and the slice's sum of squares of each row, and each of
// its 8 warps writes the 16 x 16 partial sums of one warp task.  The last CTA
// of a group to finish (an atomic counter, reset after use) adds the slices in
// a fixed order, applies the RMSNorm scale rsqrt(sum x^2 / K + eps) of each row
// (a per-row factor, so it commutes with the dot products) and runs the
// epilogue.  Each CTA thus reads a small slice of the inputs, not all of them.
// ---------------------------------------------------------------------------
// Longest K slice (staged 16-bit columns).  1024 rather than 2048 halves each
// CTA's staged inputs, so a fourth CTA fits per SM: 8B hybrid, 16 rows from
// context 2048, 5503 -> 5225 us per step (512: 5272 us).
constexpr int GM_KL_MAX = 1024;
constexpr int GM_PF_AHEAD = 2;   // 128-column steps of weights requested ahead of use

template <typename T>
__device__ __forceinline__ void mma16816_f32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
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

GemvSplitK gemv_splitk_shape(int n_tasks, int K) {
  GemvSplitK sk;
  sk.n_wtasks = (n_tasks + 7) / 8;
  sk.n_groups = (sk.n_wtasks + GEMV_WARPS - 1) / GEMV_WARPS;
  const int units = K / 256;  // K is a multiple of 256
  int best = 0;
  for (int ks = 1; ks <= units; ++ks) {
    if (units % ks || K / ks > GM_KL_MAX) continue;
    best = ks;  // the finest admissible split so far
    if ((long long)sk.n_groups * ks >= 320) break;
  }
  sk.ksplit = best;
  sk.kl = K / best;
  return sk;
}

size_t gemv_splitk_bytes(int n_tasks, int K) {
  const GemvSplitK sk = gemv_splitk_shape(n_tasks, K);
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  return up((size_t)sk.ksplit * sk.n_wtasks * 256 * 4) + up((size_t)sk.n_groups * sk.ksplit * 16 * 4) +
         up((size_t)sk.n_groups * 4);
}

template <typename WT, int MODE>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_splitk_kernel(const GemvParams p, int ksplit, int kl) {
  using C = W16<WT>;
  const WT* g = static_cast<const WT*>(p.g);
  extern __shared__ float4 gm_smem4[];
  WT* xs = reinterpret_cast<WT*>(gm_smem4);  // [16][kl + 8] staged inputs of this slice
  __shared__ float s_ss[GEMV_WARPS][16];
  __shared__ float s_rms[16];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gi = lane >> 2, ti = lane & 3;
  const int gN = blockIdx.x, kS = blockIdx.y;
  const int n_wtasks = (p.n_tasks + 7) / 8;
  const int ld = kl + 8;
  const int k0 = kS * kl;
  const int wtask = gN * GEMV_WARPS + warp;
  const int task = wtask * 8 + gi;  // the row pair of this lane
  const bool lane_active = wtask < n_wtasks && task < p.n_tasks;
  const WT* row0;
  const WT* row1;
  int kind, local, koff;
  gemv_task_rows<WT, MODE>(p, lane_active ? task : 0, row0, row1, kind, local, koff);
  pdl_trigger();
  // Weights depend on no earlier kernel: the L2 is asked for the first
  // GM_PF_AHEAD 128-column steps of this warp's rows before the wait, and for
  // step i + GM_PF_AHEAD at step i (a window: the whole slab of a large matrix
  // would not stay in L2 until it is read).  Lane (gi, ti) takes one of the
  // four 128-byte lines of its row pair per step.
  const WT* pf_row = (ti >> 1) ? row1 : row0;
  const int pf_off = k0 + (ti & 1) * 64;
  if (wtask < n_wtasks)
    for (int i = 0; i < GM_PF_AHEAD && i * 128 < kl; ++i)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(pf_row + pf_off + i * 128));
  pdl_wait();

  // 1. Stage x * g for rows 0..15 of this slice (zero rows past B) and the
  //    slice's sum of squares of each row.  Item i = (row i / (kl/8), 8 columns);
  //    kl / 8 is a multiple of 32, so a warp's items share one row.
  s_ss[warp][lane & 15] = 0.f;
  __syncwarp();
  const int per_row = kl / 8;
  for (int i = tid; i < 16 * per_row; i += GEMV_THREADS) {
    const int b = i / per_row, k8 = (i % per_row) * 8;
    uint4 pk = make_uint4(0, 0, 0, 0);
    float sq = 0.f;
    if (b < p.B) {
      const float* src = p.x + (size_t)b * p.ldx + k0 + k8;
      const float4 v0 = *reinterpret_cast<const float4*>(src);
      const float4 v1 = *reinterpret_cast<const float4*>(src + 4);
      sq = v0.x * v0.x + v0.y * v0.y + v0.z * v0.z + v0.w * v0.w + v1.x * v1.x + v1.y * v1.y + v1.z * v1.z +
           v1.w * v1.w;
      float sc[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
      if (g != nullptr) {
        const uint4 graw = *reinterpret_cast<const uint4*>(g + k0 + k8);
        sc[0] = C::lo(graw.x); sc[1] = C::hi(graw.x); sc[2] = C::lo(graw.y); sc[3] = C::hi(graw.y);
        sc[4] = C::lo(graw.z); sc[5] = C::hi(graw.z); sc[6] = C::lo(graw.w); sc[7] = C::hi(graw.w);
      }
      pk.x = C::pack(v0.x * sc[0], v0.y * sc[1]);
      pk.y = C::pack(v0.z * sc[2], v0.w * sc[3]);
      pk.z = C::pack(v1.x * sc[4], v1.y * sc[5]);
      pk.w = C::pack(v1.z * sc[6], v1.w * sc[7]);
    }
    *reinterpret_cast<uint4*>(xs + b * ld + k8) = pk;
    sq = warp_sum(sq);
    if (lane == 0) s_ss[warp][b] += sq;
  }
  __syncthreads();

  // 2. Partial sums of this warp task over the slice.
  float acc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  if (wtask < n_wtasks) {
    const WT* p0 = row0 + k0 + 8 * ti;
    const WT* p1 = row1 + k0 + 8 * ti;
    const WT* x0 = xs + gi * ld + 8 * ti;        // batch row gi (n tile 0)
    const WT* x1 = xs + (gi + 8) * ld + 8 * ti;  // batch row gi + 8 (n tile 1)
    int k = 0;
    for (; k + 96 < kl; k += 128) {
      if (k + GM_PF_AHEAD * 128 < kl) asm volatile("prefetch.global.L2 [%0];" ::"l"(pf_row + pf_off + k + GM_PF_AHEAD * 128));
      uint4 wa[4], wb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        wa[u] = ld_stream_u4(p0 + k + 32 * u);
        wb[u] = ld_stream_u4(p1 + k + 32 * u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 xa = *reinterpret_cast<const uint4*>(x0 + k + 32 * u);
        const uint4 xb = *reinterpret_cast<const uint4*>(x1 + k + 32 * u);
        mma16816_f32<WT>(acc[0], wa[u].x, wb[u].x, wa[u].y, wb[u].y, xa.x, xa.y);
        mma16816_f32<WT>(acc[0], wa[u].z, wb[u].z, wa[u].w, wb[u].w, xa.z, xa.w);
        mma16816_f32<WT>(acc[1], wa[u].x, wb[u].x, wa[u].y, wb[u].y, xb.x, xb.y);
        mma16816_f32<WT>(acc[1], wa[u].z, wb[u].z, wa[u].w, wb[u].w, xb.z, xb.w);
      }
    }
    for (; k < kl; k += 32) {
      const uint4 wa = ld_stream_u4(p0 + k), wb = ld_stream_u4(p1 + k);
      const uint4 xa = *reinterpret_cast<const uint4*>(x0 + k);
      const uint4 xb = *reinterpret_cast<const uint4*>(x1 + k);
      mma16816_f32<WT>(acc[0], wa.x, wb.x, wa.y, wb.y, xa.x, xa.y);
      mma16816_f32<WT>(acc[0], wa.z, wb.z, wa.w, wb.w, xa.z, xa.w);
      mma16816_f32<WT>(acc[1], wa.x, wb.x, wa.y, wb.y, xb.x, xb.y);
      mma16816_f32<WT>(acc[1], wa.z, wb.z, wa.w, wb.w, xb.z, xb.w);
    }
    float4* dst = reinterpret_cast<float4*>(p.sk_part + ((size_t)kS * n_wtasks + wtask) * 256 + lane * 8);
    dst[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
    dst[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
  }
  if (tid < 16) {
    float t = 0.f;
    for (int w = 0; w < GEMV_WARPS; ++w) t += s_ss[w][tid];
    p.sk_ss[((size_t)gN * ksplit + kS) * 16 + tid] = t;
  }

  // 3. The last CTA of the group combines the slices.
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.sk_count + gN, 1) == ksplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < 16) {
    float rm = 1.f;
    if (g != nullptr) {
      float t = 0.f;
      for (int s2 = 0; s2 < ksplit; ++s2) t += __ldcg(p.sk_ss + ((size_t)gN * ksplit + s2) * 16 + tid);
      rm = rsqrtf(t / (float)p.K + p.eps);
    }
    s_rms[tid] = rm;
  }
  if (tid == 0) p.sk_count[gN] = 0;  // ready for the next launch
  __syncthreads();
  if (!lane_active) return;
  float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s2 = 0; s2 < ksplit; ++s2) {
    const float4* src = reinterpret_cast<const float4*>(p.sk_part + ((size_t)s2 * n_wtasks + wtask) * 256 + lane * 8);
    const float4 a = __ldcg(src), c = __ldcg(src + 1);
    sum[0] += a.x; sum[1] += a.y; sum[2] += a.z; sum[3] += a.w;
    sum[4] += c.x; sum[5] += c.y; sum[6] += c.z; sum[7] += c.w;
  }
  // lane (gi, ti): pair gi, batch rows nt * 8 + 2 ti + e; first row in sum[4 nt + e], second in sum[4 nt + 2 + e]
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int b = nt * 8 + 2 * ti + e;
      if (b < p.B)
        gemv_store<WT, MODE>(p, task, b, kind, local, sum[4 * nt + e] * s_rms[b], sum[4 * nt + 2 + e] * s_rms[b]);
    }
}

// Residency of the decode projection kernels: the CTAs per SM that their
// registers and threads allow, and their static shared memory; with the SM's
// shared memory and the per-CTA reservation.  Read once, from gemv_configure
// (model creation), never inside a stream capture.
struct GemvResidency {
  int ctas[2][3][5] = {};         // GEMV: [weight dtype][batch tile 1, 2, 4][mode]
  int static_smem[2][3][5] = {};
  int mma_ctas[2][4] = {};        // split-K projection: [weight dtype][mode]
  int mma_static_smem[2][4] = {};
  int smem_per_sm = 0;
  int smem_reserved = 0;
};

static void residency_of(const void* fn, int& ctas, int& static_smem) {
  int n = 0;
  cudaFuncAttributes a{};
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, GEMV_THREADS, 0) == cudaSuccess &&
      cudaFuncGetAttributes(&a, fn) == cudaSuccess) {
    ctas = n;
    static_smem = (int)a.sharedSizeBytes;
  } else {
    (void)cudaGetLastError();  // leave the rules that use it off for this kernel (ctas = 0)
  }
}

template <typename WT>
static void gemv_mma_residency_row(GemvResidency& r, int w) {
  const void* f[4] = {(const void*)gemv_splitk_kernel<WT, GEMV_QKV>, (const void*)gemv_splitk_kernel<WT, GEMV_GATEUP>,
                      (const void*)gemv_splitk_kernel<WT, GEMV_RESID>, (const void*)gemv_splitk_kernel<WT, GEMV_LOGITS>};
  for (int m = 0; m < 4; ++m) residency_of(f[m], r.mma_ctas[w][m], r.mma_static_smem[w][m]);
}

template <typename WT, int BT>
static void gemv_residency_row(GemvResidency& r, int w, int b) {
  const void* f[5] = {(const void*)gemv_kernel<WT, BT, GEMV_QKV>, (const void*)gemv_kernel<WT, BT, GEMV_GATEUP>,
                      (const void*)gemv_kernel<WT, BT, GEMV_RESID>, (const void*)gemv_kernel<WT, BT, GEMV_LOGITS>,
                      (const void*)gemv_kernel<WT, BT, GEMV_PARTIAL>};
  for (int m = 0; m < 5; ++m) residency_of(f[m], r.ctas[w][b][m], r.static_smem[w][b][m]);
}

static const GemvResidency& gemv_residency() {
  static const GemvResidency r = [] {
    GemvResidency t;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      t.smem_per_sm = 0;
      return t;
    }
    gemv_residency_row<bf16, 1>(t, WDT_BF16, 0);
    gemv_residency_row<bf16, 2>(t, WDT_BF16, 1);
    gemv_residency_row<bf16, 4>(t, WDT_BF16, 2);
    gemv_residency_row<f16, 1>(t, WDT_F16, 0);
    gemv_residency_row<f16, 2>(t, WDT_F16, 1);
    gemv_residency_row<f16, 4>(t, WDT_F16, 2);
    gemv_mma_residency_row<bf16>(t, WDT_BF16);
    gemv_mma_residency_row<f16>(t, WDT_F16);
    return t;
  }();
  return r;
}

// Shared-memory carveout of one launch: the smallest share of the SM's unified
// memory that holds the CTAs per SM the launch can use (its grid over the SMs,
// at most `cap`, what registers and threads allow), so that the rest serves as
// L1 for the weight loads in flight; -1 (the driver's choice) when unknown.
// Measured on the batched projection (8B hybrid, 16 rows, context 2048): this
// request (45%, 3 CTAs per SM) 5090 -> 4930 us per step against the driver's
// choice; 50% 4910 us; 30% (2 CTAs) 5250 us; all shared memory 6100 us.
static int carveout_for(long long grid, size_t smem, int static_smem, int cap, int num_sms) {
  const GemvResidency& r = gemv_residency();
  if (cap <= 0 || r.smem_per_sm <= 0 || num_sms <= 0) return -1;
  long long want = (grid + num_sms - 1) / num_sms;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  const long long need = want * ((long long)smem + static_smem + r.smem_reserved);
  const long long pct = (need * 100 + r.smem_per_sm - 1) / r.smem_per_sm;
  return pct > 100 ? 100 : (int)pct;
}

static int gemv_carveout(int grid, size_t smem, int bt, int mode, int wdt, int num_sms) {
  const GemvResidency& r = gemv_residency();
  const int w = wdt == WDT_F16 ? WDT_F16 : WDT_BF16, b = bt == 1 ? 0 : (bt == 2 ? 1 : 2);
  return carveout_for(grid, smem, r.static_smem[w][b][mode], r.ctas[w][b][mode], num_sms);
}

template <typename WT>
static cudaError_t set_gemv_mma_attrs() {
  const int bytes = 16 * (GM_KL_MAX + 8) * 2;
  const void* fns[4] = {(const void*)gemv_splitk_kernel<WT, GEMV_QKV>, (const void*)gemv_splitk_kernel<WT, GEMV_GATEUP>,
                        (const void*)gemv_splitk_kernel<WT, GEMV_RESID>, (const void*)gemv_splitk_kernel<WT, GEMV_LOGITS>};
  cudaError_t e;
  for (const void* fn : fns)
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  return cudaSuccess;
}

// Rows b0 .. b0 + 15 (at most) of a batched projection on the tensor cores.
static cudaError_t launch_gemv_mma(GemvParams p, int mode, int wdt, int num_sms, cudaStream_t s, bool pdl) {
  if (p.sk_part == nullptr || p.sk_ss == nullptr || p.sk_count == nullptr) return cudaErrorInvalidValue;
  const GemvSplitK sk = gemv_splitk_shape(p.n_tasks, p.K);
  const dim3 grid(sk.n_groups, sk.ksplit), block(GEMV_THREADS);
  const size_t smem = (size_t)16 * (sk.kl + 8) * 2;
  int co = -1;
  if (p.carve) {
    const GemvResidency& r = gemv_residency();
    const int w = wdt == WDT_F16 ? WDT_F16 : WDT_BF16, m = mode < 4 ? mode : GEMV_LOGITS;
    co = carveout_for((long long)grid.x * grid.y, smem, r.mma_static_smem[w][m], r.mma_ctas[w][m], num_sms);
  }
  auto go = [&](auto kern) { return launch_k_carveout(kern, grid, block, smem, s, pdl, co, p, sk.ksplit, sk.kl); };
  if (wdt == WDT_F16) {
    switch (mode) {
      case GEMV_QKV: return go(gemv_splitk_kernel<f16, GEMV_QKV>);
      case GEMV_GATEUP: return go(gemv_splitk_kernel<f16, GEMV_GATEUP>);
      case GEMV_RESID: return go(gemv_splitk_kernel<f16, GEMV_RESID>);
      default: return go(gemv_splitk_kernel<f16, GEMV_LOGITS>);
    }
  }
  switch (mode) {
    case GEMV_QKV: return go(gemv_splitk_kernel<bf16, GEMV_QKV>);
    case GEMV_GATEUP: return go(gemv_splitk_kernel<bf16, GEMV_GATEUP>);
    case GEMV_RESID: return go(gemv_splitk_kernel<bf16, GEMV_RESID>);
    default: return go(gemv_splitk_kernel<bf16, GEMV_LOGITS>);
  }
}

int gemv_chunk(int B, int K) {
  const int bt = B <= 1 ? 1 : (B <= 2 ? 2 : 4);
  int kc = GEMV_SMEM_FLOATS / bt;
  kc -= kc % 256;
  return K < kc ? K : kc;
}

template <typename WT, int BT>
static cudaError_t set_gemv_attrs() {
  const int bytes = GEMV_SMEM_FLOATS * 4;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<WT, BT, GEMV_QKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<WT, BT, GEMV_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<WT, BT, GEMV_RESID>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  if ((e = cudaFuncSetAttribute(gemv_kernel<WT, BT, GEMV_PARTIAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))) return e;
  return cudaFuncSetAttribute(gemv_kernel<WT, BT, GEMV_LOGITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Longest staged chunk -- at most kc_max columns, a multiple of `align`, the row
// cut into equal chunks -- with which a launch of `grid` CTAs is resident at
// once (one wave); 0 when no chunk of at least 2048 columns gives that.  A
// second wave of a few CTAs, alone on their SMs, streams its rows at a fraction
// of the bandwidth.  Chunk boundaries at multiples of 256 leave each lane's
// columns and the order of its products unchanged.
static int gemv_wave_chunk(int kfull, int kc_max, int align, long long grid, int bt, int mode, int wdt,
                           int num_sms) {
  const GemvResidency& r = gemv_residency();
  const int w = wdt == WDT_F16 ? WDT_F16 : WDT_BF16, b = bt == 1 ? 0 : (bt == 2 ? 1 : 2);
  const int cap = r.ctas[w][b][mode];
  if (cap <= 0 || r.smem_per_sm <= 0 || kfull % align) return 0;
  kc_max -= kc_max % align;
  if (kc_max <= 0) return 0;
  for (int nch = (kfull + kc_max - 1) / kc_max;; ++nch) {
    const int kc = ((kfull + nch - 1) / nch + align - 1) / align * align;
    if (kc < 2048) return 0;
    const int per_cta = bt * kc * (int)sizeof(float) + r.static_smem[w][b][mode] + r.smem_reserved;
    int fit = r.smem_per_sm / per_cta;
    if (fit > cap) fit = cap;
    if ((long long)fit * num_sms >= grid) return kc;
  }
}

static long long gemv_grid(int n_tasks, int ks, int num_sms) {
  const int tpc = GEMV_WARPS / ks;
  const long long g = (n_tasks + tpc - 1) / tpc;
  return g < (long long)num_sms * 8 ? g : (long long)num_sms * 8;
}

cudaError_t gemv_configure() {
  (void)gemv_residency();
  cudaError_t e;
  if ((e = set_gemv_attrs<bf16, 1>())) return e;
  if ((e = set_gemv_attrs<bf16, 2>())) return e;
  if ((e = set_gemv_attrs<bf16, 4>())) return e;
  if ((e = set_gemv_attrs<f16, 1>())) return e;
  if ((e = set_gemv_attrs<f16, 2>())) return e;
  if ((e = set_gemv_attrs<f16, 4>())) return e;
  if ((e = set_gemv_mma_attrs<bf16>())) return e;
  return set_gemv_mma_attrs<f16>();
}

template <typename WT, int BT>
static cudaError_t gemv_dispatch(const GemvParams& p, int mode, int grid, size_t smem, cudaStream_t s, bool pdl,
                                 int co) {
  const dim3 g(grid), b(GEMV_THREADS);
  switch (mode) {
    case GEMV_QKV: return launch_k_carveout(gemv_kernel<WT, BT, GEMV_QKV>, g, b, smem, s, pdl, co, p);
    case GEMV_GATEUP: return launch_k_carveout(gemv_kernel<WT, BT, GEMV_GATEUP>, g, b, smem, s, pdl, co, p);
    case GEMV_RESID: return launch_k_carveout(gemv_kernel<WT, BT, GEMV_RESID>, g, b, smem, s, pdl, co, p);
    case GEMV_PARTIAL: return launch_k_carveout(gemv_kernel<WT, BT, GEMV_PARTIAL>, g, b, smem, s, pdl, co, p);
    default: return launch_k_carveout(gemv_kernel<WT, BT, GEMV_LOGITS>, g, b, smem, s, pdl, co, p);
  }
}

template <typename WT>
static cudaError_t gemv_dispatch_bt(const GemvParams& p, int bt, int mode, int grid, size_t smem, cudaStream_t s,
                                    bool pdl, int co) {
  if (bt == 1) return gemv_dispatch<WT, 1>(p, mode, grid, smem, s, pdl, co);
  if (bt == 2) return gemv_dispatch<WT, 2>(p, mode, grid, smem, s, pdl, co);
  return gemv_dispatch<WT, 4>(p, mode, grid, smem, s, pdl, co);
}

// Batches of 1..4 rows run on the CUDA-core GEMV; larger batches run on the
// tensor-core kernel in chunks of 16 rows (shard partials stay on the GEMV, in
// chunks of 4).
// From three rows on, the tensor-core projection (weights streamed once for up
// to 16 rows) beats the GEMV's batch tile of 4 (8B hybrid, graph decode step:
// B = 3 608 vs 561 tok/s, B = 4 814 vs 713; B = 2 stays on the GEMV, 498 vs 416).
static bool gemv_use_mma(int B, int mode) { return B > 2 && mode != GEMV_PARTIAL; }

int gemv_launch_count(int B, int K, int mode) { return gemv_use_mma(B, mode) ? (B + 15) / 16 : (B + 3) / 4; }

// Batches larger than 4 run as consecutive chunks of at most 4 rows.
cudaError_t launch_gemv(const GemvParams& p0, int mode, int wdt, int num_sms, cudaStream_t s, bool pdl) {
  if (gemv_use_mma(p0.B, mode)) {
    for (int b0 = 0; b0 < p0.B; b0 += 16) {
      GemvParams p = p0;
      p.B = p0.B - b0 < 16 ? p0.B - b0 : 16;
      p.x = p0.x + (size_t)b0 * p0.ldx;
      p.out = p0.out + (size_t)b0 * p0.ldo;
      if (p0.x_res) p.x_res = p0.x_res + (size_t)b0 * p0.ldr;
      if (p0.pos) p.pos = p0.pos + b0;
      if (p0.kv.block_table) p.kv.block_table = p0.kv.block_table + (size_t)b0 * p0.kv.max_pages;
      p.kfull = p.K;
      p.ldw = p.K;
      p.shard_tasks = p.n_tasks;
      cudaError_t e = launch_gemv_mma(p, mode, wdt, num_sms, s, pdl);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  for (int b0 = 0; b0 < p0.B; b0 += 4) {
    GemvParams p = p0;
    p.B = p0.B - b0 < 4 ? p0.B - b0 : 4;
    p.x = p0.x + (size_t)b0 * p0.ldx;
    p.out = p0.out + (size_t)b0 * p0.ldo;
    if (p0.x_res) p.x_res = p0.x_res + (size_t)b0 * p0.ldr;
    if (p0.pos) p.pos = p0.pos + b0;
    if (p0.kv.block_table) p.kv.block_table = p0.kv.block_table + (size_t)b0 * p0.kv.max_pages;
    const int bt = p.B <= 1 ? 1 : (p.B <= 2 ? 2 : 4);
    if (mode != GEMV_PARTIAL) {
      p.kfull = p.K;
      p.ldw = p.K;
      p.shard_tasks = p.n_tasks;
    }
    // Shard partials stage one shard's K-slice of the row (one chunk).
    p.kc = mode == GEMV_PARTIAL ? p.K : gemv_chunk(p.B, p.kfull);
    if (mode == GEMV_PARTIAL && p.kc > gemv_chunk(p.B, p.K)) return cudaErrorInvalidValue;
    // K split: the smallest that gives at least 1.5 CTAs per SM (more warps in
    // flight for short, wide matrices) while each slice stays a multiple of 256.
    // Residual projections (O, down: few outputs, long rows) split K at least
    // 4 ways (measured on the 1.2B and 8B decode steps: 1.2% and 4.8% faster
    // than the 1.5-CTAs-per-SM rule alone); QKV never splits.
    p.ks = 1;
    if (p.kc >= p.kfull || mode == GEMV_PARTIAL) {
      while (p.ks < GEMV_WARPS && (long long)p.n_tasks * p.ks < (long long)num_sms * 12 &&
             (p.K / (2 * p.ks)) % 256 == 0)
        p.ks *= 2;
      if (mode == GEMV_RESID)
        while (p.ks < 4 && (p.K / (4 * p.ks)) % 256 == 0) p.ks *= 2;
      // QKV keeps whole rows per warp (its epilogue, rotation and cache write,
      // runs once per task; measured 0.8% faster on the 1.2B step than K split 2)
      if (mode == GEMV_QKV) p.ks = 1;
    }
    // Rows longer than one chunk (70B down projection, K = 28672): chunks short
    // enough for one wave.  64 KB chunks gave 3 CTAs per SM and 512 CTAs in 1.12
    // waves (104.5 us per launch, serialised); 3 chunks of 9728 columns give 4
    // CTAs per SM (registers) in one wave: 70B decode step 22.64 -> 20.59 ms,
    // logits bit-identical.
    if (p.kc < p.kfull && mode != GEMV_PARTIAL) {
      const int kc = gemv_wave_chunk(p.kfull, p.kc, 256, gemv_grid(p.n_tasks, 1, num_sms), bt, mode, wdt, num_sms);
      if (kc) p.kc = kc;
    }
    // Residual projections (O, down): the largest K split of 4, 2 or 1 whose
    // launch fits one wave, staging the rows in chunks where that raises the
    // CTAs per SM; when none does, the split chosen above.  8B: O at K split 2
    // (512 CTAs, was 1024 in 1.68 waves), down at K split 2 in two chunks of
    // 7168 (was 1024 CTAs in 2.25 waves at 3 per SM); 70B O at no split (512
    // CTAs, was 1216 in two waves).  Decode step, graph, context 2048: 8B hybrid
    // B = 1 3057 -> 2908 us, B = 2 4228 -> 3759 us, 70B 20.87 -> 20.78 ms; the
    // 1.2B launches already fitted (unchanged).
    if (mode == GEMV_RESID) {
      for (int ks = 4; ks >= 1; ks /= 2) {
        const int kc = gemv_wave_chunk(p.kfull, gemv_chunk(p.B, p.kfull), 256 * ks, gemv_grid(p.n_tasks, ks, num_sms),
                                       bt, mode, wdt, num_sms);
        if (kc) {
          p.ks = ks;
          p.kc = kc;
          break;
        }
      }
    }
    const size_t smem = (size_t)bt * p.kc * sizeof(float);
    const int tpc = GEMV_WARPS / p.ks;
    int grid = (p.n_tasks + tpc - 1) / tpc;
    const int cap = num_sms * 8;
    if (grid > cap) grid = cap;
    const int co = p.carve ? gemv_carveout(grid, smem, bt, mode, wdt, num_sms) : -1;
    cudaError_t e = wdt == WDT_F16 ? gemv_dispatch_bt<f16>(p, bt, mode, grid, smem, s, pdl, co)
                                   : gemv_dispatch_bt<bf16>(p, bt, mode, grid, smem, s, pdl, co);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ladder
