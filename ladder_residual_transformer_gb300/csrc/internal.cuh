// Internal declarations shared by the CUDA translation units of libladder.so.
// Nothing here is part of the public ABI (include/ladder.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;
typedef __half f16;

namespace ladder {

// ---------------------------------------------------------------------------
// 16-bit storage types of weights and tensor-core operands.  `lo`/`hi` widen
// the first/second element of a packed pair; `pack` rounds two floats to
// nearest even; `umma_fmt` is the operand format code of tcgen05 kind::f16.
// ---------------------------------------------------------------------------
enum WeightDtype { WDT_BF16 = 0, WDT_F16 = 1 };

template <typename T> struct W16;
template <> struct W16<bf16> {
  static __device__ __forceinline__ float lo(uint32_t v) { return __uint_as_float(v << 16); }
  static __device__ __forceinline__ float hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
  }
  // either half of a packed pair is inf or NaN
  static __device__ __forceinline__ bool bad(uint32_t v) {
    return (v & 0x7f800000u) == 0x7f800000u || (v & 0x7f80u) == 0x7f80u;
  }
  static constexpr uint32_t umma_fmt = 1;
};
template <> struct W16<f16> {
  static __device__ __forceinline__ float lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))); }
  static __device__ __forceinline__ float hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    __half2 t = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
  }
  // either half of a packed pair is inf or NaN (overflow past 65504 included)
  static __device__ __forceinline__ bool bad(uint32_t v) {
    return (v & 0x7c000000u) == 0x7c000000u || (v & 0x7c00u) == 0x7c00u;
  }
  static constexpr uint32_t umma_fmt = 0;
};

// Error-word bits set by the kernels (read back with ladder_get_device_error).
enum ErrorBits {
  ERR_TOKEN = 1,      // token id out of range (its row was computed from a zero embedding)
  ERR_TIMEOUT = 2,    // a pipeline wait ran out of time; the kernel stopped early
  ERR_NONFINITE = 4   // a projection produced inf or NaN (e.g. a value beyond the 16-bit range)
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  // Weights are read exactly once per step: bypass L1 allocation.
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// silu(z) = z / (1 + e^-z) with the fast exponential and divide: straight-line
// code (no slow-path branch), so that the independent evaluations of an
// epilogue interleave.  For z below about -88, e^-z overflows and the result is
// the correct limit 0.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Programmatic dependent launch.  pdl_trigger lets the next kernel of the stream
// start launching its CTAs; pdl_wait blocks until the previous kernel of the
// stream has completed and its writes are visible.  Both are no-ops for a
// kernel launched without the programmatic-serialization attribute.  Every
// kernel launched with the attribute calls pdl_wait before it reads or writes
// anything that an earlier kernel touches, so completion stays transitive.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// cudaLaunchKernelEx with the programmatic-serialization attribute when `pdl`.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// launch_k with a preferred shared-memory carveout for this launch (percent of
// the SM's maximum shared memory; the rest of the unified memory is L1; a
// negative value leaves the choice to the driver).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_carveout(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     bool pdl, int carveout_pct, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (carveout_pct >= 0) {
    attr[n].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
    attr[n].val.sharedMemCarveout = (unsigned)carveout_pct;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------------------
// Kernel parameter blocks
// ---------------------------------------------------------------------------

// Paged KV cache view of one layer: 16-bit (the weight dtype) [num_pages][2][n_kv][page_size][head_dim].
struct KvLayer {
  void* base;
  const int* block_table;  // [max_batch][max_pages]
  int max_pages;
  int page_size;
  int page_shift;  // log2(page_size)
  int n_kv;
  int head_dim;
  __device__ __forceinline__ size_t page_elems() const { return (size_t)2 * n_kv * page_size * head_dim; }
  // element offset of (position p of sequence b, kv 0/1, head h, dim 0)
  __device__ __forceinline__ size_t slot(int b, int p, int kv, int h) const {
    const int page = block_table[b * max_pages + (p >> page_shift)];
    return (size_t)page * page_elems() + ((size_t)(kv * n_kv + h) * page_size + (p & (page_size - 1))) * head_dim;
  }
};

enum GemvMode { GEMV_QKV = 0, GEMV_GATEUP = 1, GEMV_RESID = 2, GEMV_LOGITS = 3, GEMV_PARTIAL = 4 };

struct GemvParams {
  const float* x;    // input rows [B][ldx] fp32
  int ldx;
  const void* g;     // RMSNorm gain [K] (weight dtype), or nullptr for no norm
  float eps;
  int B, K;
  const void* w0;    // QKV: wq, GATEUP: w_gate, RESID/LOGITS: w (weight dtype)
  const void* w1;    // QKV: wk, GATEUP: w_up
  const void* w2;    // QKV: wv
  int n_tasks;       // row pairs (QKV, RESID, LOGITS) or rows (GATEUP)
  int kc;            // K chunk staged in shared memory (multiple of 256)
  int ks;            // warps that split one task's K range (1, 2, 4, 8; with chunked rows, of each chunk)
  int* err;          // device error word
  int carve;         // 1: the launch asks for the smallest shared-memory carveout holding its CTAs
  // Row-parallel shard partials (GEMV_PARTIAL): K is one shard's depth, kfull
  // the whole input row, ldw the weight row stride; task t is row pair
  // t % shard_tasks of shard t / shard_tasks.  Other modes: kfull = ldw = K.
  int kfull, ldw, shard_tasks;
  float* out;        // QKV: q [B][ldo]; GATEUP: act [B][ldo]; RESID: x_out; LOGITS: logits
  int ldo;
  const float* x_res;  // RESID: residual rows [B][ldr]
  int ldr;
  // QKV
  int nq_hd, nkv_hd;
  const float* rope_cos;  // [max_seq][head_dim / 2]
  const float* rope_sin;
  const int* pos;         // position of row b (the sequence length before this step)
  KvLayer kv;
  // Batched rows (B > 2): split-K workspace of this projection (gemv_splitk_bytes
  // bytes laid out as partial sums, per-slice sums of squares, group counters;
  // counters zero before the first launch and left zero by every launch).
  float* sk_part;
  float* sk_ss;
  int* sk_count;
};

// Split-K shape of a batched decode projection with n_tasks GEMV tasks and depth K.
struct GemvSplitK {
  int n_wtasks, n_groups, ksplit, kl;
};
GemvSplitK gemv_splitk_shape(int n_tasks, int K);
size_t gemv_splitk_bytes(int n_tasks, int K);

struct AttnDecodeParams {
  const float* q;      // [B][n_q * hd] rotated queries
  KvLayer kv;
  const int* seq_lens;  // context of row b = seq_lens[b] + 1
  int n_q;
  int split_len;        // keys per split (multiple of page_size)
  int nsplit;
  float scale;
  float* part_o;        // [B][n_q][nsplit][hd]
  float* part_ml;       // [B][n_q][nsplit][2]
  float* out;           // [B][n_q * hd]
};

enum GemmMode { GEMM_QKV = 0, GEMM_GATEUP = 1, GEMM_RESID = 2 };

// The RMSNorm of the prefill projections, split between the kernel that writes
// a stream state x_j and the GEMMs of the modules that read it.  The producer
// writes, per 128-column block c and row m, the partial sum of squares
// ss[c * ld_ss + m], and for each reading module i the 16-bit operand
// x ⊙ g_i (the hi plane at u[i]; with u_lo > 0 the rounding remainder in the
// lo plane at u[i] + u_lo), rows of the state's width.  The reading GEMM scales
// its accumulator row m by rsqrt(sum_c ss[c][m] / width + eps): the row factor
// commutes with the contraction over the row, so the product equals the one
// with the normalised row.
struct NormOut {
  float* ss;         // [width / 128][ld_ss] fp32, or nullptr (no reader)
  int ld_ss;
  void* u[2];        // operand bases of up to two readers (weight dtype), nullptr when absent
  const void* g[2];  // their RMSNorm gains [width] (weight dtype)
  size_t u_lo;       // element offset of the lo plane (0: hi plane only)
};

struct GemmParams {
  int M, N, K;
  void* out_h;          // QKV: q [M][ldo]; GATEUP: act [M][ldo] (weight dtype)
  int lo_row;           // GATEUP with hi/lo operands: first row of the lo plane in the e_out map (0: none)
  float* out_f;         // RESID: x_out [M][ldo]
  int ldo;
  const float* x_res;   // RESID
  // QKV
  int nq_hd, nkv_hd;
  const float* rope_cos;
  const float* rope_sin;
  const int* row_b;     // sequence of packed row m
  const int* row_pos;   // position of packed row m
  KvLayer kv;
  // QKV / GATEUP: the RMSNorm row factors from the producer's sums of squares
  // (nss blocks of 128 columns, ld_ss rows apart; inv_k = 1 / K); nullptr: none.
  const float* ss_in;
  int nss, ld_ss;
  float inv_k, eps;
  // RESID: the operands and sums of squares for the modules that read x_out.
  NormOut nout;
};

struct AttnPrefillParams {
  const void* q;        // [M][n_q * hd] rotated queries (weight dtype, like the KV cache); read through a tensor map
  KvLayer kv;
  const int* seq_start; // first packed row of sequence b
  const int* seq_len;   // length of sequence b
  int n_q;
  float scale;
  void* out;            // [M][n_q * hd] in the weight dtype (operand of the O projection)
  size_t lo_off;        // > 0: the rounding remainders go to out + lo_off (the lo plane)
};

// ---------------------------------------------------------------------------
// Launchers (each returns the cudaError_t of its launch)
// ---------------------------------------------------------------------------
cudaError_t launch_embed(const int* tok, int M, const void* E, int wdt, int d, int vocab, float* x, int* err,
                         cudaStream_t s, bool pdl = false);
// Prefill embedding: x_0 rows plus the RMSNorm outputs of the modules that read x_0.
cudaError_t launch_embed_norm(const int* tok, int M, const void* E, int wdt, int d, int vocab, float* x,
                              const NormOut& no, int* err, cudaStream_t s, bool pdl);
cudaError_t launch_gemv(const GemvParams& p, int mode, int wdt, int num_sms, cudaStream_t s, bool pdl = false);
cudaError_t gemv_configure();
int gemv_chunk(int B, int K);
int gemv_launch_count(int B, int K, int mode);
cudaError_t launch_attn_decode(const AttnDecodeParams& p, int B, int n_kv, int hd, int kv_dtype, cudaStream_t s,
                               bool pdl = false);
// Merge of the per-split partials (part_o, part_ml) into out.
cudaError_t launch_attn_combine(const AttnDecodeParams& p, int B, int hd, cudaStream_t s, bool pdl);
// Decode attention on the tensor cores (mma.sync), K/V pages through the layer's
// KV pool map (make_kv_tma_map); split_len 128, head_dim 64 or 128, up to 8 query
// heads per KV head.  Launches the split kernel (programmatic dependent launch
// when `pdl`) and the combine step (when `pdl_combine`).
cudaError_t attn_decode_tc_configure();
cudaError_t launch_attn_decode_tc(const void* kv_map, const AttnDecodeParams& p, int B, int n_kv, int hd, int wdt,
                                  int* err, cudaStream_t s, bool pdl, bool pdl_combine);
// Temperature / top-k sampling of the next token (sample.cu); row b draws with
// position pos[b] + pos_off.  temperature must be > 0.
cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k, uint64_t seed,
                          const int* pos, int pos_off, int* out, cudaStream_t s, bool pdl);
cudaError_t launch_argmax(const float* logits, int B, int V, float* part_v, int* part_i, int nblk,
                          int* out, cudaStream_t s, bool pdl = false);
cudaError_t launch_advance(int* seq_lens, int B, cudaStream_t s, bool pdl = false);
// Rotary frequency scaling by wavelength band (off when factor <= 1).
struct RopeScaling {
  double factor, low_freq_factor, high_freq_factor, original_max_pos;
};
cudaError_t launch_rope_tables(float* cos_t, float* sin_t, int max_seq, int hd, float theta, RopeScaling sc,
                               cudaStream_t s);

// Prefill launches take `pdl` (programmatic dependent launch); every kernel
// launched with it waits for the previous kernel before touching its data.
// Tensor-core GEMM (tcgen05 + TMA).  Maps are CUtensorMap objects made by make_tma_map.
// 2-D map of a row-major [rows, cols] 16-bit matrix, box 64 columns x 128 rows.
bool make_tma_map(void* map_out, const void* base, uint64_t rows, uint64_t cols, int wdt);
// GEMM operand: the same matrix as 3-D [cols / 64][rows][64], with boxes of
// 128 rows x 1 and x 2 chunks (box[0], box[1]).  An activation operand held
// as a hi/lo pair of planes (the hi matrix [rows][cols], then the lo matrix
// right after it) also gets `pair`: a 4-D view [cols / 64][2][rows][64] whose
// box of 128 rows x 2 planes x 1 chunk lands as the hi block, then the lo block.
struct TmaOperand {
  CUtensorMap box[2];
  CUtensorMap pair;
};
bool make_tma_operand(TmaOperand* out, const void* base, uint64_t rows, uint64_t cols, int wdt,
                      bool with_pair = false);
// Epilogue block map (box 32 x 32): fp32 rows (elem_bytes 4) or weight-dtype rows (2).
bool make_tma_map_epilogue(void* map_out, const void* base, uint64_t rows, uint64_t cols, int elem_bytes, int wdt);
// One layer of the paged KV pool as a 3-D map (see gemm_tcgen05.cu).
bool make_kv_tma_map(void* map_out, const void* base, uint64_t num_pages, int n_kv, int page_size, int hd, int wdt);
cudaError_t gemm_tc_configure();
// e_in / e_out: make_tma_map_epilogue maps of the residual rows and the output
// rows (RESID, fp32) or of the SwiGLU output rows (GATEUP e_out, weight dtype).
// wide: A is a hi/lo pair (a->pair); every k step multiplies both halves by
// the same weight tile, so C = W * (hi + lo).
cudaError_t launch_gemm_tc(const TmaOperand* a, const TmaOperand* b0, const TmaOperand* b1, const TmaOperand* b2,
                           const void* e_in, const void* e_out, const GemmParams& p, int mode, int wdt, int num_sms,
                           int* err, cudaStream_t s, bool pdl = false, bool wide = false);
// Tensor-core causal attention for packed prefill rows (mma.sync, bf16 Q/K/V).
// Prefill attention on tcgen05: q_map = make_tma_map of the query rows, kv_map =
// make_kv_tma_map of the layer; head_dim 64 or 128.
cudaError_t attn_prefill_tcgen05_configure();
cudaError_t launch_attn_prefill_tcgen05(const void* q_map, const void* kv_map, const AttnPrefillParams& p, int hd,
                                        int wdt, int B, int max_len, int* err, cudaStream_t s, bool pdl = false);
cudaError_t launch_gather_rows(const float* x, int d, const int* rows, int B, float* out,
                               cudaStream_t s, bool pdl = false);
cudaError_t launch_set_lens(const int* lens, int B, int* seq_lens, cudaStream_t s, bool pdl = false);
// x_out[b, n] = x_res[b, n] + sum_{s < k} part[b][s][n], summed in the fixed order s = 0..k-1.
cudaError_t launch_shard_reduce(const float* part, int k, int B, int d, const float* x_res, float* x_out,
                                cudaStream_t s, bool pdl);

}  // namespace ladder
