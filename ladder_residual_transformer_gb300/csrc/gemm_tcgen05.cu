// Prefill projection GEMM on the 5th-generation tensor cores (sm_103a):
//   C[m, n] = sum_k A[m, k] * W[n, k],  A = bf16 activations [M, K],
//   W = bf16 weights [N, K] (both K-major), fp32 accumulation in TMEM.
//
// Persistent CTAs (one per SM) loop over 128 x BN tiles (BN = 256, or 128 for
// narrow matrices) with tcgen05.mma (cta_group::1, kind::f16, M = 128, N = BN,
// K = 16 per instruction).  Warp roles:
//   warp 4: one elected thread issues the TMA loads of A (128 rows) and of the
//           two 128-row halves of B (each half may come from a different
//           weight matrix: q/k/v rows, or the gate and up rows of SwiGLU),
//           K = 64 (BN = 256) or 128 (BN = 128) per stage;
//   warp 5: allocates 2 x BN TMEM columns (two accumulator buffers) and one
//           elected thread issues the MMAs, releasing each shared-memory stage
//           with tcgen05.commit and each finished accumulator to the epilogue;
//   warps 0-3: epilogue, reading the accumulator with tcgen05.ld (warp w owns
//           TMEM lanes 32w..32w+31, i.e. tile rows), transposing each 32x32
//           block through shared memory so that every global load and store
//           of a warp covers a contiguous row segment, and applying the fused
//           RoPE + KV scatter, SwiGLU, or residual add; then it hands the
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

// A stage holds K = 64 * KC of each operand as KC 64-element (128-byte) chunks,
// loaded by one 3-D TMA box per operand ([chunk][row][64]): KC = 2 makes every
// row of a box a 256-byte contiguous run of global memory, which the 128-wide
// tiles need to keep the tensor cores fed; 256-wide tiles use KC = 1 and a
// deeper ring.
constexpr int TC_BM = 128;
constexpr int TC_CHUNK = 128 * 64 * 2;  // one 128-row x 64-element chunk, 16 KB
// Stage ring: 3 stages of 64 KB at BN = 128 (KC = 2), 4 of 48 KB at BN = 256 (KC = 1).
constexpr int TC_RING = 3 * 4 * TC_CHUNK;
// Epilogue buffers: per epilogue warp two 4 KB blocks (32 x 32 fp32, or 32 x 32
// 16-bit values in the first half) that TMA fills and drains; the QKV epilogue
// uses the same space as a 32 x 33 fp32 transpose block.
constexpr int TC_EP_LD = 33;
constexpr int TC_EP_WARP = 8192;
constexpr int TC_EP_BYTES = 4 * TC_EP_WARP;
constexpr int TC_SMEM = TC_RING + TC_EP_BYTES + 1024 + 256;
constexpr int TC_THREADS = 192;
constexpr int TC_PAIR_KC = 1;  // 64-wide K chunks per stage of the paired 256 x 256 tiles
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

// RMSNorm row factor of row `row` for a reading GEMM: rsqrt(sum of the producer's
// per-128-column sums of squares / K + eps), summed in a fixed order (eight
// interleaved partial sums whose loads are all in flight at once, then a tree).
__device__ __forceinline__ float row_rms_factor(const GemmParams& p, int row) {
  if (row >= p.M) return 1.f;
  const float* s = p.ss_in + row;
  const size_t ld = (size_t)p.ld_ss;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int c = 0;
  for (; c + 8 <= p.nss; c += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldg(s + (size_t)(c + j) * ld);
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] += v[j];
  }
  for (; c < p.nss; ++c) a[c & 7] += __ldg(s + (size_t)c * ld);
  const float t = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  return rsqrtf(t * p.inv_k + p.eps);
}

// The RMSNorm outputs of one 32-column chunk of a new stream row x (see NormOut):
// x ⊙ g for each reading module as a 16-bit hi (and lo) plane row segment.
// Returns the chunk's sum of squares (the caller adds four chunks per 128-column
// entry of no.ss).
template <typename WT>
__device__ __forceinline__ float norm_outputs(const NormOut& no, const float (&x)[32], int row, int col, int width) {
  using C = W16<WT>;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    s0 = fmaf(x[4 * j], x[4 * j], s0);
    s1 = fmaf(x[4 * j + 1], x[4 * j + 1], s1);
    s2 = fmaf(x[4 * j + 2], x[4 * j + 2], s2);
    s3 = fmaf(x[4 * j + 3], x[4 * j + 3], s3);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (!no.u[k]) continue;
    const uint4* gp = reinterpret_cast<const uint4*>(static_cast<const WT*>(no.g[k]) + col);
    WT* dst = static_cast<WT*>(no.u[k]) + (size_t)row * width + col;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 gr = __ldg(gp + q);
      const float u0 = x[8 * q] * C::lo(gr.x), u1 = x[8 * q + 1] * C::hi(gr.x);
      const float u2 = x[8 * q + 2] * C::lo(gr.y), u3 = x[8 * q + 3] * C::hi(gr.y);
      const float u4 = x[8 * q + 4] * C::lo(gr.z), u5 = x[8 * q + 5] * C::hi(gr.z);
      const float u6 = x[8 * q + 6] * C::lo(gr.w), u7 = x[8 * q + 7] * C::hi(gr.w);
      uint4 hi;
      hi.x = C::pack(u0, u1);
      hi.y = C::pack(u2, u3);
      hi.z = C::pack(u4, u5);
      hi.w = C::pack(u6, u7);
      *reinterpret_cast<uint4*>(dst + 8 * q) = hi;
      if (no.u_lo) {
        uint4 lo;
        lo.x = C::pack(u0 - C::lo(hi.x), u1 - C::hi(hi.x));
        lo.y = C::pack(u2 - C::lo(hi.y), u3 - C::hi(hi.y));
        lo.z = C::pack(u4 - C::lo(hi.z), u5 - C::hi(hi.z));
        lo.w = C::pack(u6 - C::lo(hi.w), u7 - C::hi(hi.w));
        *reinterpret_cast<uint4*>(dst + no.u_lo + 8 * q) = lo;
      }
    }
  }
  return (s0 + s1) + (s2 + s3);
}

struct TcMaps {
  CUtensorMap a;
  CUtensorMap b[3];
  CUtensorMap e_in;   // RESID: residual rows x_res (fp32, box 32 x 32, 128-byte swizzle)
  CUtensorMap e_out;  // RESID: output rows (fp32, as e_in); GATEUP: SwiGLU rows (16-bit, box 32 x 32, 64-byte swizzle)
};

// Persistent CTA: tiles t = blockIdx.x + i * gridDim.x, tile t -> (m = t % m_tiles,
// n = t / m_tiles) so that CTAs running together share the weight tile in L2.
// The accumulator is double-buffered in TMEM (2 x BN columns): the MMA warp
// fills buffer i & 1 while the epilogue warps drain the other one.
//
// PAIR = 1 (BN = 256): clusters of two CTAs compute 256 x 256 tiles with the
// paired MMA (tcgen05 cta_group::2): each CTA holds the A rows of its own m
// tile and one 128-row half of B, so a stage is 32 KB instead of 48 KB (6
// stages instead of 4) and each SM's shared memory serves half as many B bytes
// per MMA.  Both CTAs' copies signal the leader's full barrier; the leader
// issues the M = 256 MMAs and commits to both CTAs' empty and accumulator-full
// barriers; both CTAs' epilogue warps arrive on the leader's accumulator-empty
// barrier.
template <int PAIR>
__device__ __forceinline__ int gemm_tile_count(int m_tiles, int n_tiles) {
  const int units = PAIR ? (m_tiles / 2) * n_tiles : m_tiles * n_tiles;
  const int id = PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const int nid = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;
  return id < units ? (units - 1 - id) / nid + 1 : 0;
}
template <int PAIR>
__device__ __forceinline__ void gemm_tile(int i, int m_tiles, uint32_t crank, int& m_tile, int& tile_n) {
  if (PAIR) {
    const int u = (int)blockIdx.x / 2 + i * ((int)gridDim.x / 2), mp = m_tiles / 2;
    m_tile = 2 * (u % mp) + (int)crank;
    tile_n = u / mp;
  } else {
    const int t = blockIdx.x + i * gridDim.x;
    m_tile = t % m_tiles;
    tile_n = t / m_tiles;
  }
}

// WIDE = 1: A is a hi/lo pair of planes.  Each stage holds the hi and the lo
// block of every A chunk (A_BYTES doubles, KC = 1), and each k step issues the
// hi MMA and then the lo MMA against the same B tile, so the accumulator sums
// W * hi + W * lo and the activations enter the product with about 22
// significant bits instead of 11.
template <typename WT, int MODE, int BN, int KC, int PAIR, int WIDE>
__global__ void __launch_bounds__(TC_THREADS, 1) gemm_tc_kernel(const __grid_constant__ TcMaps maps,
                                                                const GemmParams p, int m_tiles, int n_tiles,
                                                                int* err) {
  using C = W16<WT>;
  constexpr int HALVES = BN / 128;
  constexpr int BK = 64 * KC;
  static_assert(!WIDE || KC == 1, "hi/lo operands use one 64-wide chunk per stage");
  constexpr int A_BYTES = KC * TC_CHUNK * (WIDE ? 2 : 1);   // 128 rows of A (hi and lo blocks when WIDE)
  constexpr int BH_BYTES = KC * TC_CHUNK;  // one 128-row half of B
  constexpr int HB = PAIR ? 1 : HALVES;  // B halves held by this CTA
  constexpr int STAGE = A_BYTES + HB * BH_BYTES;
  constexpr int NST = TC_RING / STAGE;
  static_assert(!PAIR || BN == 256, "paired tiles are 256 x 256");
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ep_all = smem + TC_RING;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TC_RING + TC_EP_BYTES);
  uint64_t* empty = full + NST;
  uint64_t* tfull = empty + NST;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;    // [2] accumulator drained
  uint64_t* ebar = tempty + 2;     // [4 warps][2] epilogue block loaded
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ebar + 8);
  int* bail = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = p.K / BK;
  const int my_tiles = gemm_tile_count<PAIR>(m_tiles, n_tiles);
  pdl_trigger();
  const uint32_t crank = PAIR ? cluster_ctarank() : 0;
  const bool leader = crank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 8 : 4);  // one arrival per epilogue warp (of both CTAs)
    }
    for (int e = 0; e < 8; ++e) mbar_init(&ebar[e], 1);
    *bail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    if (PAIR) {  // one warp of each CTA of the pair allocates collectively
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(2 * BN)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                   "r"(2 * BN)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  if (PAIR) cluster_sync_all();  // the leader's barriers exist before the peer signals them
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched early (programmatic dependent launch), the prologue above overlaps
  // the previous kernel; no thread touches global memory before it completes.
  pdl_wait();

  if (warp == 4) {
    if (lane == 0) {
      int it = 0;  // running k-block index across tiles
      bool ok = true;
      for (int i = 0; ok && i < my_tiles; ++i) {
        int mt_, tn;
        gemm_tile<PAIR>(i, m_tiles, crank, mt_, tn);
        const int m0 = mt_ * TC_BM;
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
          if (PAIR) {
            // this CTA's A rows and B half r; both signal the leader's full barrier
            const uint32_t fb = smem_map_rank(&full[s], 0);
            if (leader) mbar_expect_tx(&full[s], 2 * STAGE);
            if (WIDE) tma_load_4d_pair(st, &maps.a, 0, m0, 0, kb, fb);
            else tma_load_3d_pair(st, &maps.a, 0, m0, kb * KC, fb);
            if (crank == 0) tma_load_3d_pair(st + A_BYTES, &maps.b[map0], 0, row0, kb * KC, fb);
            else tma_load_3d_pair(st + A_BYTES, &maps.b[map1], 0, row1, kb * KC, fb);
            continue;
          }
          mbar_expect_tx(&full[s], STAGE);
          if (WIDE) tma_load_4d(st, &maps.a, 0, m0, 0, kb, &full[s]);
          else tma_load_3d(st, &maps.a, 0, m0, kb * KC, &full[s]);
          tma_load_3d(st + A_BYTES, &maps.b[map0], 0, row0, kb * KC, &full[s]);
          if (HALVES == 2) tma_load_3d(st + A_BYTES + BH_BYTES, &maps.b[map1], 0, row1, kb * KC, &full[s]);
          // The CTAs of a tile column read the same weight boxes at about the same
          // time; for 128-wide tiles the first m tile asks L2 for them 2 * NST
          // steps ahead, so that the ring's copies hit L2 instead of waiting on
          // DRAM (measured: faster for 128-wide tiles, slower for the 256-wide
          // gate/up tiles).
          if (BN == 128 && m0 == 0 && kb + 2 * NST < nkb) {
            tma_prefetch_3d(&maps.b[map0], 0, row0, (kb + 2 * NST) * KC);
            if (HALVES == 2) tma_prefetch_3d(&maps.b[map1], 0, row1, (kb + 2 * NST) * KC);
          }
        }
      }
      // Make sure no copy into this CTA's shared memory is still in flight (the
      // leader's full barriers also count the peer's copies; the peer's last
      // copies have landed once the leader's MMAs consumed them, before the
      // final cluster barrier).
      if (leader)
        for (int k = it - NST < 0 ? 0 : it - NST; k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1);
    }
  } else if (warp == 5) {
    if (lane == 0 && leader) {
      // KC = 1: the two B halves are contiguous, one N = BN MMA per k step.
      // KC = 2: each half is its own [chunk][row] box, one N = 128 MMA per half.
      // PAIR: one M = 256 paired MMA per k step.
      constexpr int MMA_N = (PAIR || KC == 1) ? BN : 128;
      constexpr int MMAS = (PAIR || KC == 1) ? 1 : HALVES;
      constexpr uint32_t idesc = umma_idesc(PAIR ? 2 * TC_BM : TC_BM, MMA_N, C::umma_fmt);
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
          const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
          for (int c = 0; c < KC; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
#pragma unroll
              for (int w = 0; w <= WIDE; ++w) {  // w = 0: hi block (or the only one), 1: lo block
                const uint32_t a_off = ((WIDE ? 2 : 1) * c + w) * TC_CHUNK + kk * 32;
                const uint32_t accum = (kb | c | kk | w) != 0;
#pragma unroll
                for (int hh = 0; hh < MMAS; ++hh)
                  if (PAIR)
                    umma_f16_pair(d, umma_desc(a_base + a_off), umma_desc(b_base + c * TC_CHUNK + kk * 32), idesc,
                                  accum);
                  else
                    umma_f16(d + hh * 128, umma_desc(a_base + a_off),
                             umma_desc(b_base + hh * BH_BYTES + c * TC_CHUNK + kk * 32), idesc, accum);
              }
          if (PAIR) umma_commit_pair(&empty[s], 3);
          else umma_commit(&empty[s]);
        }
        // also after a bail, so that the MMAs in flight finish first
        if (PAIR) umma_commit_pair(&tfull[acc], 3);
        else umma_commit(&tfull[acc]);
      }
    }
  } else {
    // Epilogue warp w owns tile rows 32w .. 32w + 31 (its TMEM lanes; lane =
    // row).  RESID and GATEUP move 32 x 32 blocks through TMA: the residual
    // block is loaded before it is needed, lane r adds accumulator row r to
    // row r of the block in shared memory, and a TMA store writes the block
    // out.  QKV transposes each 32 x 32 block through shared memory so that
    // a warp's global stores (q rows, paged K/V slots) are row segments.
    const int hd = p.kv.head_dim;
    uint8_t* ewarp = ep_all + warp * TC_EP_WARP;
    float* ep = reinterpret_cast<float*>(ewarp);
    uint64_t* eb = ebar + warp * 2;
    constexpr int NCH = BN / 32;  // 32-column chunks of a tile
    uint32_t nload[2] = {0, 0}, nwait[2] = {0, 0};  // loads issued / consumed per buffer (warp-uniform)
    bool ep_ok = true;
    const int cp = 2 * (lane & 15), rsub = lane >> 4;  // 16-bit outputs: column pair, row parity
    for (int i = 0; i < my_tiles; ++i) {
      const int acc = i & 1;
      int mt_, tile_n;
      gemm_tile<PAIR>(i, m_tiles, crank, mt_, tile_n);
      const int mrow0 = mt_ * TC_BM + warp * 32;
      // RMSNorm factor of this lane's row (reading GEMMs), before the accumulator is awaited
      const float rnorm = (MODE != GEMM_RESID && p.ss_in) ? row_rms_factor(p, mrow0 + lane) : 1.f;
      // Row metadata of this lane's row (QKV), fetched before the accumulator is
      // awaited: position and the element offset of its slot in the paged cache
      // (page base + slot * hd; the kv / head term is added per column).
      int my_pos = 0;
      long long my_slot = 0;
      if (MODE == GEMM_QKV && mrow0 + lane < p.M) {
        my_pos = p.row_pos[mrow0 + lane];
        const int bb = p.row_b[mrow0 + lane];
        const int page = p.kv.block_table[bb * p.kv.max_pages + (my_pos >> p.kv.page_shift)];
        my_slot = (long long)page * (long long)p.kv.page_elems() + (long long)(my_pos & (p.kv.page_size - 1)) * hd;
      }
      if (MODE == GEMM_RESID) {
        // the first two residual blocks of the tile, while its accumulator is computed
        if (lane == 0) bulk_wait_read_all();  // the previous tile's stores have left the buffers
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (lane == 0) {
            mbar_expect_tx(&eb[c], 4096);
            tma_load_2d(ewarp + c * 4096, &maps.e_in, tile_n * BN + c * 32, mrow0, &eb[c]);
          }
          ++nload[c];
        }
      }
      const bool ok = mbar_wait(&tfull[acc], (i >> 1) & 1);
      tc_fence_after();
      if (!ok) {
        if (lane == 0) atomicOr(err, 2);
        ep_ok = false;
        break;
      }
      if (__shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(bail), 0)) break;
      const uint32_t trow = tmem + acc * BN + ((uint32_t)(warp * 32) << 16);
      auto stage = [&](const float (&v)[32]) {
#pragma unroll
        for (int j = 0; j < 32; ++j) ep[lane * TC_EP_LD + j] = v[j];
        __syncwarp();
      };
      if (MODE == GEMM_GATEUP) {
        for (int c = 0; c < 4; ++c) {
          uint8_t* buf = ewarp + (c & 1) * 4096;
          // buffer c & 1 was last stored two chunks ago
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          __syncwarp();
          float gv[32], uv[32];
          tmem_ld32(trow + c * 32, gv);
          tmem_ld32(trow + 128 + c * 32, uv);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            gv[j] *= rnorm;
            uv[j] *= rnorm;
          }
          uint32_t pk[16], pl[16];
          bool bad = false;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a0 = silu_f(gv[2 * j]) * uv[2 * j], a1 = silu_f(gv[2 * j + 1]) * uv[2 * j + 1];
            pk[j] = C::pack(a0, a1);
            bad |= mrow0 + lane < p.M && C::bad(pk[j]);  // rows past M hold padding
            if (WIDE) pl[j] = C::pack(a0 - C::lo(pk[j]), a1 - C::hi(pk[j]));  // rounding remainders
          }
          if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, ERR_NONFINITE);
          // row lane, 64-byte rows, 16-byte chunk q at q ^ ((row >> 1) & 3) (64-byte swizzle);
          // the lo block (WIDE) is the second 2 KB of the buffer
          uint4* rowp = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            rowp[q ^ ((lane >> 1) & 3)] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            if (WIDE)
              rowp[128 + (q ^ ((lane >> 1) & 3))] = make_uint4(pl[4 * q], pl[4 * q + 1], pl[4 * q + 2], pl[4 * q + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&maps.e_out, buf, tile_n * 128 + c * 32, mrow0);
            if (WIDE) tma_store_2d(&maps.e_out, buf + 2048, tile_n * 128 + c * 32, p.lo_row + mrow0);
            bulk_commit();
          }
        }
      } else if (MODE == GEMM_RESID) {
        float sq128 = 0.f;  // sum of squares of this row's current 128 columns
        for (int c = 0; c < NCH; ++c) {
          const int bi = c & 1;
          float* buf = reinterpret_cast<float*>(ewarp + bi * 4096);
          const bool okc = __all_sync(0xffffffffu, mbar_wait(&eb[bi], nwait[bi] & 1));
          ++nwait[bi];
          if (!okc) {
            if (lane == 0) atomicOr(err, 2);
            ep_ok = false;
            break;
          }
          float v[32];
          tmem_ld32(trow + c * 32, v);
          // row lane of the block: 16-byte chunk q at q ^ (row & 7) (128-byte swizzle)
          float4* rowp = reinterpret_cast<float4*>(buf + lane * 32);
          bool bad = false;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 xv = rowp[q ^ (lane & 7)];
            xv.x += v[4 * q];
            xv.y += v[4 * q + 1];
            xv.z += v[4 * q + 2];
            xv.w += v[4 * q + 3];
            bad |= mrow0 + lane < p.M && !(isfinite(xv.x) && isfinite(xv.y) && isfinite(xv.z) && isfinite(xv.w));
            rowp[q ^ (lane & 7)] = xv;
            v[4 * q] = xv.x;  // v now holds this lane's 32 new stream values
            v[4 * q + 1] = xv.y;
            v[4 * q + 2] = xv.z;
            v[4 * q + 3] = xv.w;
          }
          if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, ERR_NONFINITE);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&maps.e_out, buf, tile_n * BN + c * 32, mrow0);
            bulk_commit();
          }
          // the RMSNorm inputs of the modules that read this stream state
          if (p.nout.ss && mrow0 + lane < p.M) {
            sq128 += norm_outputs<WT>(p.nout, v, mrow0 + lane, tile_n * BN + c * 32, p.N);
            if ((c & 3) == 3) {
              p.nout.ss[(size_t)((tile_n * BN + c * 32) >> 7) * p.nout.ld_ss + mrow0 + lane] = sq128;
              sq128 = 0.f;
            }
          }
          if (c + 2 < NCH) {
            if (lane == 0) {
              bulk_wait_read_all();  // the store above has read the buffer
              mbar_expect_tx(&eb[bi], 4096);
              tma_load_2d(buf, &maps.e_in, tile_n * BN + (c + 2) * 32, mrow0, &eb[bi]);
            }
            ++nload[bi];
          }
        }
        if (!ep_ok) break;
      } else {  // GEMM_QKV
        for (int c = 0; c < BN / 32; ++c) {
          int map, row;
          if (!b_half<GEMM_QKV, BN>(p, tile_n, c >> 2, map, row)) break;
          float v[32];
          tmem_ld32(trow + c * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= rnorm;
          const int col = row + (c & 3) * 32 + cp;  // column inside its matrix (even: a RoPE pair)
          const int head = col / hd, dim = col % hd;
          // Rotation of each of this lane's 16 rows, all table loads in flight at
          // once (rows past M have position 0: in-bounds loads, no store).  The
          // code below is branch-free per row so that the rows interleave.
          float cs[16], sn[16];
          if (map < 2) {
#pragma unroll
            for (int r2 = 0; r2 < 16; ++r2) {
              const int pos = __shfl_sync(0xffffffffu, my_pos, 2 * r2 + rsub);
              const size_t tj = (size_t)pos * (hd >> 1) + (dim >> 1);
              cs[r2] = __ldg(p.rope_cos + tj);
              sn[r2] = __ldg(p.rope_sin + tj);
            }
          } else {
#pragma unroll
            for (int r2 = 0; r2 < 16; ++r2) {
              cs[r2] = 1.f;
              sn[r2] = 0.f;
            }
          }
          long long off[16];
#pragma unroll
          for (int r2 = 0; r2 < 16; ++r2) {
            const int m = mrow0 + 2 * r2 + rsub;
            const long long slot = __shfl_sync(0xffffffffu, my_slot, 2 * r2 + rsub);
            off[r2] = map == 0 ? (long long)m * p.ldo : slot;
          }
          stage(v);
          float a[32];
#pragma unroll
          for (int r2 = 0; r2 < 16; ++r2) {
            const int r = 2 * r2 + rsub;
            a[2 * r2] = ep[r * TC_EP_LD + cp];
            a[2 * r2 + 1] = ep[r * TC_EP_LD + cp + 1];
          }
          __syncwarp();
          // q, K and V are stored in the weight dtype (the attention operands)
          WT* base = map == 0 ? static_cast<WT*>(p.out_h) + col
                              : static_cast<WT*>(p.kv.base) +
                                    ((long long)((map - 1) * p.kv.n_kv + head) * p.kv.page_size * hd + dim);
          bool bad = false;
#pragma unroll
          for (int r2 = 0; r2 < 16; ++r2) {
            const float r0 = a[2 * r2] * cs[r2] - a[2 * r2 + 1] * sn[r2];
            const float r1 = a[2 * r2] * sn[r2] + a[2 * r2 + 1] * cs[r2];
            const uint32_t pk = C::pack(r0, r1);
            const bool live = mrow0 + 2 * r2 + rsub < p.M;
            bad |= live && C::bad(pk);
            if (live) *reinterpret_cast<uint32_t*>(base + off[r2]) = pk;
          }
          if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, ERR_NONFINITE);
        }
      }
      // hand the accumulator buffer back to the (leader's) MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR) mbar_arrive_cluster(smem_map_rank(&tempty[acc], 0));
        else asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty[acc])) : "memory");
      }
    }
    // Nothing may be in flight into or out of shared memory at exit: outstanding
    // block loads (only after an error) and the last block stores.
    if (lane == 0) {
      for (int bi = 0; bi < 2; ++bi)
        for (; nwait[bi] < nload[bi]; ++nwait[bi]) mbar_wait(&eb[bi], nwait[bi] & 1);
      bulk_wait_all();
    }
    (void)ep_ok;
  }
  tc_fence_before();
  // PAIR: neither CTA releases its TMEM or leaves while the leader's MMAs or the
  // peer's copies may still touch it.
  if (PAIR) cluster_sync_all();
  else __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    if (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BN) : "memory");
    else
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
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = wdt == WDT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(map_out), dt, 2, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// GEMM operand: row-major 16-bit [rows, cols] viewed as [cols / 64][rows][64]
// (dimension order x = element in chunk, y = row, z = 64-element chunk), with a
// box of 64 x 128 rows x KC chunks (KC = 1 and 2), 128-byte swizzle.  With
// `with_pair`, a second [rows, cols] matrix (the lo plane) follows the first
// one, and `pair` views both as [cols / 64][2][rows][64] (x = element, y = row,
// z = plane, w = chunk) with a box of 64 x 128 rows x 2 planes x 1 chunk: the
// hi block lands first, the lo block 16 KB after it.
bool make_tma_operand(TmaOperand* out, const void* base, uint64_t rows, uint64_t cols, int wdt, bool with_pair) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows % 128 || cols % 128 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  const CUtensorMapDataType dt = wdt == WDT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  for (int kc = 1; kc <= 2; ++kc) {
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, 128, (cuuint32_t)kc};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(&out->box[kc - 1], dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  memcpy(&out->pair, &out->box[0], sizeof(CUtensorMap));
  if (with_pair) {
    cuuint64_t dims[4] = {64, rows, 2, cols / 64};
    cuuint64_t strides[3] = {cols * 2, rows * cols * 2, 128};
    cuuint32_t box[4] = {64, 128, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(&out->pair, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

// Epilogue block map of a row-major [rows, cols] matrix: fp32 (elem_bytes 4,
// 128-byte swizzle) or the weight dtype (elem_bytes 2, 64-byte swizzle), box of
// 32 columns x 32 rows.  Stores outside [rows, cols] are dropped by the TMA.
bool make_tma_map_epilogue(void* map_out, const void* base, uint64_t rows, uint64_t cols, int elem_bytes, int wdt) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || cols % 32 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : wdt == WDT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = elem_bytes == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(map_out), dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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

template <typename WT, int WIDE>
static cudaError_t gemm_tc_configure_w() {
  constexpr int KN = WIDE ? 1 : 2;  // box depth of the 128-wide tiles
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_QKV, 256, 1, 0, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_QKV, 256, TC_PAIR_KC, 1, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_QKV, 128, KN, 0, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_GATEUP, 256, 1, 0, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_GATEUP, 256, TC_PAIR_KC, 1, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_RESID, 256, 1, 0, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  if ((e = cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_RESID, 256, TC_PAIR_KC, 1, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM))) return e;
  return cudaFuncSetAttribute(gemm_tc_kernel<WT, GEMM_RESID, 128, KN, 0, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
}

cudaError_t gemm_tc_configure() {
  cudaError_t e = gemm_tc_configure_w<bf16, 0>();
  if (e == cudaSuccess) e = gemm_tc_configure_w<f16, 0>();
  if (e == cudaSuccess) e = gemm_tc_configure_w<bf16, 1>();
  if (e == cudaSuccess) e = gemm_tc_configure_w<f16, 1>();
  return e;
}

// Tile width BN with its box depth: 256-wide tiles take 1-chunk boxes, 128-wide
// 2-chunk boxes (1-chunk with hi/lo operands, whose stages carry two A blocks
// per chunk).  256-wide tiles with an even number of m tiles run as paired
// 256 x 256 tiles on clusters of two CTAs, as many clusters as can be resident.
template <typename WT, int MODE, int BN, int WIDE>
static cudaError_t gemm_tc_go(const TmaOperand* a, const TmaOperand* const* b, const void* const* e,
                              const GemmParams& p, int mt, int nt, int num_sms, int* err, cudaStream_t s, bool pdl) {
  constexpr int KC = (BN == 256 || WIDE) ? 1 : 2;
  constexpr int BOX = (BN == 256 ? TC_PAIR_KC : KC) - 1;  // paired tiles use TC_PAIR_KC-chunk boxes
  TcMaps maps;
  memcpy(&maps.e_in, e[0] ? e[0] : &a->box[0], sizeof(CUtensorMap));
  memcpy(&maps.e_out, e[1] ? e[1] : &a->box[0], sizeof(CUtensorMap));
  if constexpr (BN == 256) {
    if (mt % 2 == 0) {
      memcpy(&maps.a, WIDE ? &a->pair : &a->box[BOX], sizeof(CUtensorMap));
      for (int i = 0; i < 3; ++i) memcpy(&maps.b[i], &(b[i] ? b[i] : b[0])->box[BOX], sizeof(CUtensorMap));
      auto kern = gemm_tc_kernel<WT, MODE, BN, TC_PAIR_KC, 1, WIDE>;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.blockDim = dim3(TC_THREADS);
      cfg.dynamicSmemBytes = TC_SMEM;
      cfg.stream = s;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      static int resident = 0;  // clusters of this kernel that fit on the GPU at once
      if (resident == 0) {
        cfg.gridDim = dim3(2 * (num_sms / 2));
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = num_sms / 2;
        resident = n;
      }
      const int units = (mt / 2) * nt;
      cfg.gridDim = dim3(2 * (units < resident ? units : resident));
      cudaLaunchAttribute attr2[2] = {attr[0], {}};
      attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr2[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr2;
      cfg.numAttrs = pdl ? 2 : 1;
      return cudaLaunchKernelEx(&cfg, kern, maps, p, mt, nt, err);
    }
  }
  memcpy(&maps.a, WIDE ? &a->pair : &a->box[KC - 1], sizeof(CUtensorMap));
  for (int i = 0; i < 3; ++i) memcpy(&maps.b[i], &(b[i] ? b[i] : b[0])->box[KC - 1], sizeof(CUtensorMap));
  const int total = mt * nt;
  const int grid = total < num_sms ? total : num_sms;
  return launch_k(gemm_tc_kernel<WT, MODE, BN, KC, 0, WIDE>, dim3(grid), dim3(TC_THREADS), (size_t)TC_SMEM, s, pdl,
                  maps, p, mt, nt, err);
}

// 256-wide tiles unless that leaves most SMs idle (narrow N at small M).
template <typename WT, int WIDE>
static cudaError_t gemm_tc_dispatch(const TmaOperand* a, const TmaOperand* const* b, const void* const* e,
                                    const GemmParams& p, int mode, int mt, int num_sms, int* err, cudaStream_t s,
                                    bool pdl) {
  if (mode == GEMM_GATEUP)
    return gemm_tc_go<WT, GEMM_GATEUP, 256, WIDE>(a, b, e, p, mt, p.N / 128, num_sms, err, s, pdl);
  const int nt256 = (p.N + 255) / 256;
  const bool narrow = (long long)mt * nt256 * 4 < (long long)num_sms * 3;
  if (mode == GEMM_RESID) {
    if (narrow) return gemm_tc_go<WT, GEMM_RESID, 128, WIDE>(a, b, e, p, mt, (p.N + 127) / 128, num_sms, err, s, pdl);
    return gemm_tc_go<WT, GEMM_RESID, 256, WIDE>(a, b, e, p, mt, nt256, num_sms, err, s, pdl);
  }
  if (narrow) return gemm_tc_go<WT, GEMM_QKV, 128, WIDE>(a, b, e, p, mt, (p.N + 127) / 128, num_sms, err, s, pdl);
  return gemm_tc_go<WT, GEMM_QKV, 256, WIDE>(a, b, e, p, mt, nt256, num_sms, err, s, pdl);
}

cudaError_t launch_gemm_tc(const TmaOperand* a, const TmaOperand* b0, const TmaOperand* b1, const TmaOperand* b2,
                           const void* e_in, const void* e_out, const GemmParams& p, int mode, int wdt, int num_sms,
                           int* err, cudaStream_t s, bool pdl, bool wide) {
  if (p.M <= 0) return cudaSuccess;
  // RESID reads and writes its rows through the epilogue maps, GATEUP writes through e_out
  if ((mode == GEMM_RESID && (!e_in || !e_out)) || (mode == GEMM_GATEUP && !e_out)) return cudaErrorInvalidValue;
  if (mode == GEMM_RESID && p.N % 256) return cudaErrorInvalidValue;  // every 32-column block of a tile exists
  if (wide && mode == GEMM_GATEUP && p.lo_row <= 0) return cudaErrorInvalidValue;  // where the lo plane's rows start
  const TmaOperand* b[3] = {b0, b1, b2};
  const void* e[2] = {e_in, e_out};
  const int mt = (p.M + TC_BM - 1) / TC_BM;
  if (wide)
    return wdt == WDT_F16 ? gemm_tc_dispatch<f16, 1>(a, b, e, p, mode, mt, num_sms, err, s, pdl)
                          : gemm_tc_dispatch<bf16, 1>(a, b, e, p, mode, mt, num_sms, err, s, pdl);
  return wdt == WDT_F16 ? gemm_tc_dispatch<f16, 0>(a, b, e, p, mode, mt, num_sms, err, s, pdl)
                        : gemm_tc_dispatch<bf16, 0>(a, b, e, p, mode, mt, num_sms, err, s, pdl);
}

}  // namespace ladder
