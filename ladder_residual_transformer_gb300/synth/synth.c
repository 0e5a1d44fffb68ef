/*
 * Seeded synthetic inputs for the Ladder Transformer forward pass.
 *
 * This file generates random-init weights and random token ids.  It holds none
 * of the model's arithmetic: both the CUDA path and the CPU oracle read the
 * values it writes, so that they are compared on bit-identical inputs.
 *
 * Generator (counter based, so any element can be produced independently):
 *   mix(z)      = the SplitMix64 output function (Steele, Lea and Flood,
 *                 "Fast splittable pseudorandom number generators", 2014):
 *                 z += 0x9E3779B97F4A7C15;
 *                 z  = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                 z  = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *                 return z ^ (z >> 31);
 *   key(s, t)   = mix(mix(s) ^ t)                  (seed s, tensor/stream id t)
 *   normal      : element i draws h0 = mix(key + 2i), h1 = mix(key + 2i + 1),
 *                 splits them into eight 16-bit uniforms, and sums them
 *                 (Irwin-Hall, n = 8).  The centred integer sum c = S - 4*65535
 *                 is exact in fp32 (|c| < 2^24); w = (float)c * scale with
 *                 scale = std / sqrt(8 * (65536^2 - 1) / 12) rounded once to
 *                 fp32, then w is rounded to bf16 (round to nearest, ties to
 *                 even).  Only integer operations and one IEEE fp32 multiply
 *                 are involved, so every platform produces the same bits.
 *   tokens      : token i = mix(key + i) mod vocab.
 */
#include <stdint.h>
#include <math.h>

static inline uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
  return mix64(mix64(seed) ^ tensor_id);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* The fp32 scale that maps the centred Irwin-Hall sum to standard deviation `std`. */
float synth_normal_scale(float std) {
  const double var_one = (65536.0 * 65536.0 - 1.0) / 12.0;
  return (float)((double)std / sqrt(8.0 * var_one));
}

/* out[j] = bf16 sample number (offset + j) of tensor `tensor_id` under `seed`. */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t offset, uint64_t n,
                       float std, uint16_t* out) {
  const uint64_t key = stream_key(seed, tensor_id);
  const float scale = synth_normal_scale(std);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nn; ++j) {
    uint64_t i = offset + (uint64_t)j;
    uint64_t h0 = mix64(key + 2 * i);
    uint64_t h1 = mix64(key + 2 * i + 1);
    int64_t s = 0;
    for (int b = 0; b < 4; ++b) {
      s += (int64_t)((h0 >> (16 * b)) & 0xFFFFu);
      s += (int64_t)((h1 >> (16 * b)) & 0xFFFFu);
    }
    int32_t c = (int32_t)(s - 4 * 65535);
    float w = (float)c * scale;
    out[j] = f32_to_bf16_rne(w);
  }
}

/* out[j] = fp32 value of the same sample as synth_normal_bf16 (exact widening of the bf16 bits). */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t offset, uint64_t n, float std, float* out) {
  const uint64_t key = stream_key(seed, tensor_id);
  const float scale = synth_normal_scale(std);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nn; ++j) {
    uint64_t i = offset + (uint64_t)j;
    uint64_t h0 = mix64(key + 2 * i);
    uint64_t h1 = mix64(key + 2 * i + 1);
    int64_t s = 0;
    for (int b = 0; b < 4; ++b) {
      s += (int64_t)((h0 >> (16 * b)) & 0xFFFFu);
      s += (int64_t)((h1 >> (16 * b)) & 0xFFFFu);
    }
    int32_t c = (int32_t)(s - 4 * 65535);
    union { float f; uint32_t u; } v;
    v.u = (uint32_t)f32_to_bf16_rne((float)c * scale) << 16;
    out[j] = v.f;
  }
}

/* out[j] = token number (offset + j) of stream `stream_id` under `seed`, in [0, vocab). */
void synth_tokens(uint64_t seed, uint64_t stream_id, uint64_t offset, uint64_t n,
                  uint32_t vocab, int32_t* out) {
  const uint64_t key = stream_key(seed, stream_id);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nn; ++j) {
    uint64_t i = offset + (uint64_t)j;
    out[j] = (int32_t)(mix64(key + i) % (uint64_t)vocab);
  }
}

/* Stream key of (seed, tensor id), for the device twin of the generator. */
uint64_t synth_stream_key(uint64_t seed, uint64_t tensor_id) { return stream_key(seed, tensor_id); }

/* Plain SplitMix64 output function, exported so tests can check it against its definition. */
uint64_t synth_mix64(uint64_t z) { return mix64(z); }
