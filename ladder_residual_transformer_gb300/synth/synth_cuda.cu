// Device twin of synth.c's normal generator, for filling large weight tensors
// in place on the GPU.  It computes exactly the same bits as the host code:
// SplitMix64 counters, an Irwin-Hall sum of eight 16-bit uniforms (integer
// arithmetic), one IEEE fp32 multiply by the fp32 scale computed on the host,
// and round-to-nearest-even to bf16.  It holds no model arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t offset, uint64_t n, float scale, uint16_t* out) {
  for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n; j += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t i = offset + j;
    const uint64_t h0 = mix64(key + 2 * i);
    const uint64_t h1 = mix64(key + 2 * i + 1);
    int64_t s = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      s += (int64_t)((h0 >> (16 * b)) & 0xFFFFu);
      s += (int64_t)((h1 >> (16 * b)) & 0xFFFFu);
    }
    const int32_t c = (int32_t)(s - 4 * 65535);
    const float w = __fmul_rn((float)c, scale);
    uint32_t u = __float_as_uint(w);
    u += 0x7FFFu + ((u >> 16) & 1u);
    out[j] = (uint16_t)(u >> 16);
  }
}

// key = mix(mix(seed) ^ tensor_id), as in synth.c; scale from synth_normal_scale.
extern "C" int synth_normal_bf16_device(uint64_t key, uint64_t offset, uint64_t n, float scale, void* out,
                                        void* stream) {
  if (n == 0) return 0;
  const unsigned blocks = (unsigned)((n + 255) / 256 < 65535 * 4 ? (n + 255) / 256 : 65535 * 4);
  normal_bf16_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(key, offset, n, scale, (uint16_t*)out);
  return (int)cudaGetLastError();
}
