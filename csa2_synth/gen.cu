// Device twin of csa2_synth: fills device buffers with the same seeded
// values as the numpy generator (SplitMix64 counter form + Irwin-Hall sum of
// twelve 16-bit uniforms).  Used only to build large synthetic workloads on
// the GPU quickly; it holds none of the attention method's arithmetic.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float ih_normal(uint64_t key, uint64_t i) {
  int64_t tot = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    uint64_t r = mix64(key + (3 * i + j + 1) * kGamma);
    tot += (int64_t)(r & 0xFFFF) + (int64_t)((r >> 16) & 0xFFFF) +
           (int64_t)((r >> 32) & 0xFFFF) + (int64_t)(r >> 48);
  }
  // |tot - mean| < 2^19: exact in fp32, then an exact power-of-two scaling.
  return __int2float_rn((int)(tot - 393210)) * 0x1p-16f;
}

__device__ __forceinline__ uint16_t bf16_rne(float f) {
  uint32_t b = __float_as_uint(f);
  return (uint16_t)((b + (((b >> 16) & 1u) + 0x7FFFu)) >> 16);
}

__global__ void fill_f32(uint64_t key, uint64_t first, uint64_t n, float scale,
                         float* __restrict__ out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = ih_normal(key, first + i) * scale;
}

__global__ void fill_bf16(uint64_t key, uint64_t first, uint64_t n, float scale,
                          uint16_t* __restrict__ out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = bf16_rne(ih_normal(key, first + i) * scale);
}

}  // namespace

extern "C" {

// scale must be a power of two (1 or 8 in the workloads) so that scaling and
// rounding commute and the result equals the host generator's.
int csa2_synth_fill_f32(uint64_t key, uint64_t first, uint64_t n, float scale,
                        float* out, cudaStream_t stream) {
  if (n == 0) return 0;
  fill_f32<<<1216, 256, 0, stream>>>(key, first, n, scale, out);
  return (int)cudaGetLastError();
}

int csa2_synth_fill_bf16(uint64_t key, uint64_t first, uint64_t n, float scale,
                         uint16_t* out, cudaStream_t stream) {
  if (n == 0) return 0;
  fill_bf16<<<1216, 256, 0, stream>>>(key, first, n, scale, out);
  return (int)cudaGetLastError();
}

}  // extern "C"
