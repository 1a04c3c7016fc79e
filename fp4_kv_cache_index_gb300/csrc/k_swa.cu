// k_swa.cu -- FP8 window rows (the V4.1 report, section 2.4.4, keeps the SWA
// KV cache in FP8; the row is the V4 FP8 entry of the cache breakdown: 448
// channels as E4M3 with one power-of-two UE8M0 scale per 64 channels, the 64
// RoPE channels in bf16, 8 scale bytes -- 584 bytes).
//
// One warp per row; lane l holds channels [16 l, 16 l + 16).  The scale of a
// 64-channel block follows the OCP MX rule for E4M3 elements (exponent of the
// block's largest magnitude minus 8), each code is the hardware's nearest-
// even, saturating E4M3 conversion of x / scale.
#include <cuda_fp8.h>

#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

__global__ void __launch_bounds__(256) k_swa_fp8(const uint16_t* __restrict__ rows, int64_t n,
                                                 uint8_t* __restrict__ codes,
                                                 uint16_t* __restrict__ rope,
                                                 uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= n) return;
  const uint4* src = reinterpret_cast<const uint4*>(rows + r * 512 + lane * 16);
  const uint4 a = __ldg(src), b = __ldg(src + 1);
  if (lane >= 28) {   // RoPE channels 448..511: bf16 bits unchanged
    uint4* dst = reinterpret_cast<uint4*>(rope + r * 64 + (lane - 28) * 16);
    dst[0] = a;
    dst[1] = b;
    if (lane == 28) scales[r * 8 + 7] = 0;
    return;
  }
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  // the 4 lanes of a 64-channel block (lanes 28-31 have left: mask 0x0FFFFFFF)
  amax = fmaxf(amax, __shfl_xor_sync(0x0FFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0x0FFFFFFFu, amax, 2));
  const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  const uint32_t sb = (uint32_t)(ex >= 8 ? ex - 8 : 0);
  const float sc = ue8m0_value(sb);
  uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t c =
        (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[i], sc), __NV_SATFINITE, __NV_E4M3);
    out[i >> 2] |= c << (8 * (i & 3));
  }
  *reinterpret_cast<uint4*>(codes + r * 448 + lane * 16) = make_uint4(out[0], out[1], out[2], out[3]);
  if ((lane & 3) == 0) scales[r * 8 + (lane >> 2)] = (uint8_t)sb;
}

}  // namespace

cudaError_t launch_swa_fp8(const uint16_t* rows, int64_t n, uint8_t* codes, uint16_t* rope,
                           uint8_t* scales, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_swa_fp8<<<(unsigned)((n + 7) / 8), 256, 0, s>>>(rows, n, codes, rope, scales);
  return cudaGetLastError();
}

}  // namespace csa2
