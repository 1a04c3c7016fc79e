// k_append.cu -- CSA2 compressor and FP4 quantise-append into the global KV
// cache ("DeepSeek-V4.1-Flash" report: section 2.3 for the simplified
// compressor, section 2.4.4 for the FP4 main-KV format).
//
// One warp per output entry; lane l owns channels [16 l, 16 l + 16).  Every
// floating-point step that decides a code is written with explicit IEEE
// round-to-nearest intrinsics (no contraction), so the codes and the
// compressed values are fixed bit for bit by the order written here.
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

// exp for the compressor's per-channel softmax: Cody-Waite reduction with
// ln 2 split as 0.693359375 - 2.12194440e-4 (Cephes' expf split), degree-7
// Taylor polynomial in Horner form on fused multiply-adds, exact scaling by
// 2^n.  Defined on [-87, 88]; 0 below.
__device__ __forceinline__ float cw_expf(float x) {
  if (x != x) return x;
  if (x < -87.0f) return 0.0f;
  if (x > 88.0f) return __int_as_float(0x7f800000);
  const float t = __fmul_rn(x, 0x1.715476p+0f);  // log2(e) in fp32
  const float n = rintf(t);
  float r = __fmaf_rn(-n, 0x1.63p-1f, x);         // 0.693359375
  r = __fmaf_rn(-n, -0x1.bd0106p-13f, r);         // -2.12194440e-4
  float p = 0x1.a01a02p-13f;                      // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);           // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);            // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);            // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);            // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int ni = (int)n;                          // in [-126, 128] here
  const float two_n = __uint_as_float((uint32_t)(ni + 127) << 23);
  return __fmul_rn(p, two_n);
}

// Compressed value of one channel: softmax over the m logits of the block,
// fp32, j in increasing order, sums started from the j = 0 term.
__device__ __forceinline__ float compress_channel(const uint16_t* __restrict__ c,
                                                  const float* __restrict__ z, int m,
                                                  int64_t stride) {
  float mx = __ldg(z);
  for (int j = 1; j < m; ++j) {
    const float v = __ldg(z + j * stride);
    if (v > mx) mx = v;
  }
  float sum = 0.0f;
  for (int j = 0; j < m; ++j) {
    const float e = cw_expf(__fsub_rn(__ldg(z + j * stride), mx));
    sum = (j == 0) ? e : __fadd_rn(sum, e);
  }
  float acc = 0.0f;
  for (int j = 0; j < m; ++j) {
    const float e = cw_expf(__fsub_rn(__ldg(z + j * stride), mx));
    const float w = __fdiv_rn(e, sum);
    const float term = __fmul_rn(w, bf16_bits_to_float(__ldg(c + j * stride)));
    acc = (j == 0) ? term : __fadd_rn(acc, term);
  }
  return acc;
}

__global__ void __launch_bounds__(256) k_append(const __grid_constant__ AppendParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);

  if (blockIdx.x == 0 && p.mode != 0 && threadIdx.x < p.n_segs)
    p.d_len[p.seg[threadIdx.x].seq] = p.seg[threadIdx.x].new_len;
  if (row >= p.rows) return;

  int s = 0;
  while (s + 1 < p.n_segs && p.seg[s + 1].first <= row) ++s;
  const int64_t src = p.seg[s].src_row + (row - p.seg[s].first);
  const int64_t dst = p.seg[s].dst_row + (row - p.seg[s].first);
  const int dim = p.dim;
  const int c0 = lane * 16;
  if (c0 >= dim) return;
  if (p.mode != 0 && !CSA2_IN_BOUNDS(dst >= 0 && dst < p.total, p.err)) return;

  float x[16];
  if (p.mode == 1) {
    const float4* e4 = reinterpret_cast<const float4*>(p.entries + src * dim + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(e4 + i);
      x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
    }
  } else {
    const int m = p.ratio;
    const uint16_t* cb = p.c_tok + (src * m) * dim + c0;
    const float* zb = p.z_tok + (src * m) * dim + c0;
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = compress_channel(cb + i, zb + i, m, dim);
  }

  if (p.entries_out) {
    float4* o4 = reinterpret_cast<float4*>(p.entries_out + src * dim + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) o4[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
  }
  if (p.mode == 0) return;

  // ---- FP4 quantisation of the 16 channels of this lane
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  float sc;
  bool zero_scale = false;
  if (p.layout == 0) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // 32-channel block
    const uint32_t b = ue8m0_for_amax(amax);
    sc = ue8m0_value(b);
    if ((lane & 1) == 0) p.scales[dst * (kHeadDim / 32) + (lane >> 1)] = (uint8_t)b;
  } else {
    const uint32_t b = e4m3_encode_rn_sat(__fdiv_rn(amax, 6.0f));
    sc = e4m3_value(b);
    zero_scale = (sc == 0.0f);
    p.scales[dst * (kHeadDim / 16) + lane] = (uint8_t)b;
  }
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t c = zero_scale ? 0u : e2m1_encode(__fdiv_rn(x[i], sc));
    if (i < 8) lo |= c << (4 * i);
    else hi |= c << (4 * (i - 8));
  }
  *reinterpret_cast<uint2*>(p.codes + dst * kCodeBytes + lane * 8) = make_uint2(lo, hi);

  // ---- indexer key row: 4 channels per lane
  const uint2 kw = __ldg(reinterpret_cast<const uint2*>(p.idx_k + src * kIdxDim) + lane);
  if (!p.idx_mxfp4) {
    reinterpret_cast<uint2*>(p.cache_idxk + dst * kIdxDim)[lane] = kw;
    return;
  }
  // MXFP4 (V4.1 report, section 2.4.4): the 32-channel block of this lane is
  // held by 8 lanes; the scale and codes follow the L32 rule above
  const float k4[4] = {__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xFFFF0000u),
                       __uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xFFFF0000u)};
  float ka = fmaxf(fmaxf(fabsf(k4[0]), fabsf(k4[1])), fmaxf(fabsf(k4[2]), fabsf(k4[3])));
  ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, 1));
  ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, 2));
  ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, 4));
  const uint32_t kb = ue8m0_for_amax(ka);
  const float ks = ue8m0_value(kb);
  uint32_t kc = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) kc |= e2m1_encode(__fdiv_rn(k4[i], ks)) << (4 * i);
  reinterpret_cast<uint16_t*>(p.idx_codes + dst * (kIdxDim / 2))[lane] = (uint16_t)kc;
  if ((lane & 7) == 0) p.idx_scales[dst * (kIdxDim / 32) + (lane >> 3)] = (uint8_t)kb;
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  if (p.rows <= 0 && p.n_segs == 0) return cudaSuccess;
  const int64_t blocks = (p.rows + 7) / 8;
  k_append<<<(unsigned)(blocks > 0 ? blocks : 1), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
