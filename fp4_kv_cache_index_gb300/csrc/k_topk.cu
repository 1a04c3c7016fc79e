// k_topk.cu -- exact top-k of fp32 index scores per query (blog reading of
// the DeepSeek-V4 report, section 4.1: keep the top-k compressed entries;
// V4.1 report section 4.2.1: k = 512).
//
// One CTA per row.  Scores become order-preserving 32-bit keys (-0 folded to
// +0).  A radix select over the digits [31:21], [20:10], [9:0] finds the k-th
// largest key T and the count of keys above it:
//   - digit 1 is a shared-memory histogram of the whole row;
//   - when the bin holding T is small, its keys are gathered into shared
//     memory and digits 2-3 run there; otherwise digits 2-3 re-read the row.
// A final ordered pass emits, in increasing index order, every key > T and
// the first (k - count_above) keys == T, so ties go to the lower index and
// the output is sorted by index.  Integer atomics only: the result is the
// same on every run.
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kCandCap = 8192;

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Shared {
  uint32_t hist[kBins];
  uint32_t cand[kCandCap];
  uint32_t warp_sum[kWarps];
  uint32_t n_cand;
  uint32_t sel_bin;
  uint32_t sel_above;
  uint32_t done;
};

// Inclusive suffix sum over the block (thread t gets sum over t' >= t).
__device__ __forceinline__ uint32_t block_suffix_sum(uint32_t v, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_down_sync(0xffffffffu, v, o);
    if (lane + o < 32) v += n;
  }
  if (lane == 0) sh.warp_sum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = sh.warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_down_sync(0xffffffffu, w, o);
      if (lane + o < 32) w += n;
    }
    sh.warp_sum[lane] = w;  // inclusive suffix over warps
  }
  __syncthreads();
  const uint32_t later = (warp + 1 < kWarps) ? sh.warp_sum[warp + 1] : 0u;
  __syncthreads();
  return v + later;
}

// Inclusive prefix sum over the block.
__device__ __forceinline__ uint32_t block_prefix_sum(uint32_t v, Shared& sh, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sh.warp_sum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = sh.warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    sh.warp_sum[lane] = w;
  }
  __syncthreads();
  const uint32_t before = warp ? sh.warp_sum[warp - 1] : 0u;
  total = sh.warp_sum[kWarps - 1];
  __syncthreads();
  return v + before;
}

// Adds one to hist[bin] for every active lane, one atomic per distinct bin.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool active, uint32_t bin) {
  const uint32_t key = active ? bin : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, key);
  const int lane = threadIdx.x & 31;
  if (active && lane == __ffs(peers) - 1) atomicAdd(hist + bin, (uint32_t)__popc(peers));
}

// Picks the bin holding the rem-th largest key among those counted in hist
// (nbins <= 2 * kThreads); records it and the count strictly above it.
__device__ __forceinline__ void select_bin(Shared& sh, int nbins, uint32_t rem) {
  const int t = threadIdx.x;
  const uint32_t h0 = (2 * t < nbins) ? sh.hist[2 * t] : 0u;
  const uint32_t h1 = (2 * t + 1 < nbins) ? sh.hist[2 * t + 1] : 0u;
  const uint32_t suf = block_suffix_sum(h0 + h1, sh);  // sum over bins >= 2t
  const uint32_t suf1 = suf - h0;                        // bins >= 2t+1
  const uint32_t suf2 = suf1 - h1;                       // bins >= 2t+2
  if (2 * t + 1 < nbins && suf1 >= rem && suf2 < rem) { sh.sel_bin = 2 * t + 1; sh.sel_above = suf2; }
  if (2 * t < nbins && suf >= rem && suf1 < rem) { sh.sel_bin = 2 * t; sh.sel_above = suf1; }
  __syncthreads();
}

__device__ __forceinline__ void load4(const float* row, int64_t e, int64_t n, bool vec, float (&v)[4]) {
  if (vec && e + 3 < n) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(row + e));
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (e + i < n) ? __ldg(row + e + i) : 0.0f;
  }
}

__device__ __forceinline__ void clear_hist(Shared& sh) {
  for (int i = threadIdx.x; i < kBins; i += kThreads) sh.hist[i] = 0u;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) k_topk(const __grid_constant__ TopkParams p,
                                                       int row0) {
  extern __shared__ uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  const int row = row0 + blockIdx.x;
  if (row >= p.rows) return;
  int64_t n;
  if (p.formula) {
    const int64_t v = (p.pos0 + row + 1) / p.ratio;
    n = v < p.pre_len ? v : p.pre_len;
  } else {
    n = p.n_valid[row];
  }
  const int k = p.k;
  const float* srow = p.scores + (int64_t)row * p.ld;
  int32_t* orow = p.idx_out + (int64_t)row * k;
  float* osc = p.score_out ? p.score_out + (int64_t)row * k : nullptr;
  const int tid = threadIdx.x;

  if (n <= k) {
    for (int i = tid; i < k; i += kThreads) {
      orow[i] = (i < n) ? i : -1;
      if (osc) osc[i] = (i < n) ? srow[i] : 0.0f;
    }
    return;
  }
  const bool vec = ((reinterpret_cast<uintptr_t>(srow) & 15u) == 0);
  const int64_t chunk = (int64_t)kThreads * 4;

  // ---- digit 1: keys [31:21] over the whole row
  clear_hist(sh);
  if (tid == 0) sh.n_cand = 0;
  // every loop below runs the same trip count in all threads (block-uniform
  // chunk loop) so that the warp-collective intrinsics see full warps
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    const int64_t e = c0 + (int64_t)tid * 4;
    float v[4];
    load4(srow, e, n, vec, v);
#pragma unroll
    for (int i = 0; i < 4; ++i) hist_add(sh.hist, e + i < n, score_key(v[i]) >> 21);
  }
  __syncthreads();
  select_bin(sh, kBins, (uint32_t)k);
  uint32_t prefix = sh.sel_bin;  // high bits of T found so far
  uint32_t above = sh.sel_above;
  const uint32_t in_bin = sh.hist[prefix];
  __syncthreads();

  if (in_bin <= (uint32_t)kCandCap) {
    // ---- gather the keys of the selected bin, then digits 2 and 3 in smem
    for (int64_t c0 = 0; c0 < n; c0 += chunk) {
      const int64_t e = c0 + (int64_t)tid * 4;
      float v[4];
      load4(srow, e, n, vec, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t key = score_key(v[i]);
        const bool hit = (e + i < n) && (key >> 21) == prefix;
        const uint32_t b = __ballot_sync(0xffffffffu, hit);
        uint32_t base = 0;
        if ((tid & 31) == 0 && b) base = atomicAdd(&sh.n_cand, (uint32_t)__popc(b));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (hit) sh.cand[base + __popc(b & ((1u << (tid & 31)) - 1u))] = key;
      }
    }
    __syncthreads();
    const uint32_t nc = sh.n_cand;
    // digit 2: bits [20:10]
    clear_hist(sh);
    for (uint32_t i = tid; i < ((nc + 31u) & ~31u); i += kThreads) {
      const bool ok = i < nc;
      const uint32_t key = ok ? sh.cand[i] : 0u;
      hist_add(sh.hist, ok, (key >> 10) & 0x7FFu);
    }
    __syncthreads();
    select_bin(sh, kBins, (uint32_t)k - above);
    prefix = (prefix << 11) | sh.sel_bin;
    above += sh.sel_above;
    __syncthreads();
    // digit 3: bits [9:0]
    clear_hist(sh);
    for (uint32_t i = tid; i < ((nc + 31u) & ~31u); i += kThreads) {
      const bool ok = i < nc && (sh.cand[i] >> 10) == prefix;
      const uint32_t key = (i < nc) ? sh.cand[i] : 0u;
      hist_add(sh.hist, ok, key & 0x3FFu);
    }
    __syncthreads();
    select_bin(sh, 1024, (uint32_t)k - above);
    prefix = (prefix << 10) | sh.sel_bin;
    above += sh.sel_above;
    __syncthreads();
  } else {
    // ---- a crowded bin (many equal or near-equal scores): digits 2 and 3
    //      re-read the row with the prefix as a filter
    clear_hist(sh);
    for (int64_t c0 = 0; c0 < n; c0 += chunk) {
      const int64_t e = c0 + (int64_t)tid * 4;
      float v[4];
      load4(srow, e, n, vec, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t key = score_key(v[i]);
        hist_add(sh.hist, (e + i < n) && (key >> 21) == prefix, (key >> 10) & 0x7FFu);
      }
    }
    __syncthreads();
    select_bin(sh, kBins, (uint32_t)k - above);
    prefix = (prefix << 11) | sh.sel_bin;
    above += sh.sel_above;
    __syncthreads();
    clear_hist(sh);
    for (int64_t c0 = 0; c0 < n; c0 += chunk) {
      const int64_t e = c0 + (int64_t)tid * 4;
      float v[4];
      load4(srow, e, n, vec, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t key = score_key(v[i]);
        hist_add(sh.hist, (e + i < n) && (key >> 10) == prefix, key & 0x3FFu);
      }
    }
    __syncthreads();
    select_bin(sh, 1024, (uint32_t)k - above);
    prefix = (prefix << 10) | sh.sel_bin;
    above += sh.sel_above;
    __syncthreads();
  }

  // ---- ordered emission: keys > T, then the first (k - above) keys == T
  const uint32_t T = prefix;
  const uint32_t need_eq = (uint32_t)k - above;
  uint32_t base_gt = 0, base_eq = 0;
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    const int64_t e = c0 + (int64_t)tid * 4;
    float v[4];
    load4(srow, e, n, vec, v);
    uint32_t gt = 0, eq = 0;
    uint32_t key[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      key[i] = score_key(v[i]);
      const bool ok = e + i < n;
      gt += (ok && key[i] > T);
      eq += (ok && key[i] == T);
    }
    uint32_t tot;
    const uint32_t incl = block_prefix_sum(gt | (eq << 16), sh, tot);
    uint32_t g_before = base_gt + ((incl - (gt | (eq << 16))) & 0xFFFFu);
    uint32_t q_before = base_eq + ((incl - (gt | (eq << 16))) >> 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (e + i >= n) break;
      const bool is_gt = key[i] > T, is_eq = key[i] == T;
      if (is_gt || (is_eq && q_before < need_eq)) {
        const uint32_t pos = g_before + (q_before < need_eq ? q_before : need_eq);
        orow[pos] = (int32_t)(e + i);
        if (osc) osc[pos] = v[i];
      }
      g_before += is_gt;
      q_before += is_eq;
    }
    base_gt += tot & 0xFFFFu;
    base_eq += tot >> 16;
    if (base_gt + (base_eq < need_eq ? base_eq : need_eq) >= (uint32_t)k) break;
  }
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
  const int smem = (int)sizeof(Shared);
  cudaError_t e = cudaFuncSetAttribute(k_topk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  for (int r0 = 0; r0 < p.rows; r0 += kTopkMaxRowsPerLaunch) {
    const int nr = (p.rows - r0 < kTopkMaxRowsPerLaunch) ? p.rows - r0 : kTopkMaxRowsPerLaunch;
    k_topk<<<nr, kThreads, smem, s>>>(p, r0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa2
