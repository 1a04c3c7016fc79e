// k_hsi.cu -- pieces of the Hierarchical Sparse Indexer ("DeepSeek-V4.1-Flash"
// report, section 2.3.2): block scores (maximum index score of 8 consecutive
// positions) that feed the block top-k, and the mapping from a Reindex
// layer's selected pool slots back to entry indices.  The pool scoring itself
// is the indexer kernel in pool mode (k_index.cu).
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

// One thread per block of 8 scores (two 16-byte loads when aligned).
__global__ void __launch_bounds__(256) k_block_max(const __grid_constant__ HsiParams p) {
  const int r = blockIdx.y;
  const int64_t n = p.n[r];
  const int64_t nb = (n + kHsiBlock - 1) / kHsiBlock;
  const float* row = p.scores + (int64_t)r * p.ld;
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nb;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e0 = b * kHsiBlock;
    float m = -INFINITY;
    if (e0 + kHsiBlock <= n && ((reinterpret_cast<uintptr_t>(row + e0) & 15u) == 0)) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(row + e0));
      const float4 c = __ldg(reinterpret_cast<const float4*>(row + e0) + 1);
      m = fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(c.x, c.y), fmaxf(c.z, c.w)));
    } else {
      for (int i = 0; i < kHsiBlock && e0 + i < n; ++i) m = fmaxf(m, __ldg(row + e0 + i));
    }
    if (CSA2_IN_BOUNDS(b < p.ld_b, p.err)) p.bmax[(int64_t)r * p.ld_b + b] = m;
  }
}

__global__ void __launch_bounds__(256) k_pool_map(const __grid_constant__ HsiParams p) {
  const int r = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= p.k) return;
  const int32_t slot = p.sel[(int64_t)r * p.k + j];
  int32_t e = -1;
  if (slot >= 0) {
    const int32_t blk = p.pool[(int64_t)r * p.pool_blocks + slot / kHsiBlock];
    const int64_t ent = (int64_t)blk * kHsiBlock + slot % kHsiBlock;
    if (blk >= 0 && ent < p.n[r]) e = (int32_t)ent;
  }
  p.out[(int64_t)r * p.k + j] = e;
  if (p.score_out && e < 0) p.score_out[(int64_t)r * p.k + j] = 0.0f;
}

}  // namespace

cudaError_t launch_block_max(const HsiParams& p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  int64_t nb = 1;
  for (int r = 0; r < p.rows; ++r) nb = p.n[r] / kHsiBlock + 1 > nb ? p.n[r] / kHsiBlock + 1 : nb;
  const int gx = (int)((nb + 255) / 256 < 64 ? (nb + 255) / 256 : 64);
  k_block_max<<<dim3(gx, p.rows), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_pool_map(const HsiParams& p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  k_pool_map<<<dim3((p.k + 255) / 256, p.rows), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace csa2
