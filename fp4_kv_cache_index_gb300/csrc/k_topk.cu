// k_topk.cu -- exact top-k of fp32 index scores per query (blog reading of
// the DeepSeek-V4 report, section 4.1: keep the top-k compressed entries;
// V4.1 report section 4.2.1: k = 512), or of bf16-rounded scores (same
// blog, section 7), read as 16-bit values and handled as their fp32.
//
// One CTA per row.  Scores become order-preserving 32-bit keys (-0 folded to
// +0).  The k-th largest key T is found by a radix select over the digits
// [31:21], [20:10], [9:0]:
//   1. the digit-1 histogram comes from the indexer (score-key histogram) or
//      from one pass over the row into eight replicated shared histograms;
//      it gives the bin b1 that holds T and the count of keys above b1;
//   2. when those candidates (keys in bins >= b1, a few thousand for
//      continuous scores) fit in shared memory, one ordered pass compacts
//      them, in index order, and digits 2-3 plus the emission run there;
//      With a score-key histogram and a scratch buffer, that compaction is
//      split over segments of 8192 scores, one CTA each (k_topk_seg), and
//      the row's CTA reads the segments back in order;
//   3. otherwise (many equal or nearly equal scores) digits 2-3 and the
//      emission re-read the row.
// Emission writes, in increasing index order, every key > T and the first
// (k - count above T) keys == T: ties go to the lower index.  Integer
// atomics only, so the result is the same on every run.
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

// Row kernel: kT threads per row, 1024 (one row per SM, for a few long
// rows) or 512 (two rows per SM, for many rows: one row's block-wide steps
// overlap the other's loads).
constexpr int kBins = 2048;
constexpr int kCandCap = 8192;
constexpr int kSubHists = 8;
constexpr int kTopkManyRows = 512;   // rows of a launch from which kT = 512


template <int kT>
struct Shared {
  uint32_t hist[kBins];
  union {
    struct {
      uint32_t key[kCandCap];
      int32_t idx[kCandCap];
    } cand;
    uint32_t sub[kSubHists][kBins];
  } u;
  uint32_t warp_sum[kT / 32];
  uint32_t sel_bin;
  uint32_t sel_above;
};

// Inclusive suffix sum over the block (thread t gets the sum over t' >= t).
template <int kT>
__device__ __forceinline__ uint32_t block_suffix_sum(uint32_t v, Shared<kT>& sh) {
  constexpr int kWarps = kT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_down_sync(0xffffffffu, v, o);
    if (lane + o < 32) v += n;
  }
  if (lane == 0) sh.warp_sum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? sh.warp_sum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_down_sync(0xffffffffu, w, o);
      if (lane + o < 32) w += n;
    }
    if (lane < kWarps) sh.warp_sum[lane] = w;
  }
  __syncthreads();
  const uint32_t later = (warp + 1 < kWarps) ? sh.warp_sum[warp + 1] : 0u;
  __syncthreads();
  return v + later;
}

// Inclusive prefix sum over the block; `total` gets the block sum.
template <int kT>
__device__ __forceinline__ uint32_t block_prefix_sum(uint32_t v, Shared<kT>& sh,
                                                     uint32_t& total) {
  constexpr int kWarps = kT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) sh.warp_sum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? sh.warp_sum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kWarps) sh.warp_sum[lane] = w;
  }
  __syncthreads();
  const uint32_t before = warp ? sh.warp_sum[warp - 1] : 0u;
  total = sh.warp_sum[kWarps - 1];
  __syncthreads();
  return v + before;
}

// One atomic per distinct bin of the warp (for rows whose keys may all be
// equal); called by full warps only.
__device__ __forceinline__ void hist_add_aggregated(uint32_t* hist, bool active, uint32_t bin) {
  const uint32_t key = active ? bin : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, key);
  if (active && (int)(threadIdx.x & 31) == __ffs(peers) - 1)
    atomicAdd(hist + bin, (uint32_t)__popc(peers));
}

// "The key of f lies in a digit-1 bin >= b1", on the raw bits of f.  For b1
// above the bin of +0 (b1 > 1024) the keys >= b1 << 21 are exactly the
// floats whose bits, read as a signed integer, are >= (b1 << 21) & 0x7FFFFFFF:
// negative floats and -0 (whose key equals that of +0) fall below it, +NaN
// above, as their keys do.  Otherwise the key itself is formed.
struct BinTest {
  uint32_t b1;
  int32_t t;
  bool fast;
  __device__ __forceinline__ explicit BinTest(uint32_t b)
      : b1(b), t((int32_t)((b << 21) & 0x7FFFFFFFu)), fast(b > 1024u) {}
  __device__ __forceinline__ bool operator()(float f) const {
    return fast ? (int32_t)__float_as_uint(f) >= t : (score_key(f) >> 21) >= b1;
  }
};

// Bin holding the rem-th largest key counted in hist (nbins = 1024 or 2048,
// a multiple of kT: thread t holds bins [nb t, nb t + nb)); records it and
// the count strictly above it.
template <int kT>
__device__ __forceinline__ void select_bin(Shared<kT>& sh, int nbins, uint32_t rem) {
  constexpr int kMaxB = kBins / kT;
  const int t = threadIdx.x, nb = nbins / kT;
  uint32_t h[kMaxB], mine = 0u;
#pragma unroll
  for (int j = 0; j < kMaxB; ++j) {
    h[j] = j < nb ? sh.hist[nb * t + j] : 0u;
    mine += h[j];
  }
  const uint32_t suf = block_suffix_sum<kT>(mine, sh);   // bins >= nb t
  uint32_t above = suf - mine;                             // bins >= nb t + nb
#pragma unroll
  for (int j = kMaxB - 1; j >= 0; --j) {
    if (j < nb) {
      if (above < rem && above + h[j] >= rem) { sh.sel_bin = nb * t + j; sh.sel_above = above; }
      above += h[j];
    }
  }
  __syncthreads();
}

// A row of scores: fp32, or bf16 (uint16) when the selector runs on
// bf16-rounded scores; either way a score is handled as the fp32 of its value.
struct ScoreRow {
  const void* base;
  bool bf16;
  __device__ __forceinline__ float at(int64_t i) const {
    return bf16 ? bf16_bits_to_float(__ldg(static_cast<const uint16_t*>(base) + i))
                : __ldg(static_cast<const float*>(base) + i);
  }
  __device__ __forceinline__ bool aligned16() const {
    return (reinterpret_cast<uintptr_t>(base) & 15u) == 0;
  }
  // v[0..7] = scores e .. e + 7 (caller: e % 8 == 0, the row 16-byte aligned)
  __device__ __forceinline__ void load8(int64_t e, float* v) const {
    if (bf16) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + e));
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    } else {
      const float4* f4 = reinterpret_cast<const float4*>(static_cast<const float*>(base) + e);
      const float4 a = __ldg(f4), b = __ldg(f4 + 1);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
  }
};

__device__ __forceinline__ ScoreRow score_row(const TopkParams& p, int row) {
  ScoreRow r;
  r.bf16 = p.score_bf16 != 0;
  r.base = r.bf16 ? static_cast<const void*>(reinterpret_cast<const uint16_t*>(p.scores) +
                                             (int64_t)row * p.ld)
                  : static_cast<const void*>(p.scores + (int64_t)row * p.ld);
  return r;
}

// Each thread takes kPer consecutive scores per chunk (16-byte loads when
// the row is 16-byte aligned).
constexpr int kPer = 8;
__device__ __forceinline__ void load_run(const ScoreRow& row, int64_t e, int64_t n, bool vec,
                                         float (&v)[kPer]) {
  if (vec && e + kPer - 1 < n) {
    row.load8(e, v);
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] = (e + i < n) ? row.at(e + i) : 0.0f;
  }
}

template <int kT>
__device__ __forceinline__ void clear(uint32_t* h, int n) {
  for (int i = threadIdx.x; i < n; i += kT) h[i] = 0u;
  __syncthreads();
}

// Scratch of one (row, segment): [count][pad to 16 B][key x cap][idx x cap].
constexpr int kSegWords = 4 + 2 * kCandCap;

__device__ __forceinline__ int64_t row_valid_count(const TopkParams& p, int row) {
  if (p.formula) {
    const int64_t v = (p.pos0 + row + 1) / p.ratio;
    return v < p.pre_len ? v : p.pre_len;
  }
  return p.n_valid[row];
}

// Ordered compaction of one segment's candidates (keys in bins >= b1).  256
// threads, each owning 32 consecutive scores, in two passes over them:
// count (after an L2 prefetch issued with the histogram loads), then re-read
// the 8-score chunks that hold candidates and write them in index order.
// Holding no scores across the block-wide steps keeps the registers low
// enough for 8 CTAs per SM: a batch of 64 x 128K scores is one wave.
constexpr int kSegThreads = 256;
constexpr int kSegWarps = kSegThreads / 32;
constexpr int kSegPer = kTopkSegLen / kSegThreads;  // 32
constexpr int kSegBinsPer = kBins / kSegThreads;    // 8
struct SegShared {
  uint32_t warp_sum[kSegWarps];
  uint32_t sel_bin, sel_above, sel_count;
};

// Scores e0 + 8q .. e0 + 8q + 7 of the row (0 past n).
__device__ __forceinline__ void seg_chunk(const ScoreRow& srow, int64_t e0, int q, int64_t n,
                                          bool vec, float (&v)[8]) {
  if (vec) {
    srow.load8(e0 + 8 * q, v);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = (e0 + 8 * q + i < n) ? srow.at(e0 + 8 * q + i) : 0.0f;
  }
}

__global__ void __launch_bounds__(kSegThreads, 8) k_topk_seg(const __grid_constant__ TopkParams p,
                                                             int row0) {
  __shared__ SegShared sh;
  griddep_wait();
  const int row = row0 + blockIdx.y, seg = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  if (row >= p.rows) return;
  const int64_t n = row_valid_count(p, row);
  uint32_t* out = p.seg_ws + ((int64_t)row * p.n_seg + seg) * kSegWords;
  const int64_t s0 = (int64_t)seg * kTopkSegLen;
  if (n <= p.k || s0 >= n) {
    if (tid == 0) out[0] = 0u;
    return;
  }
  const ScoreRow srow = score_row(p, row);
  const int64_t e0 = s0 + (int64_t)tid * kSegPer;
  const bool vec = srow.aligned16() && e0 + kSegPer <= n;
  if (e0 < n) {
    const char* a = static_cast<const char*>(srow.base) + e0 * (srow.bf16 ? 2 : 4);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
  }
  // threshold bin: thread t holds bins [8t, 8t + 8)
  const uint4* hp = reinterpret_cast<const uint4*>(p.key_hist + (int64_t)row * kBins) + 2 * tid;
  const uint4 ha = __ldg(hp), hb = __ldg(hp + 1);
  const uint32_t h[kSegBinsPer] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
  uint32_t hs = 0;
#pragma unroll
  for (int i = 0; i < kSegBinsPer; ++i) hs += h[i];
  uint32_t suf = hs;  // inclusive suffix over the threads of the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += t;
  }
  if (lane == 0) sh.warp_sum[warp] = suf;
  __syncthreads();
  for (int w = warp + 1; w < kSegWarps; ++w) suf += sh.warp_sum[w];   // bins >= 8 tid
  const uint32_t k = (uint32_t)p.k;
  uint32_t above_mine = suf - hs;                                      // bins >= 8 tid + 8
#pragma unroll
  for (int i = kSegBinsPer - 1; i >= 0; --i) {
    if (above_mine < k && above_mine + h[i] >= k) {
      sh.sel_bin = kSegBinsPer * tid + i;
      sh.sel_above = above_mine;
      sh.sel_count = h[i];
    }
    above_mine += h[i];
  }
  __syncthreads();
  const uint32_t b1 = sh.sel_bin;
  if (sh.sel_above + sh.sel_count > (uint32_t)kCandCap) return;  // the row falls back
  // pass 1: which of the 32 scores are candidates
  const BinTest in_bins(b1);
  const int lim = (int)(n - e0 > kSegPer ? kSegPer : n - e0);   // e0 < n here or lim <= 0
  uint32_t mask = 0;
#pragma unroll
  for (int q = 0; q < kSegPer / 8; ++q) {
    float v[8];
    seg_chunk(srow, e0, q, n, vec, v);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      mask |= (uint32_t)(8 * q + i < lim && in_bins(v[i])) << (8 * q + i);
  }
  const uint32_t cnt = (uint32_t)__popc(mask);
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();   // every warp has read the warp_sum values of the first scan
  if (lane == 31) sh.warp_sum[warp] = incl;
  __syncthreads();
  uint32_t before = 0, total = 0;
  for (int w = 0; w < kSegWarps; ++w) {
    const uint32_t ws = sh.warp_sum[w];
    if (w < warp) before += ws;
    total += ws;
  }
  // pass 2: the chunks holding candidates again, written in index order
  uint32_t pos = before + incl - cnt;
#pragma unroll
  for (int q = 0; q < kSegPer / 8; ++q) {
    if (((mask >> (8 * q)) & 0xFFu) == 0u) continue;
    float v[8];
    seg_chunk(srow, e0, q, n, vec, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((mask >> (8 * q + i)) & 1u) {
        if (pos < (uint32_t)kCandCap) {
          out[4 + pos] = score_key(v[i]);
          out[4 + kCandCap + pos] = (uint32_t)(e0 + 8 * q + i);
        }
        ++pos;
      }
    }
  }
  if (tid == 0) out[0] = total < (uint32_t)kCandCap ? total : (uint32_t)kCandCap;
}

template <int kT>
__global__ void __launch_bounds__(kT, 1024 / kT) k_topk(const __grid_constant__ TopkParams p,
                                                         int row0) {
  constexpr int kThreads = kT;
  extern __shared__ uint8_t smem_raw[];
  Shared<kT>& sh = *reinterpret_cast<Shared<kT>*>(smem_raw);
  griddep_wait();
  const int row = row0 + blockIdx.x;
  if (row >= p.rows) return;
  const int64_t n = row_valid_count(p, row);
  const int k = p.k;
  const ScoreRow srow = score_row(p, row);
  int32_t* orow = p.idx_out + (int64_t)row * k;
  float* osc = p.score_out ? p.score_out + (int64_t)row * k : nullptr;
  const int tid = threadIdx.x, warp = tid >> 5;

  if (n <= k) {
    for (int i = tid; i < k; i += kThreads) {
      orow[i] = (i < n) ? i : -1;
      if (osc) osc[i] = (i < n) ? key_score(score_key(srow.at(i))) : 0.0f;
    }
    return;
  }
  const bool vec = srow.aligned16();
  const int64_t chunk = (int64_t)kThreads * kPer;

  // ---- digit 1: keys [31:21]
  if (p.key_hist) {
    const uint32_t* hrow = p.key_hist + (int64_t)row * kBins;
    for (int i = tid; i < kBins; i += kThreads) sh.hist[i] = hrow[i];
    __syncthreads();
  } else {
    clear<kT>(&sh.u.sub[0][0], kSubHists * kBins);
    uint32_t* mine = sh.u.sub[warp & (kSubHists - 1)];
    for (int64_t c0 = 0; c0 < n; c0 += chunk) {
      const int64_t e = c0 + (int64_t)tid * kPer;
      float v[kPer];
      load_run(srow, e, n, vec, v);
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (e + i < n) atomicAdd(mine + (score_key(v[i]) >> 21), 1u);
    }
    __syncthreads();
    for (int i = tid; i < kBins; i += kThreads) {
      uint32_t s = 0;
#pragma unroll
      for (int j = 0; j < kSubHists; ++j) s += sh.u.sub[j][i];
      sh.hist[i] = s;
    }
    __syncthreads();
  }
  select_bin<kT>(sh, kBins, (uint32_t)k);
  const uint32_t b1 = sh.sel_bin;
  uint32_t above = sh.sel_above;
  const uint32_t n_cand = above + sh.hist[b1];
  __syncthreads();

  uint32_t T;
  if (n_cand <= (uint32_t)kCandCap && p.seg_ws && p.key_hist) {
    // ---- candidates from the segments, concatenated in segment order: all
    //      counts are read at once (one segment per thread), their exclusive
    //      prefix goes to sh.hist (free until digit 2), and each candidate
    //      position finds its segment by binary search
    const int nseg = (int)((n + kTopkSegLen - 1) / kTopkSegLen);   // <= kT (host)
    const uint32_t cnt = (tid < nseg) ? p.seg_ws[((int64_t)row * p.n_seg + tid) * kSegWords] : 0u;
    uint32_t tot;
    const uint32_t incl = block_prefix_sum<kT>(cnt, sh, tot);
    if (tid < nseg) sh.hist[tid] = incl - cnt;
    __syncthreads();
    for (uint32_t pos = tid; pos < tot && pos < (uint32_t)kCandCap; pos += kThreads) {
      int lo = 0, hi = nseg - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sh.hist[mid] <= pos) lo = mid;
        else hi = mid - 1;
      }
      const uint32_t* src = p.seg_ws + ((int64_t)row * p.n_seg + lo) * kSegWords;
      const uint32_t i = pos - sh.hist[lo];
      sh.u.cand.key[pos] = src[4 + i];
      sh.u.cand.idx[pos] = (int32_t)src[4 + kCandCap + i];
    }
    __syncthreads();
  } else if (n_cand <= (uint32_t)kCandCap) {
    // ---- ordered compaction of every key in bins >= b1: two runs of kPer
    //      scores per thread (a and b, one chunk apart) share one block-wide
    //      scan, their counts packed in one word (a chunk holds at most 8192)
    const BinTest in_bins(b1);
    uint32_t base = 0;
    for (int64_t c0 = 0; c0 < n; c0 += 2 * chunk) {
      const int64_t ea = c0 + (int64_t)tid * kPer, eb = ea + chunk;
      const int la = (int)(n - ea < 0 ? 0 : (n - ea > kPer ? kPer : n - ea));
      const int lb = (int)(n - eb < 0 ? 0 : (n - eb > kPer ? kPer : n - eb));
      float va[kPer], vb[kPer];
      load_run(srow, ea, n, vec, va);
      load_run(srow, eb, n, vec, vb);
      uint32_t ma = 0u, mb = 0u;
      if (la == kPer && lb == kPer) {   // every chunk but the row's last
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          ma |= (uint32_t)in_bins(va[i]) << i;
          mb |= (uint32_t)in_bins(vb[i]) << i;
        }
      } else {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          ma |= (uint32_t)(i < la && in_bins(va[i])) << i;
          mb |= (uint32_t)(i < lb && in_bins(vb[i])) << i;
        }
      }
      const uint32_t ca = (uint32_t)__popc(ma), cb = (uint32_t)__popc(mb);
      uint32_t tot;
      const uint32_t incl = block_prefix_sum<kT>(ca | (cb << 16), sh, tot);
      uint32_t pa = base + (incl & 0xFFFFu) - ca;
      uint32_t pb = base + (tot & 0xFFFFu) + (incl >> 16) - cb;
      base += (tot & 0xFFFFu) + (tot >> 16);
      if ((ma | mb) == 0u) continue;    // most runs hold no candidate
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        if ((ma >> i) & 1u) {
          if (pa < (uint32_t)kCandCap) {
            sh.u.cand.key[pa] = score_key(va[i]);
            sh.u.cand.idx[pa] = (int32_t)(ea + i);
          }
          ++pa;
        }
        if ((mb >> i) & 1u) {
          if (pb < (uint32_t)kCandCap) {
            sh.u.cand.key[pb] = score_key(vb[i]);
            sh.u.cand.idx[pb] = (int32_t)(eb + i);
          }
          ++pb;
        }
      }
    }
  }
  if (n_cand <= (uint32_t)kCandCap) {
    // ---- digit 2 (bits [20:10]) and digit 3 (bits [9:0]) on the candidates
    clear<kT>(sh.hist, kBins);
    for (uint32_t i = tid; i < n_cand; i += kThreads) {
      const uint32_t key = sh.u.cand.key[i];
      if ((key >> 21) == b1) atomicAdd(sh.hist + ((key >> 10) & 0x7FFu), 1u);
    }
    __syncthreads();
    select_bin<kT>(sh, kBins, (uint32_t)k - above);
    const uint32_t p2 = (b1 << 11) | sh.sel_bin;
    above += sh.sel_above;
    __syncthreads();
    clear<kT>(sh.hist, 1024);
    for (uint32_t i = tid; i < n_cand; i += kThreads) {
      const uint32_t key = sh.u.cand.key[i];
      if ((key >> 10) == p2) atomicAdd(sh.hist + (key & 0x3FFu), 1u);
    }
    __syncthreads();
    select_bin<kT>(sh, 1024, (uint32_t)k - above);
    T = (p2 << 10) | sh.sel_bin;
    above += sh.sel_above;
    __syncthreads();
    // ---- emission from the candidates (already in index order)
    const uint32_t need_eq = (uint32_t)k - above;
    const uint32_t per = (n_cand + kThreads - 1) / kThreads;  // <= 8192 / kT
    const uint32_t i0 = tid * per;
    uint32_t gt = 0, eq = 0;
    for (uint32_t i = i0; i < i0 + per && i < n_cand; ++i) {
      gt += sh.u.cand.key[i] > T;
      eq += sh.u.cand.key[i] == T;
    }
    uint32_t tot;
    const uint32_t packed = gt | (eq << 16);
    const uint32_t before = block_prefix_sum<kT>(packed, sh, tot) - packed;
    uint32_t g_before = before & 0xFFFFu, q_before = before >> 16;
    for (uint32_t i = i0; i < i0 + per && i < n_cand; ++i) {
      const uint32_t key = sh.u.cand.key[i];
      const bool is_gt = key > T, is_eq = key == T;
      if (is_gt || (is_eq && q_before < need_eq)) {
        const uint32_t pos = g_before + (q_before < need_eq ? q_before : need_eq);
        if (CSA2_IN_BOUNDS(pos >= 0 && pos < k, p.err)) {
          orow[pos] = sh.u.cand.idx[i];
          if (osc) osc[pos] = key_score(key);
        }
      }
      g_before += is_gt;
      q_before += is_eq;
    }
    return;
  }

  // ---- crowded bin: digits 2 and 3 re-read the row
  uint32_t prefix = b1;
  clear<kT>(sh.hist, kBins);
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    const int64_t e = c0 + (int64_t)tid * kPer;
    float v[kPer];
    load_run(srow, e, n, vec, v);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const uint32_t key = score_key(v[i]);
      hist_add_aggregated(sh.hist, (e + i < n) && (key >> 21) == prefix, (key >> 10) & 0x7FFu);
    }
  }
  __syncthreads();
  select_bin<kT>(sh, kBins, (uint32_t)k - above);
  prefix = (prefix << 11) | sh.sel_bin;
  above += sh.sel_above;
  __syncthreads();
  clear<kT>(sh.hist, kBins);
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    const int64_t e = c0 + (int64_t)tid * kPer;
    float v[kPer];
    load_run(srow, e, n, vec, v);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const uint32_t key = score_key(v[i]);
      hist_add_aggregated(sh.hist, (e + i < n) && (key >> 10) == prefix, key & 0x3FFu);
    }
  }
  __syncthreads();
  select_bin<kT>(sh, 1024, (uint32_t)k - above);
  T = (prefix << 10) | sh.sel_bin;
  above += sh.sel_above;
  __syncthreads();

  // ---- ordered emission over the row: keys > T, then the first keys == T
  const uint32_t need_eq = (uint32_t)k - above;
  uint32_t base_gt = 0, base_eq = 0;
  for (int64_t c0 = 0; c0 < n; c0 += chunk) {
    const int64_t e = c0 + (int64_t)tid * kPer;
    float v[kPer];
    load_run(srow, e, n, vec, v);
    uint32_t gt = 0, eq = 0;
    uint32_t key[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      key[i] = score_key(v[i]);
      const bool ok = e + i < n;
      gt += (ok && key[i] > T);
      eq += (ok && key[i] == T);
    }
    uint32_t tot;
    const uint32_t packed = gt | (eq << 16);
    const uint32_t before = block_prefix_sum<kT>(packed, sh, tot) - packed;
    uint32_t g_before = base_gt + (before & 0xFFFFu);
    uint32_t q_before = base_eq + (before >> 16);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (e + i >= n) break;
      const bool is_gt = key[i] > T, is_eq = key[i] == T;
      if (is_gt || (is_eq && q_before < need_eq)) {
        const uint32_t pos = g_before + (q_before < need_eq ? q_before : need_eq);
        if (CSA2_IN_BOUNDS(pos >= 0 && pos < k && e + i < n, p.err)) {
          orow[pos] = (int32_t)(e + i);
          if (osc) osc[pos] = key_score(key[i]);
        }
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

int topk_segments(int64_t max_valid) {
  return (int)((max_valid + kTopkSegLen - 1) / kTopkSegLen);
}

size_t topk_seg_bytes(int32_t rows, int64_t max_valid) {
  return (size_t)rows * (size_t)topk_segments(max_valid) * kSegWords * sizeof(uint32_t);
}

cudaError_t launch_topk(const TopkParams& p, cudaStream_t s) {
  // many rows: two 512-thread rows per SM; few (long) rows, or more than 512
  // segments a row (one per thread when the row reads them back): one row of
  // 1024 threads per SM
  const bool seg = p.seg_ws && p.key_hist && p.n_seg > 0;
  const bool many = p.rows >= kTopkManyRows && !(seg && p.n_seg > 512);
  const int smem = many ? (int)sizeof(Shared<512>) : (int)sizeof(Shared<1024>);
  cudaError_t e = many ? cudaFuncSetAttribute(k_topk<512>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                       : cudaFuncSetAttribute(k_topk<1024>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (int r0 = 0; r0 < p.rows; r0 += kTopkMaxRowsPerLaunch) {
    const int nr = (p.rows - r0 < kTopkMaxRowsPerLaunch) ? p.rows - r0 : kTopkMaxRowsPerLaunch;
    if (seg) {
      cfg.gridDim = dim3((unsigned)p.n_seg, (unsigned)nr);
      cfg.blockDim = dim3(kSegThreads);
      cfg.dynamicSmemBytes = 0;
      e = cudaLaunchKernelEx(&cfg, k_topk_seg, p, r0);
      if (e != cudaSuccess) return e;
    }
    cfg.gridDim = dim3((unsigned)nr);
    cfg.blockDim = dim3(many ? 512 : 1024);
    cfg.dynamicSmemBytes = (size_t)smem;
    e = many ? cudaLaunchKernelEx(&cfg, k_topk<512>, p, r0)
             : cudaLaunchKernelEx(&cfg, k_topk<1024>, p, r0);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa2
