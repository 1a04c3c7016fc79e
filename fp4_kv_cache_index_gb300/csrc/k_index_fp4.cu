// k_index_fp4.cu -- CSA2 indexer scores over MXFP4 indexer keys and queries.
//
// The V4.1 report (section 2.4.4) keeps the indexer's queries and keys in
// OCP MXFP4: E2M1 codes with one power-of-two (UE8M0) scale per 32
// channels, 64 + 4 bytes per 128-channel key (the 68 B of the cache-size
// breakdown).  The score is the one of the bf16 indexer,
//     I[q, s] = sum_h w[q, h] * ReLU(q^[q, h] . K^[s]),
// over the dequantised values q^, K^.  An E2M1 value times a scale 2^e is
// exactly an E5M2 value for e in [-13, 13], so both operands become E5M2
// bytes (a byte permute per four codes through a per-block table) and the
// tensor cores take them as kind::f8f6f4 with fp32 accumulation: the same
// products as the dequantised values, one byte per channel in shared
// memory.  A block scale outside that range (values below 2^-14 or above
// 2^16) is clamped into it and reported in the device error word.
//
// Warp roles (576 threads):
//   warp 0      bulk-copies the raw tiles (128 keys: 8 KB of codes and their
//               scale words) into a ring 12 deep in decode (4 in prefill,
//               whose 8-query tiles need the room), and the query tile (TMA);
//   warps 10-17 convert each raw tile into a 128B-swizzled E5M2 K-major
//               stage, and at every new query group take the query tile
//               (bf16) to the MXFP4 grid and on to E5M2;
//   warp 1      issues the tcgen05 MMAs (M = 128 keys, N = 32 heads x qpg,
//               K = 128 as 4 x 32) from the converted stage and queries;
//   warps 2-9   the epilogue of the bf16 indexer (ReLU, head weights, fp32
//               or bf16 score store, score-key histogram).
// Every wait is bounded.
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

// A tile is 256 keys in decode (two M = 128 MMA groups: the per-tile cost of
// the warp hand-offs, a fixed ~0.3 us, is then spread over twice the keys)
// and 128 keys in prefill (8 queries per tile already give N = 256).
constexpr int kTileMax = 256;
constexpr int kRawStagesMax = 5;
constexpr int kStagesMax = 3;                           // converted E5M2 stages
constexpr int kKStageBytes = kTileMax * kIdxDim;        // 32 KB
constexpr int kRawCodeBytes = kTileMax * kIdxDim / 2;   // 16 KB
constexpr int kRawScaleBytes = 1056;                    // (256 + 4) words, 16-byte padded
constexpr int kRawStageBytes = kRawCodeBytes + kRawScaleBytes;
constexpr int kThreads = 576;
constexpr int kEpiThreads = 256;   // warps 2-9
constexpr int kCvtThreads = 256;   // warps 10-17
constexpr int kCvtBase = 320;
constexpr int kCvtWarps = kCvtThreads / 32;
constexpr int kEpiWarps = kEpiThreads / 32;

__host__ __device__ inline int raw_stages(int qpg) { return qpg == 1 ? kRawStagesMax : 2; }
__host__ __device__ inline int k_stages(int qpg) { return qpg == 1 ? kStagesMax : 2; }
__host__ __device__ inline int tile_rows_of(int qpg) { return qpg == 1 ? 256 : 128; }

struct SmemLayout {
  int raw_off, q_off, q8_off, w_off, hist_off, bar_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(int qpg) {
  SmemLayout L;
  L.raw_off = k_stages(qpg) * kKStageBytes;
  L.q_off = L.raw_off + raw_stages(qpg) * kRawStageBytes;
  L.q_off = (L.q_off + 1023) & ~1023;
  L.q8_off = L.q_off + qpg * 32 * kIdxDim * 2;          // E5M2 queries (1024-aligned)
  L.w_off = L.q8_off + qpg * 32 * kIdxDim;
  L.hist_off = L.w_off + qpg * 32 * 4;
  L.bar_off = L.hist_off + kKeyHistBins * 4;
  L.total = L.bar_off + 48 * 8 + 16 + 1024;  // barriers, tmem slot, alignment slack
  return L;
}

__device__ __forceinline__ int group_nvis_query(const IndexParams& p, int g, int j) {
  if (!p.prefill) return p.nvis[g];
  const int64_t q = (int64_t)g * p.qpg + j;
  const int64_t v = (p.pos0 + q + 1) / p.ratio;
  return (int)(v < p.pre_len ? v : p.pre_len);
}

__device__ __forceinline__ int64_t group_base(const IndexParams& p, int g) {
  return p.prefill ? p.pre_base : p.entry_base[g];
}

// First key row of item `it` in group g, the keys it copies (the cache ends
// at p.idx_total rows) and the first row of its 16-byte aligned scale window.
struct TileRows {
  int64_t row0, s0;
  int32_t nrows;
};
__device__ __forceinline__ TileRows tile_rows(const IndexParams& p, int g, int t, int tile_e) {
  TileRows r;
  r.row0 = group_base(p, g) + (int64_t)t * tile_e;
  const int64_t left = p.idx_total - r.row0;
  r.nrows = (int32_t)(left < tile_e ? left : tile_e);
  r.s0 = r.row0 & ~(int64_t)3;
  return r;
}

// E5M2 exponent offset of a UE8M0 byte, clamped to [-13, 13] (flagged).
__device__ __forceinline__ int block_exp(uint32_t ue8m0, bool nonzero, uint32_t* err) {
  int e = (int)ue8m0 - 127;
  if (nonzero && (e < -13 || e > 13)) {
    set_error(err, kErrRange);
    e = e < -13 ? -13 : 13;
  }
  return e;
}

// Block b (32 channels) of query row r: bf16 in the 128B-swizzled two-half
// tile -> MXFP4 (UE8M0 scale of the block's largest magnitude, OCP MX;
// E2M1 code of x / scale, nearest, ties to even, saturating) -> E5M2 bytes
// in the 128B-swizzled one-row-per-128-bytes tile q8.
__device__ __forceinline__ void query_block_to_e5m2(const uint8_t* qbuf, uint8_t* q8, int qrows,
                                                    int r, int b, uint32_t* err) {
  const uint8_t* half = qbuf + (b >> 1) * (qrows * 128) + r * 128;
  float x[32];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = (b & 1) * 4 + k;
    const uint4 w = *reinterpret_cast<const uint4*>(half + ((chunk ^ (r & 7)) << 4));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[8 * k + 2 * i] = __uint_as_float(u[i] << 16);
      x[8 * k + 2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t sb = ue8m0_for_amax(amax);
  const float sc = ue8m0_value(sb);
  uint32_t codes[4];
  uint32_t any = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) c |= e2m1_encode(__fdiv_rn(x[8 * k + i], sc)) << (4 * i);
    codes[k] = c;
    any |= c & 0x77777777u;
  }
  uint32_t tlo, thi;
  e5m2_table(block_exp(sb, any != 0, err), tlo, thi);
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) e2m1x8_to_e5m2x8(codes[k], tlo, thi, o[2 * k], o[2 * k + 1]);
  uint8_t* row = q8 + r * 128;
  *reinterpret_cast<uint4*>(row + (((2 * b) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4*>(row + (((2 * b + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_index_fp4(const __grid_constant__ IndexParams p, const __grid_constant__ CUtensorMap tm_q) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const SmemLayout L = smem_layout(p.qpg);
  uint8_t* kbuf = smem;
  uint8_t* raw = smem + L.raw_off;
  uint8_t* qbuf = smem + L.q_off;
  uint8_t* q8 = smem + L.q8_off;
  float* wbuf = reinterpret_cast<float*>(smem + L.w_off);
  uint32_t* hs = reinterpret_cast<uint32_t*>(smem + L.hist_off);  // score-key histogram
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* raw_full = bars;            // [kRawStagesMax]
  uint64_t* raw_empty = bars + 12;      // [kRawStagesMax]
  uint64_t* k_full = bars + 24;         // [kStagesMax]
  uint64_t* k_empty = bars + 28;        // [kStagesMax]
  uint64_t* acc_full = bars + 32;       // [nacc <= 4]
  uint64_t* acc_empty = bars + 36;      // [nacc <= 4]
  uint64_t* q_full = bars + 40;
  uint64_t* q_ready = bars + 41;
  uint64_t* q_empty = bars + 42;
  uint64_t* drain = bars + 43;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 44);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = 32 * p.qpg;               // MMA N (columns per accumulator)
  const int qrows = 32 * p.qpg;
  // decode (one query per group): 256-key tiles as two M-groups whose
  // accumulators sit side by side (2 x 32 columns), 4 accumulators, each
  // epilogue half takes one M-group; prefill: 128-key tiles, 2 accumulators
  // of 256 columns, the halves split the 8 queries of every tile
  const bool two_groups = p.qpg == 1;
  const int tile_e = tile_rows_of(p.qpg);
  const int mgroups = tile_e / 128;
  const int nacc = two_groups ? 4 : 2;
  const int acc_cols = mgroups * N;
  const uint32_t tmem_cols = (uint32_t)(nacc * acc_cols) < 32u ? 32u : (uint32_t)(nacc * acc_cols);
  const int n_raw = raw_stages(p.qpg);
  const int n_k = k_stages(p.qpg);

  if (threadIdx.x == 0) {
    for (int i = 0; i < n_raw; ++i) {
      mbar_init(raw_full + i, 1);
      mbar_init(raw_empty + i, kCvtWarps);
    }
    // consumer barriers count warps: each warp arrives once, from lane 0,
    // after a __syncwarp over its lanes' work
    for (int i = 0; i < n_k; ++i) { mbar_init(k_full + i, kCvtWarps); mbar_init(k_empty + i, 1); }
    for (int i = 0; i < nacc; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, kEpiWarps);
    }
    mbar_init(q_full, 1);
    mbar_init(q_ready, kCvtWarps);
    mbar_init(q_empty, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, tmem_cols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();

  const int total = p.tile_prefix[p.n_groups];
  const int begin = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
  const int end = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);
  int g0 = 0;
  while (g0 < p.n_groups && p.tile_prefix[g0 + 1] <= begin) ++g0;

  if (warp == 0 && lane == 0 && begin < end) {
    // ------------------------------------------------ bulk-copy producer
    int g = g0, cur = -1, rs = 0;
    uint32_t rph = 0, qph = 0;
    uint32_t armed = 0, armed_ph = 0;   // raw stages filled at least once, parity of the last fill
    bool ok = true;
    const uint64_t keys_pol = l2_policy_evict_first();
    for (int it = begin; it < end && ok; ++it) {
      while (p.tile_prefix[g + 1] <= it) ++g;
      if (g != cur) {
        ok = mbar_wait(q_empty, qph ^ 1, p.err);
        qph ^= 1;
        if (!ok) break;
        mbar_arrive_expect_tx(q_full, (uint32_t)(qrows * kIdxDim * 2));
        tma_load_2d(qbuf, &tm_q, 0, g * qrows, q_full);
        tma_load_2d(qbuf + qrows * 128, &tm_q, 64, g * qrows, q_full);
        cur = g;
      }
      ok = mbar_wait(raw_empty + rs, rph ^ 1, p.err);
      if (!ok) break;
      const TileRows tr = tile_rows(p, g, it - p.tile_prefix[g], tile_e);
      const int64_t s1 = (tr.row0 + tr.nrows + 3) & ~(int64_t)3;
      const uint32_t code_bytes = (uint32_t)tr.nrows * (kIdxDim / 2);
      const uint32_t scale_bytes = (uint32_t)(s1 - tr.s0) * 4u;
      uint8_t* dst = raw + rs * kRawStageBytes;
      mbar_arrive_expect_tx(raw_full + rs, code_bytes + scale_bytes);
      bulk_load(dst, p.idx_codes + tr.row0 * (kIdxDim / 2), code_bytes, raw_full + rs, keys_pol);
      bulk_load(dst + kRawCodeBytes, p.idx_scales + tr.s0 * 4, scale_bytes, raw_full + rs,
                keys_pol);
      armed |= 1u << rs;
      armed_ph = (armed_ph & ~(1u << rs)) | (rph << rs);
      if (++rs == n_raw) { rs = 0; rph ^= 1; }
    }
    // make sure no bulk copy is still writing into this CTA's shared memory
    for (int s = 0; s < n_raw; ++s)
      if (armed & (1u << s)) mbar_wait(raw_full + s, (armed_ph >> s) & 1u, p.err);
    if (cur >= 0) mbar_wait(q_full, qph ^ 1, p.err);
  } else if (warp >= 10 && begin < end) {
    // ------------------------------------------------ converters
    const int ct = threadIdx.x - kCvtBase;          // 0..255
    const int cw = ct >> 5;                         // converter warp 0..7
    const int b = ct & 3;                           // 32-channel block of the key
    int g = g0, cur = -1, rs = 0, ks = 0;
    uint32_t rph = 0, kph = 0, qph = 0;
    bool ok = true;
    for (int it = begin; it < end && ok; ++it) {
      while (p.tile_prefix[g + 1] <= it) ++g;
      if (g != cur) {
        // a new query tile: onto the MXFP4 grid before its first MMA
        ok = mbar_wait(q_full, qph, p.err);
        qph ^= 1;
        if (!ok) break;
        for (int i = ct; i < qrows * 4; i += kCvtThreads)
          query_block_to_e5m2(qbuf, q8, qrows, i >> 2, i & 3, p.err);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
        cur = g;
      }
      ok = mbar_wait(raw_full + rs, rph, p.err) && mbar_wait(k_empty + ks, kph ^ 1, p.err);
      if (!ok) break;
      const int t = it - p.tile_prefix[g];
      const TileRows tr = tile_rows(p, g, t, tile_e);
      // rows holding appended keys (the rest of the copy is unused capacity
      // or the next sequence: converted as zeros, never range-checked)
      const int32_t len = p.prefill ? p.pre_len : p.nvis[g];
      const int32_t live = min(tr.nrows, len - t * tile_e);
      const uint8_t* src = raw + rs * kRawStageBytes;
      const uint32_t* sw = reinterpret_cast<const uint32_t*>(src + kRawCodeBytes) + (tr.row0 - tr.s0);
      uint8_t* dst = kbuf + ks * kKStageBytes;
#pragma unroll 1
      for (int pass = 0; pass < tile_e / 64; ++pass) {
        const int r = pass * 64 + cw * 8 + (lane >> 2);   // key row of the tile
        uint4 c4 = make_uint4(0u, 0u, 0u, 0u);
        uint32_t sb = 127u;
        if (r < live) {
          c4 = *reinterpret_cast<const uint4*>(src + r * (kIdxDim / 2) + b * 16);
          sb = (sw[r] >> (8 * b)) & 0xFFu;
        }
        const uint32_t any = (c4.x | c4.y | c4.z | c4.w) & 0x77777777u;
        uint32_t tlo, thi;
        e5m2_table(block_exp(sb, any != 0, p.err), tlo, thi);
        uint32_t o[8];
        e2m1x8_to_e5m2x8(c4.x, tlo, thi, o[0], o[1]);
        e2m1x8_to_e5m2x8(c4.y, tlo, thi, o[2], o[3]);
        e2m1x8_to_e5m2x8(c4.z, tlo, thi, o[4], o[5]);
        e2m1x8_to_e5m2x8(c4.w, tlo, thi, o[6], o[7]);
        uint8_t* rowp = dst + r * 128;
        *reinterpret_cast<uint4*>(rowp + (((2 * b) ^ (r & 7)) << 4)) =
            make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(rowp + (((2 * b + 1) ^ (r & 7)) << 4)) =
            make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(k_full + ks);
        mbar_arrive(raw_empty + rs);
      }
      if (++rs == n_raw) { rs = 0; rph ^= 1; }
      if (++ks == n_k) { ks = 0; kph ^= 1; }
    }
  } else if (warp == 1 && lane == 0 && begin < end) {
    // ------------------------------------------------ MMA issuer
    // the f16-kind descriptor: format fields 1 / 1 read as E5M2 / E5M2 here
    const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)N, false, false);
    int g = g0, cur = -1, stage = 0, acc = 0;
    uint32_t ph = 0, qph = 0, aph = 0;
    bool ok = true;
    for (int it = begin; it < end && ok; ++it) {
      while (p.tile_prefix[g + 1] <= it) ++g;
      if (g != cur) {
        ok = mbar_wait(q_ready, qph, p.err);
        qph ^= 1;
        if (!ok) break;
        cur = g;
      }
      ok = mbar_wait(k_full + stage, ph, p.err) && mbar_wait(acc_empty + acc, aph ^ 1, p.err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t b0 = smem_u32(q8);
      // one 128-byte swizzled row holds all 128 channels: K steps of 32 bytes
      for (int mg = 0; mg < mgroups; ++mg) {
        const uint32_t a0 = smem_u32(kbuf + stage * kKStageBytes + mg * 128 * 128);
        const uint32_t d = tmem_base + (uint32_t)(acc * acc_cols + mg * N);
#pragma unroll
        for (int ks = 0; ks < kIdxDim / 32; ++ks)
          umma_e5m2(d, sdesc_sw128(a0 + ks * 32, 16, 1024), sdesc_sw128(b0 + ks * 32, 16, 1024),
                    idesc, ks > 0 ? 1u : 0u);
      }
      umma_commit(k_empty + stage);
      umma_commit(acc_full + acc);
      const bool last_of_group = (it + 1 == end) || (p.tile_prefix[g + 1] <= it + 1);
      if (last_of_group) umma_commit(q_empty);
      if (++stage == n_k) { stage = 0; ph ^= 1; }
      if (++acc == nacc) { acc = 0; aph ^= 1; }
    }
    umma_commit(drain);
    mbar_wait(drain, 0, p.err);
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------ epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int et = threadIdx.x - 64;           // 0..255
    const int half = (warp - 2) >> 2;          // M-group (decode) or queries (prefill)
    const int row = (two_groups ? half * 128 : 0) + quad * 32 + lane;   // key within the tile
    const int jq = (p.qpg + 1) >> 1;
    const int j0 = half * jq, j1 = min(p.qpg, j0 + jq);
    const bool use_hist = p.key_hist != nullptr && p.qpg == 1;
    auto flush = [&](int qq) {
      asm volatile("bar.sync 1, 256;" ::: "memory");
      for (int i = et; i < kKeyHistBins; i += kEpiThreads) {
        const uint32_t v = hs[i];
        if (v) atomicAdd(p.key_hist + (int64_t)qq * kKeyHistBins + i, v);
        hs[i] = 0u;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
    };
    if (use_hist) {
      for (int i = et; i < kKeyHistBins; i += kEpiThreads) hs[i] = 0u;
    }
    int g = g0, cur = -1;
    bool ok = true;
    for (int it = begin; it < end; ++it) {
      while (p.tile_prefix[g + 1] <= it) ++g;
      if (g != cur) {
        if (use_hist && cur >= 0) flush(cur);
        asm volatile("bar.sync 1, 256;" ::: "memory");
        for (int i = et; i < qrows; i += kEpiThreads) {
          const int q = g * p.qpg + (i >> 5);
          wbuf[i] = (q < p.nq) ? __ldg(p.w + (int64_t)q * kIdxHeads + (i & 31)) : 0.0f;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        cur = g;
      }
      const int u = it - begin;
      if (!ok) continue;
      const int acc = u % nacc;
      if (!mbar_wait(acc_full + acc, (uint32_t)((u / nacc) & 1), p.err)) { ok = false; continue; }
      tc_fence_after();
      const int t = it - p.tile_prefix[g];
      const int e = t * tile_e + row;
      const int ja = two_groups ? 0 : j0, jb = two_groups ? 1 : j1;
      const uint32_t col0 = (uint32_t)(acc * acc_cols + (two_groups ? half * N : 0));
      for (int j = ja; j < jb; ++j) {
        uint32_t r[32];
        tmem_ld32(tmem_base + ((uint32_t)(quad * 32) << 16) + col0 + (uint32_t)(j * 32), r);
        const float* wj = wbuf + j * 32;
        float s = 0.0f;
#pragma unroll
        for (int h = 0; h < 32; ++h) s = fmaf(wj[h], fmaxf(__uint_as_float(r[h]), 0.0f), s);
        const int q = g * p.qpg + j;
        if (q < p.nq && e < group_nvis_query(p, g, j)) {
          if (p.score_bf16) {
            const uint32_t bb = float_to_bf16_bits(s);
            reinterpret_cast<uint16_t*>(p.scores)[(int64_t)q * p.ld + e] = (uint16_t)bb;
            if (use_hist) atomicAdd(hs + (score_key(bf16_bits_to_float(bb)) >> 21), 1u);
          } else {
            p.scores[(int64_t)q * p.ld + e] = s;
            if (use_hist) atomicAdd(hs + (score_key(s) >> 21), 1u);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + acc);
    }
    if (use_hist && cur >= 0) flush(cur);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace

int index_fp4_smem_bytes(int qpg) { return smem_layout(qpg).total; }

cudaError_t launch_index_fp4(const IndexParams& p, const CUtensorMap& tm_q, int grid,
                             cudaStream_t s) {
  const int smem = index_fp4_smem_bytes(p.qpg);
  cudaError_t e = cudaFuncSetAttribute(k_index_fp4, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_index_fp4, p, tm_q);
}

}  // namespace csa2
