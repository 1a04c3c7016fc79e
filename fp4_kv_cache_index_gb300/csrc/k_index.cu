// k_index.cu -- CSA2 indexer scores on the 5th-generation tensor cores.
//
// Score (blog reading of the DeepSeek-V4 report, section 4.1, "lightning
// indexer"; V4.1 report section 2.3 keeps the same indexer):
//     I[q, s] = sum_h w[q, h] * ReLU(q_idx[q, h] . K_I[s])
// with 32 heads of dim 128 (V4.1 report, section 4.2.1).
//
// Mapping: one MMA is D[128 entries x 32*qpg] = K_I[128 x 128] *
// Q[32*qpg x 128]^T (M = 128 entries, N = heads of qpg queries, K = 128), bf16
// operands from 128B-swizzled shared memory, fp32 accumulators in TMEM.  The
// ReLU and the head-weighted sum run in the epilogue on the accumulator rows.
// Decode uses qpg = 1 (each query reads its own sequence) with tiles of two
// such M-groups (256 keys: half the per-tile waits and commits of the MMA
// issuer per key); prefill groups 8 consecutive queries of one sequence so
// that a 128-key K_I tile feeds 256 columns.
//
// Pool mode (Reindex layers of the Hierarchical Sparse Indexer, V4.1 report
// section 2.3.2): a tile is 32 blocks of 8 consecutive keys named by the
// query's candidate pool (two M-groups of 16 blocks; a pool of an odd number
// of 16-block halves ends with a half tile), one 3-D TMA box per block (2 KB:
// its two 1 KB swizzled column halves), so the MMA walks 8-row atoms 2 KB
// apart; pool slots past the sequence score -inf.  Block ids of the next
// tile are loaded one tile ahead by the producer and by the epilogue.
//
// Scores are stored as fp32, or (selector precision of the V4 blog reading,
// section 7) rounded to bf16 with the histogram taken on the rounded value.
//
// Persistent CTAs walk a balanced contiguous range of (group, tile) items.
// Warp roles: warp 0 = TMA producer (lane 0; every lane in pool mode), warp 1
// = MMA issuer (and TMEM owner), then the epilogue warps (TMEM -> registers
// -> scores): eight with one query per group (two sets of four taking
// alternate tiles), sixteen with several (four warps per TMEM lane quadrant,
// each taking a quarter of the group's queries, so that the ReLU and head sums
// of a tile's 256 columns run on every scheduler with enough warps to cover
// the TMEM load latency).  Every wait is bounded.
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

constexpr int kTileE = 128;                          // keys of one M-group
constexpr int kMGroupBytes = kTileE * kIdxDim * 2;   // 32 KB
constexpr int kMaxStages = 4;
constexpr int kMaxQpg = 8;                 // queries per group (N <= 256)
constexpr int kMaxAcc = 4;                 // accumulators in TMEM (decode 4, several queries 2)
constexpr int kBars = 2 * kMaxStages + 2 * kMaxAcc + 4;   // k full / empty, acc full / empty, q full / empty, drain

// One query per group: stages of two M-groups (decode tiles are 256
// contiguous keys, pool tiles 32 blocks of 8); several
// queries: stages of one M-group (128-key tiles).  Three stages either way
// (with several queries the score-key histograms of the group's queries
// take the room of a fourth).
__host__ __device__ constexpr int stages_of(int) { return 3; }
__host__ __device__ constexpr int stage_bytes_of(int qpg) {
  return qpg == 1 ? 2 * kMGroupBytes : kMGroupBytes;
}

struct SmemLayout {
  int q_off, w_off, hist_off, bar_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(int qpg) {
  SmemLayout L;
  L.q_off = stages_of(qpg) * stage_bytes_of(qpg);
  L.w_off = L.q_off + qpg * 32 * kIdxDim * 2;
  L.hist_off = L.w_off + (qpg > 2 ? qpg : 2) * 32 * 4;
  // one histogram per epilogue set (one query per group) or per query
  L.bar_off = L.hist_off + (qpg == 1 ? 2 : qpg) * kKeyHistBins * 4;
  L.total = L.bar_off + kBars * 8 + 16 + 1024;  // barriers, tmem slot, alignment slack
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

// Position in the tile list: group g holds tiles [lo, hi).  The parameter
// tables are read only when the group changes: a dynamic index into the
// kernel parameters goes through the constant cache, and reading a large
// table there on every tile kept missing it (several hundred cycles a tile).
struct GroupCursor {
  int g, lo, hi;
  __device__ __forceinline__ void init(const IndexParams& p, int g0) {
    g = g0;
    lo = p.tile_prefix[g0];
    hi = p.tile_prefix[g0 + 1];
  }
  // moves to the group of tile `it` (at or after the current one); true if
  // the group changed
  __device__ __forceinline__ bool advance(const IndexParams& p, int it) {
    if (it < hi) return false;
    do {
      ++g;
      lo = hi;
      hi = p.tile_prefix[g + 1];
    } while (hi <= it);
    return true;
  }
};

// kEpiW epilogue warps: 8 for one query per group, 16 for several.
template <int kEpiW>
__global__ void __launch_bounds__(64 + 32 * kEpiW, 1)
    k_index(const __grid_constant__ IndexParams p, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_q) {
  constexpr int kEpiThreads = 32 * kEpiW;
  constexpr int kParts = kEpiW / 4;                      // warps per TMEM lane quadrant
  constexpr int kMaxQ = (kMaxQpg + kParts - 1) / kParts;   // queries of one epilogue thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const SmemLayout L = smem_layout(p.qpg);
  uint8_t* kbuf = smem;
  uint8_t* qbuf = smem + L.q_off;
  float* wbuf = reinterpret_cast<float*>(smem + L.w_off);
  uint32_t* hs = reinterpret_cast<uint32_t*>(smem + L.hist_off);  // score-key histogram
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* k_full = bars;                    // [n_stages]
  uint64_t* k_empty = bars + kMaxStages;      // [n_stages]
  uint64_t* acc_full = bars + 2 * kMaxStages; // [kMaxAcc]
  uint64_t* acc_empty = acc_full + kMaxAcc;   // [kMaxAcc]
  uint64_t* q_full = acc_full + 2 * kMaxAcc;
  uint64_t* q_empty = q_full + 1;
  uint64_t* drain = q_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = 32 * p.qpg;               // MMA N (columns per M-group)
  const int qrows = 32 * p.qpg;
  const int n_stages = stages_of(p.qpg), stage_bytes = stage_bytes_of(p.qpg);
  // one query: two M-groups of 128 keys (contiguous, or 16 pool blocks
  // each); several queries: one
  const int mgroups = p.qpg == 1 ? 2 : 1;
  const int tile_e = kTileE * mgroups;
  const int acc_cols = mgroups * N;
  // one query (N = 32) keeps four accumulators in flight, several queries
  // per tile (N = 256) two
  const int nacc = p.qpg == 1 ? 4 : 2;
  const uint32_t tmem_cols = (acc_cols * nacc <= 32) ? 32u : (uint32_t)(acc_cols * nacc);

  if (threadIdx.x == 0) {
    for (int i = 0; i < n_stages; ++i) { mbar_init(k_full + i, 1); mbar_init(k_empty + i, 1); }
    // acc_empty: decode, every thread of the set of four warps that took the
    // tile; several queries, one arrival per epilogue warp
    for (int i = 0; i < nacc; ++i) { mbar_init(acc_full + i, 1); mbar_init(acc_empty + i, p.qpg == 1 ? 128 : kEpiW); }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, tmem_cols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();
  const long long wl = wait_limit(p.wait_cycles);   // bounded-wait limit (cycles)

  const int total = p.tile_prefix[p.n_groups];
  const int begin = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
  const int end = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);
  int g0 = 0;
  while (g0 < p.n_groups && p.tile_prefix[g0 + 1] <= begin) ++g0;
  // block b of pool tile `it` (whose group is at or after the cursor's), or
  // -1 past the pool's end
  auto pool_blk = [&](int it, GroupCursor c, int b) -> int32_t {
    c.advance(p, it);
    const int i = (it - c.lo) * (tile_e / 8) + b;
    return i < p.pool_blocks ? __ldg(p.pool + (int64_t)c.g * p.pool_blocks + i) : -1;
  };
  GroupCursor c0;
  c0.init(p, g0);

  if (warp == 0 && begin < end) {
    // ------------------------------------------------ TMA producer (warp 0)
    // Lane 0 owns the barriers; in pool mode every lane copies one block.
    GroupCursor gc = c0;
    int cur = -1, stage = 0;
    int64_t gbase = 0;
    uint32_t ph = 0, qph = 0;
    uint32_t armed = 0, armed_ph = 0;   // stages filled at least once, parity of the last fill
    bool ok = true;
    const bool pool_lane = p.pool != nullptr && lane < tile_e / 8;
    const uint64_t keys_pol = l2_policy_evict_first();
    int32_t nxt = pool_lane ? pool_blk(begin, c0, lane) : -1;
    for (int it = begin; it < end && ok; ++it) {
      gc.advance(p, it);
      const int g = gc.g;
      if (g != cur) {
        gbase = group_base(p, g);
        if (lane == 0) {
          ok = mbar_wait(q_empty, qph ^ 1, p.err, wl);
          if (ok) {
            mbar_arrive_expect_tx(q_full, (uint32_t)(qrows * kIdxDim * 2));
            tma_load_2d(qbuf, &tm_q, 0, g * qrows, q_full);
            tma_load_2d(qbuf + qrows * 128, &tm_q, 64, g * qrows, q_full);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        qph ^= 1;
        if (!ok) break;
        cur = g;
      }
      if (lane == 0) ok = mbar_wait(k_empty + stage, ph ^ 1, p.err, wl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (p.inject & kInjectNoKeyLoads) {   // tests: nothing arrives on k_full
        if (++stage == n_stages) { stage = 0; ph ^= 1; }
        continue;
      }
      uint8_t* dst = kbuf + stage * stage_bytes;
      if (p.pool) {
        const int32_t blk = nxt;
        if (pool_lane && it + 1 < end) nxt = pool_blk(it + 1, gc, lane);
        const uint32_t n_ok = (uint32_t)__popc(__ballot_sync(0xffffffffu, blk >= 0));
        if (lane == 0) mbar_arrive_expect_tx(k_full + stage, n_ok * 8 * kIdxDim * 2);
        __syncwarp();
        if (blk >= 0) {
          const int32_t row = (int32_t)(gbase + (int64_t)blk * 8);
          tma_load_3d(dst + lane * 2048, &tm_k, 0, row, 0, k_full + stage, keys_pol);
        }
      } else if (lane == 0) {
        // each M-group: its two 64-channel column halves
        const int64_t row = gbase + (int64_t)(it - gc.lo) * tile_e;
        mbar_arrive_expect_tx(k_full + stage, (uint32_t)(mgroups * kMGroupBytes));
        for (int mg = 0; mg < mgroups; ++mg) {
          uint8_t* d = dst + mg * kMGroupBytes;
          const int32_t r = (int32_t)(row + mg * kTileE);
          tma_load_2d(d, &tm_k, 0, r, k_full + stage, keys_pol);
          tma_load_2d(d + kMGroupBytes / 2, &tm_k, 64, r, k_full + stage, keys_pol);
        }
      }
      armed |= 1u << stage;
      armed_ph = (armed_ph & ~(1u << stage)) | (ph << stage);
      if (++stage == n_stages) { stage = 0; ph ^= 1; }
    }
    // make sure no bulk copy is still writing into this CTA's shared memory
    if (lane == 0) {
      for (int s = 0; s < n_stages; ++s)
        if (armed & (1u << s)) mbar_wait(k_full + s, (armed_ph >> s) & 1u, p.err, wl);
      if (cur >= 0) mbar_wait(q_full, qph ^ 1, p.err, wl);
    }
    __syncwarp();
  } else if (warp == 1 && lane == 0 && begin < end) {
    // ------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)N, false, false);
    // contiguous tiles: column halves 16 KB apart, 8-row atoms 1 KB apart;
    // pool tiles: halves 1 KB apart inside each block's 2 KB.  Descriptor
    // bases built once; the offsets go into the address field (shared
    // memory is below 2^18 bytes, so it never carries).
    const uint32_t a_half = p.pool ? 1024u : (uint32_t)(kMGroupBytes / 2);
    const uint64_t adesc0 = sdesc_sw128(smem_u32(kbuf), 16, p.pool ? 2048u : 1024u);
    const uint64_t bdesc0 = sdesc_sw128(smem_u32(qbuf), 16, 1024);
    GroupCursor gc = c0;
    int cur = -1, stage = 0, acc = 0;
    uint32_t ph = 0, qph = 0, aph = 0;
    bool ok = true;
    for (int it = begin; it < end && ok; ++it) {
      gc.advance(p, it);
      const int g = gc.g;
      if (g != cur) {
        ok = mbar_wait(q_full, qph, p.err, wl);
        qph ^= 1;
        if (!ok) break;
        cur = g;
      }
      ok = mbar_wait(k_full + stage, ph, p.err, wl) && mbar_wait(acc_empty + acc, aph ^ 1, p.err, wl);
      if (!ok) break;
      tc_fence_after();
      const uint64_t adesc = adesc0 + (uint64_t)((stage * stage_bytes) >> 4);
      for (int mg = 0; mg < mgroups; ++mg) {
        const uint32_t d = tmem_base + (uint32_t)(acc * acc_cols + mg * N);
#pragma unroll
        for (int ks = 0; ks < kIdxDim / 16; ++ks) {
          const uint32_t ao = (uint32_t)(mg * kMGroupBytes) + (uint32_t)(ks >> 2) * a_half +
                              (uint32_t)(ks & 3) * 32u;
          const uint32_t bo = (uint32_t)((ks >> 2) * (qrows * 128) + (ks & 3) * 32);
          umma_bf16(d, adesc + (ao >> 4), bdesc0 + (bo >> 4), idesc, ks > 0 ? 1u : 0u);
        }
      }
      umma_commit(k_empty + stage);
      umma_commit(acc_full + acc);
      const bool last_of_group = (it + 1 == end) || (gc.hi <= it + 1);
      if (last_of_group) umma_commit(q_empty);
      if (++stage == n_stages) { stage = 0; ph ^= 1; }
      if (++acc == nacc) { acc = 0; aph ^= 1; }
    }
    umma_commit(drain);
    mbar_wait(drain, 0, p.err, wl);
  } else if (kEpiW == 8 && warp >= 2 && p.qpg == 1) {
    // ------------------------------------------------ epilogue, one query per tile
    // Two groups of four warps take alternate tiles (group gsel the tiles
    // begin + gsel + 2k, whose accumulator is gsel), so two tiles' scores are
    // formed at once; each group keeps its own weights, histogram and named
    // barrier.  Thread: one entry of the tile (its TMEM lane), 32 heads.
    const int gsel = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int et = (threadIdx.x - 64) & 127;
    const uint32_t bar_id = 2u + (uint32_t)gsel;
    uint32_t* hsg = hs + gsel * kKeyHistBins;
    float* wg = wbuf + gsel * 32;
    const bool use_hist = p.key_hist != nullptr;
    auto gsync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory"); };
    auto flush = [&](int qq) {
      gsync();
      for (int i = et; i < kKeyHistBins; i += 128) {
        const uint32_t v = hsg[i];
        if (v) atomicAdd(p.key_hist + (int64_t)qq * kKeyHistBins + i, v);
        hsg[i] = 0u;
      }
      gsync();
    };
    if (use_hist)
      for (int i = et; i < kKeyHistBins; i += 128) hsg[i] = 0u;
    GroupCursor gc = c0;
    int cur = -1, nvis = 0;
    // pool mode: the blocks of this thread's slots (row and 128 + row) of
    // the next tile of its set
    int32_t blk_nxt[2] = {-1, -1};
    if (p.pool && begin + gsel < end) {
      blk_nxt[0] = pool_blk(begin + gsel, c0, row >> 3);
      blk_nxt[1] = pool_blk(begin + gsel, c0, 16 + (row >> 3));
    }
    for (int it = begin + gsel; it < end; it += 2) {
      gc.advance(p, it);
      const int g = gc.g;
      const int32_t blk[2] = {blk_nxt[0], blk_nxt[1]};
      if (p.pool && it + 2 < end) {
        blk_nxt[0] = pool_blk(it + 2, gc, row >> 3);
        blk_nxt[1] = pool_blk(it + 2, gc, 16 + (row >> 3));
      }
      if (g != cur) {
        if (use_hist && cur >= 0) flush(cur);
        gsync();
        if (et < 32) wg[et] = (g < p.nq) ? __ldg(p.w + (int64_t)g * kIdxHeads + et) : 0.0f;
        gsync();
        cur = g;
        nvis = group_nvis_query(p, g, 0);
      }
      const int jt = it - begin;
      const int a = jt & 3;
      // suspend-hinted wait: a polling epilogue warp would take issue slots
      // from the producer and MMA warps that share its scheduler
      if (!mbar_wait_sleep(acc_full + a, (uint32_t)((jt >> 2) & 1), p.err, wl)) break;
      tc_fence_after();
      const int t = it - gc.lo;
      const uint32_t ta = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(a * acc_cols);
      // entry row + 128 mg of the tile: score s
      auto store = [&](int mg, float s) {
        const int e = t * tile_e + mg * kTileE + row;
        if (p.pool) {
          // slots past the pool (the second half of a half tile) are not stored
          const int64_t ent = (int64_t)blk[mg] * 8 + (row & 7);
          const float v = (blk[mg] >= 0 && ent < nvis) ? s : -INFINITY;
          if (e < p.ld) {
            p.scores[(int64_t)g * p.ld + e] = v;
            if (use_hist) atomicAdd(hsg + (score_key(v) >> 21), 1u);
          }
        } else if (g < p.nq && e < nvis && CSA2_IN_BOUNDS(e < p.ld, p.err)) {
          if (p.score_bf16) {
            const uint32_t b = float_to_bf16_bits(s);
            reinterpret_cast<uint16_t*>(p.scores)[(int64_t)g * p.ld + e] = (uint16_t)b;
            if (use_hist) atomicAdd(hsg + (score_key(bf16_bits_to_float(b)) >> 21), 1u);
          } else {
            p.scores[(int64_t)g * p.ld + e] = s;
            if (use_hist) atomicAdd(hsg + (score_key(s) >> 21), 1u);
          }
        }
      };
      if (mgroups == 2) {
        // both M-groups of the tile: columns 0 and N of its accumulator
        uint32_t ra[32], rb[32];
        tmem_ld32x2(ta, ta + (uint32_t)N, ra, rb);
        tc_fence_before();
        mbar_arrive(acc_empty + a);   // the accumulator is free once read
        store(0, relu_dot32(wg, ra));
        store(1, relu_dot32(wg, rb));
      } else {
        uint32_t r[32];
        tmem_ld32(ta, r);
        tc_fence_before();
        mbar_arrive(acc_empty + a);
        store(0, relu_dot32(wg, r));
      }
    }
    if (use_hist && cur >= 0) flush(cur);
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;          // entry within the tile
    const int et = threadIdx.x - 64;           // 0 .. kEpiThreads - 1
    const int part = (warp - 2) >> 2;          // which queries of the group
    const int jq = (p.qpg + kParts - 1) / kParts;
    const int j0 = part * jq, j1 = min(p.qpg, j0 + jq);
    // score-key histograms: one per query of the group, hs[j][bin]
    const bool use_hist = p.key_hist != nullptr;
    const int hbins = p.qpg * kKeyHistBins;
    // adds this CTA's counts of group `gg`'s queries to the global
    // histograms and clears hs
    auto esync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); };
    auto flush = [&](int gg) {
      esync();
      for (int i = et; i < hbins; i += kEpiThreads) {
        const uint32_t v = hs[i];
        const int q = gg * p.qpg + i / kKeyHistBins;
        if (v && q < p.nq) atomicAdd(p.key_hist + (int64_t)q * kKeyHistBins + (i % kKeyHistBins), v);
        hs[i] = 0u;
      }
      esync();
    };
    if (use_hist) {
      for (int i = et; i < hbins; i += kEpiThreads) hs[i] = 0u;
    }
    GroupCursor gc = c0;
    int cur = -1, acc = 0;
    uint32_t aph = 0;
    int nvis[kMaxQ];   // visible entries of this thread's queries in the current group
    int32_t blk_nxt = (p.pool && begin < end) ? pool_blk(begin, c0, row >> 3) : -1;
    for (int it = begin; it < end; ++it) {
      gc.advance(p, it);
      const int g = gc.g;
      const int32_t blk = blk_nxt;
      if (p.pool && it + 1 < end) blk_nxt = pool_blk(it + 1, gc, row >> 3);
      if (g != cur) {
        if (use_hist && cur >= 0) flush(cur);
        esync();
        for (int i = et; i < qrows; i += kEpiThreads) {
          const int q = g * p.qpg + (i >> 5);
          wbuf[i] = (q < p.nq) ? __ldg(p.w + (int64_t)q * kIdxHeads + (i & 31)) : 0.0f;
        }
        esync();
        cur = g;
#pragma unroll
        for (int jj = 0; jj < kMaxQ; ++jj)
          nvis[jj] = (j0 + jj < j1) ? group_nvis_query(p, g, j0 + jj) : 0;
      }
      if (!mbar_wait(acc_full + acc, aph, p.err, wl)) break;
      tc_fence_after();
      const int t = it - gc.lo;
      const int e = t * tile_e + row;
      // score of query j of the group from its 32 head columns r
      auto emit = [&](int j, int jj, const uint32_t (&r)[32]) {
        const float s = relu_dot32(wbuf + j * 32, r);
        const int q = g * p.qpg + j;
        const int nv = nvis[jj];
        if (p.pool) {
          // slot t * 128 + row of the pool; its entry decides validity
          const int64_t ent = (int64_t)blk * 8 + (row & 7);
          const float v = (blk >= 0 && ent < nv) ? s : -INFINITY;
          if (e < p.ld) {
            p.scores[(int64_t)q * p.ld + e] = v;
            if (use_hist) atomicAdd(hs + j * kKeyHistBins + (score_key(v) >> 21), 1u);
          }
        } else if (q < p.nq && e < nv && CSA2_IN_BOUNDS(e < p.ld, p.err)) {
          uint32_t* hq = hs + j * kKeyHistBins;
          if (p.score_bf16) {
            // the selector's precision: nearest bf16, its key histogrammed
            const uint32_t b = float_to_bf16_bits(s);
            reinterpret_cast<uint16_t*>(p.scores)[(int64_t)q * p.ld + e] = (uint16_t)b;
            if (use_hist) atomicAdd(hq + (score_key(bf16_bits_to_float(b)) >> 21), 1u);
          } else {
            p.scores[(int64_t)q * p.ld + e] = s;
            if (use_hist) atomicAdd(hq + (score_key(s) >> 21), 1u);
          }
        }
      };
      const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * acc_cols);
      // the accumulator is free once this warp's last columns are read
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty + acc);
      };
      if constexpr (kMaxQ == 2) {
        // one query's 32 columns at a time (the register budget of sixteen
        // epilogue warps); the other warps of the scheduler cover the loads
        uint32_t r[32];
        if (j0 < j1) tmem_ld32(lane_base + (uint32_t)(j0 * 32), r);
        if (j0 + 1 >= j1) release();
        if (j0 < j1) emit(j0, 0, r);
        if (j0 + 1 < j1) {
          tmem_ld32(lane_base + (uint32_t)((j0 + 1) * 32), r);
          release();
          emit(j0 + 1, 1, r);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < kMaxQ; jj += 2) {   // two queries' columns under one TMEM wait
          const int j = j0 + jj;
          if (j + 1 < j1) {
            uint32_t ra[32], rb[32];
            tmem_ld32x2(lane_base + (uint32_t)(j * 32), lane_base + (uint32_t)((j + 1) * 32), ra, rb);
            emit(j, jj, ra);
            emit(j + 1, jj + 1, rb);
          } else if (j < j1) {
            uint32_t r[32];
            tmem_ld32(lane_base + (uint32_t)(j * 32), r);
            emit(j, jj, r);
          }
        }
        release();
      }
      if (++acc == 2) { acc = 0; aph ^= 1; }
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

int index_smem_bytes(int qpg) { return smem_layout(qpg).total; }

cudaError_t launch_index(const IndexParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_q,
                         int grid, cudaStream_t s) {
  // the epilogue covers at most kMaxQpg queries per tile (N <= 256)
  if (p.qpg < 1 || p.qpg > kMaxQpg) return cudaErrorInvalidValue;
  const int smem = index_smem_bytes(p.qpg);
  const int epi_warps = p.qpg == 1 ? 8 : 16;
  auto* kern = p.qpg == 1 ? k_index<8> : k_index<16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)(64 + 32 * epi_warps));
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tm_k, tm_q);
}

}  // namespace csa2
