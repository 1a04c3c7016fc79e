// k_index_fp4.cu -- CSA2 indexer scores over MXFP4 indexer keys and queries,
// on the block-scaled tensor-core MMA.
//
// The V4.1 report (section 2.4.4) keeps the indexer's queries and keys in
// OCP MXFP4: E2M1 codes with one power-of-two (UE8M0) scale per 32
// channels, 64 + 4 bytes per 128-channel key (the 68 B of the cache-size
// breakdown).  The score is the one of the bf16 indexer,
//     I[q, s] = sum_h w[q, h] * ReLU(q^[q, h] . K^[s]),
// over the dequantised values q^, K^.  tcgen05.mma.kind::mxf4.block_scale
// takes exactly these operands: E2M1 codes from shared memory (two per
// byte) and one UE8M0 scale per 32 elements of K from tensor memory, with
// fp32 accumulation, so the cached codes go to the tensor cores as they are.
//
// Operands of one MMA (M = 128 keys, N = 32 heads x qpg, K = 64):
//   A  key codes, K-major, 64-byte rows with the 64-byte swizzle.
//      Contiguous keys come in aligned tiles of 128 or 256 keys whose rows
//      are permuted: key 128 h + 4 r + q of the tile (r < 32, q < 4) is row
//      32 q + r of M-group h (one TMA box per M-group), so that the tile's
//      scale words, copied in their natural order, are already the scale
//      atoms below.  In pool mode one box per block of 8 keys (exactly one
//      512-byte swizzle atom), in pool order.  Two K steps of 32 bytes cover
//      the 128 channels;
//   B  query codes in the same layout, written by the query-preparation
//      warps (each query head rounded to the MXFP4 grid);
//   SFA / SFB  scale bytes in tensor memory: a 512-byte atom per 128 rows in
//      which row 32 q + r holds its four block scales at byte 16 r + 4 q
//      (tcgen05.cp 32x128b.warpx4 puts 32 lanes x 16 bytes into every lane
//      quadrant; the MMA reads quadrant q's lanes at column q), the K step
//      choosing the byte pair (scale id 0 or 2).
//
// Warp roles (384 threads):
//   warp 0      producer: per tile one TMA box of key codes and one bulk
//               copy of its scale words (contiguous tiles), or a box per
//               block and a 4-byte copy per scale word into its atom place
//               (pool mode);
//   warp 1      MMA issuer (and TMEM owner): per tile the MMAs, one
//               accumulator per tile, once its key scales are in place;
//   warps 2-9   epilogue: ReLU, head weights, fp32 or bf16 score store,
//               score-key histogram (the bf16 indexer's);
//   warps 10-11 query preparation: at every new query group the bf16 query
//               heads are rounded to MXFP4 codes and scales into one of two
//               B slots, ahead of the MMAs of that group;
//   warp 12     scale copies of decode tiles: per tile, once it has
//               landed, the key scale atoms into its stage's scale columns
//               (tcgen05.cp; the stage's previous tile was read by MMAs that
//               completed before the stage was refilled), signalled to the
//               MMA issuer by a commit (a single thread issuing every tcgen05
//               instruction of a tile was the decode kernel's bound).  In
//               pool mode and prefill the MMA issuer copies them itself.
// Tiles: 512 keys (four M = 128 groups) for one query per group over
// contiguous keys (decode), 512 pool slots (four M-groups) in pool mode, 128
// keys for four queries per group (prefill, N = 128).
// Every wait is bounded.
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

constexpr int kThreads = 416;
constexpr int kEpiThreads = 256;   // warps 2-9
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kPrepBase = 320;     // warps 10-11
constexpr int kSfWarp = 12;        // scale-atom copies
constexpr int kPrepThreads = 64;
constexpr int kPrepWarps = kPrepThreads / 32;
#ifndef CSA2_FP4_STAGES
#define CSA2_FP4_STAGES 5
#endif
constexpr int kStages = CSA2_FP4_STAGES;
constexpr int kTileMax = 512;
constexpr int kCodeStage = kTileMax * (kIdxDim / 2);   // 32 KB of E2M1 codes
constexpr int kSfAtom = 512;                           // scales of 128 rows
constexpr int kStageBytes = kCodeStage + (kTileMax / 128) * kSfAtom;   // 34 KB
constexpr int kMaxQpg = 4;
constexpr int kBRows = 32 * kMaxQpg;
constexpr int kBSlotBytes = 9216;    // 8 KB of query codes + one scale atom (1024-aligned)
constexpr int kPf = 4;               // tiles of scale words loaded ahead by the producer
constexpr int kNAcc = 4;               // accumulators at most
// tensor-memory columns: accumulators (as many as fit below kAccCols, at
// most kNAcc), then the key scales of each stage's tile (4 columns per
// M-group), then the query scales of the two B slots
constexpr uint32_t kAccCols = 384;
constexpr uint32_t kSfaCols = 16 * kStages;        // [kStages][4 M-groups][4 columns]
constexpr uint32_t kSfaCol = kAccCols;
constexpr uint32_t kSfbCol = kSfaCol + kSfaCols;   // [2 B slots][4 columns]
constexpr uint32_t kTmemCols = 512;
static_assert(kSfbCol + 8 <= kTmemCols, "tensor memory");

constexpr int kMaxPoolIds = 4096;    // block ids of one query's pool (pool mode)

struct SmemLayout {
  int b_off, w_off, hist_off, ids_off, bar_off, total;
};

__host__ __device__ inline SmemLayout smem_layout() {
  SmemLayout L;
  L.b_off = kStages * kStageBytes;
  L.w_off = L.b_off + 2 * kBSlotBytes;
  L.hist_off = L.w_off + kBRows * 4;
  L.ids_off = L.hist_off + kKeyHistBins * 4;
  L.bar_off = L.ids_off + kMaxPoolIds * 4;
  L.total = L.bar_off + 64 * 8 + 16 + 1024;   // barriers, tmem slot, alignment slack
  static_assert(kStages <= 6 && kNAcc <= 8, "barrier slots");
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

// Walks the tile list; group g holds tiles [lo, hi) and its keys start at
// row `base`.  The parameter tables are read only when the group changes: a
// dynamically indexed kernel parameter is read through the constant cache,
// and a miss there on every tile costs hundreds of cycles.
struct Cursor {
  int g, lo, hi;
  int64_t base;
  __device__ __forceinline__ void init(const IndexParams& p, int g0) {
    g = g0;
    lo = p.tile_prefix[g0];
    hi = p.tile_prefix[g0 + 1];
    base = group_base(p, g0);
  }
  __device__ __forceinline__ bool advance(const IndexParams& p, int it) {
    if (it < hi) return false;
    do {
      ++g;
      lo = hi;
      hi = p.tile_prefix[g + 1];
    } while (hi <= it);
    base = group_base(p, g);
    return true;
  }
};

// Shared-memory descriptor of a K-major operand in 64-byte rows with the
// 64-byte swizzle: 8-row atoms of 512 bytes, one after the other.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                      // leading byte offset 16 (unused)
  d |= (uint64_t)(512u >> 4) << 32;            // 8-row groups 512 bytes apart
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;                      // SWIZZLE_64B
  return d;
}

// Descriptor of a scale atom (32 rows of 16 bytes, no swizzle) for
// tcgen05.cp 32x128b.
__device__ __forceinline__ uint64_t sdesc_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 16;
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// 4-byte asynchronous copy global -> shared (src_bytes 0: the word is
// zero-filled and nothing is read), and an arrival on `bar` once every such
// copy of this thread has landed (the barrier's count includes it).
__device__ __forceinline__ void cp_async4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Instruction descriptor of kind::mxf4 (E2M1 x E2M1, UE8M0 scales, fp32 D,
// K-major A and B); `sf` (0 or 2) picks the scale byte pair of the K step.
__device__ __forceinline__ uint32_t idesc_mxf4(uint32_t N, uint32_t sf) {
  return (sf << 4)               // scale id of B
         | (1u << 7)             // A = E2M1
         | (1u << 10)            // B = E2M1
         | ((N >> 3) << 17)
         | (1u << 23)            // scale format UE8M0
         | ((128u >> 4) << 24)   // M = 128
         | (sf << 29);           // scale id of A
}

__device__ __forceinline__ void umma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Block b (32 channels) of query head row n: bf16 from global memory ->
// MXFP4 (UE8M0 scale of the block's largest magnitude, OCP MX rule; E2M1
// code of x / scale, nearest, ties to even, saturating) -> 16 code bytes in
// the B slot's swizzled row and the scale byte in its atom.
__device__ __forceinline__ void prep_query_block(const uint16_t* src, bool live, uint8_t* bcodes,
                                                 uint8_t* batom, int n, int b) {
  float x[32];
  if (live) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = __ldg(s4 + k);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * k + 2 * i] = __uint_as_float(u[i] << 16);
        x[8 * k + 2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t sb = ue8m0_for_amax(amax);   // 0 .. 252 for finite maxima
  // x / 2^(sb - 127) as x * 2^(127 - sb): the reciprocal (byte 254 - sb) is
  // an exact normal power of two, so the product is the correctly rounded
  // quotient
  const float inv = ue8m0_value(254u - sb);
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= e2m1_encode(__fmul_rn(x[8 * k + i], inv)) << (4 * i);
    c[k] = w;
  }
  uint8_t* row = bcodes + (n >> 3) * 512 + (n & 7) * 64;
  *reinterpret_cast<uint4*>(row + ((b ^ ((n >> 1) & 3)) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
  batom[(n & 31) * 16 + ((n >> 5) & 3) * 4 + b] = (uint8_t)sb;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_index_fp4(const __grid_constant__ IndexParams p, const __grid_constant__ CUtensorMap tm_kq,
                const __grid_constant__ CUtensorMap tm_kc8) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const SmemLayout L = smem_layout();
  uint8_t* stages = smem;
  uint8_t* bslots = smem + L.b_off;
  float* wbuf = reinterpret_cast<float*>(smem + L.w_off);
  uint32_t* hs = reinterpret_cast<uint32_t*>(smem + L.hist_off);
  int32_t* ids_s = reinterpret_cast<int32_t*>(smem + L.ids_off);   // pool ids of the group
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* k_full = bars;                 // [kStages]
  uint64_t* k_empty = bars + 16;           // [kStages]
  uint64_t* acc_full = bars + 32;          // [kNAcc]
  uint64_t* acc_empty = bars + 40;         // [kNAcc]
  uint64_t* b_full = bars + 48;            // [2]
  uint64_t* b_empty = bars + 50;           // [2]
  uint64_t* drain = bars + 52;
  uint64_t* sf_drain = bars + 53;
  uint64_t* sf_full = bars + 56;           // [kStages]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 62);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = 32 * p.qpg;                      // MMA N
  const bool pool = p.pool != nullptr;
  // keys (pool slots) per tile: 512 for one query (contiguous keys, or 64
  // pool blocks of 8), 128 for four queries
  const int tile_e = p.qpg == 1 ? 512 : 128;
  const int mgroups = tile_e / 128;
  const int acc_cols = mgroups * N;              // 128, 64 or 128 columns
  const int nacc = min(kNAcc, (int)kAccCols / acc_cols);   // 3, 4 or 3 accumulators
  const int blocks_per_tile = tile_e / 8;
  // Contiguous keys: tiles are aligned chunks of tile_e key rows, so a
  // sequence starting inside a chunk begins `lead` keys into its first tile
  // (masked); slot sl (M-group sl / 128, TMEM lane sl % 128) holds the key
  // (sl & ~127) + 4 (sl & 31) + (sl >> 5) % 4 of the tile.  Pool mode: slot
  // sl is pool slot sl of the tile, no permutation.
  const bool perm = !pool;
  // decode over contiguous keys: the key scale copies run on their own warp
  // (elsewhere the epilogue bounds the pipeline and the MMA issuer copies
  // them itself)
  const bool sf_warp = perm && p.qpg == 1;
  auto slot_key = [&](int sl) -> int {
    return perm ? (sl & ~127) + 4 * (sl & 31) + ((sl >> 5) & 3) : sl;
  };
  auto lead_of = [&](const Cursor& c) -> int { return perm ? (int)(c.base & (tile_e - 1)) : 0; };
  auto tile_row0 = [&](const Cursor& c, int it) -> int64_t {
    return (perm ? (c.base & ~(int64_t)(tile_e - 1)) : c.base) + (int64_t)(it - c.lo) * tile_e;
  };

  if (threadIdx.x == 0) {
    // k_full: the copies' transaction bytes with lane 0's arrival, plus in
    // pool mode one arrival per producer lane once its scale copies landed
    for (int i = 0; i < kStages; ++i) { mbar_init(k_full + i, pool ? 33 : 1); mbar_init(k_empty + i, 1); }
    for (int i = 0; i < kNAcc; ++i) { mbar_init(acc_full + i, 1); mbar_init(acc_empty + i, kEpiWarps); }
    for (int i = 0; i < 2; ++i) { mbar_init(b_full + i, kPrepWarps); mbar_init(b_empty + i, 1); }
    for (int i = 0; i < kStages; ++i) mbar_init(sf_full + i, 1);
    mbar_init(drain, 1);
    mbar_init(sf_drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(pool ? &tm_kc8 : &tm_kq);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, kTmemCols); tmem_relinquish(); }
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
  Cursor c0;
  c0.init(p, g0);
  // pool row of tile `it` (its group at or after the cursor's): block ids
  auto pool_row = [&](int it, Cursor c) -> const int32_t* {
    c.advance(p, it);
    return p.pool + (int64_t)c.g * p.pool_blocks + (int64_t)(it - c.lo) * blocks_per_tile;
  };
  auto pool_len = [&](int it, Cursor c) -> int {   // valid blocks in tile `it`
    c.advance(p, it);
    const int left = p.pool_blocks - (it - c.lo) * blocks_per_tile;
    return left < blocks_per_tile ? left : blocks_per_tile;
  };

  if (warp == 0 && begin < end) {
    // ------------------------------------------------ producer
    // Contiguous tiles: lane 0 issues one TMA box of key codes and one bulk
    // copy of the tile's scale words (their natural order is the atom
    // layout of the permuted rows).  Pool mode: one box per block of 8 keys
    // and each key's scale word by a 4-byte asynchronous copy straight into
    // its place in the scale atom (lane r copies rows 32 q + r), completing
    // on the stage's barrier; the block ids are loaded kPf tiles ahead, slot
    // u of the ring holding the tiles it = u (mod kPf), the loop unrolled
    // over the slots so that no register of a load in flight is ever
    // copied.  The warp never waits for a load.
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(p.idx_scales);   // one word per key
    const uint64_t keys_pol = l2_policy_evict_first();
    // pool mode: this lane's block ids (blocks lane and lane + 32) of tiles
    // it .. it + kPf - 1
    int32_t pq[kPf][2];
    Cursor pc_id = c0;
    auto load_ids = [&](int j, int h) -> int32_t {
      if (!pool || j >= end) return -1;
      pc_id.advance(p, j);
      if (lane + 32 * h >= pool_len(j, pc_id)) return -1;
      return __ldg(pool_row(j, pc_id) + lane + 32 * h);
    };
#pragma unroll
    for (int u = 0; u < kPf; ++u) {
      pq[u][0] = load_ids(begin + u, 0);
      pq[u][1] = load_ids(begin + u, 1);
    }

    Cursor gc = c0;
    int stage = 0;
    uint32_t ph = 0;
    uint32_t armed = 0, armed_ph = 0;   // stages filled at least once, parity of the last fill
    bool ok = true;
    for (int it0 = begin; it0 < end && ok; it0 += kPf) {
#pragma unroll
      for (int u = 0; u < kPf; ++u) {
        const int it = it0 + u;
        if (it >= end || !ok) break;
        gc.advance(p, it);
        if (lane == 0) ok = mbar_wait(k_empty + stage, ph ^ 1, p.err, wl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (p.inject & kInjectNoKeyLoads) {   // tests: nothing arrives on k_full
          if (++stage == kStages) { stage = 0; ph ^= 1; }
          continue;
        }
        uint8_t* st = stages + stage * kStageBytes;
        if (!pool) {
          if (lane == 0) {
            const int64_t row0 = tile_row0(gc, it);   // a multiple of tile_e
            const int32_t chunk = (int32_t)(row0 / 128);
            mbar_arrive_expect_tx(k_full + stage, (uint32_t)(mgroups * (128 * (kIdxDim / 2) + kSfAtom)));
            for (int mg = 0; mg < mgroups; ++mg)
              tma_load_4d(st + mg * 128 * (kIdxDim / 2), &tm_kq, 0, 0, 0, chunk + mg, k_full + stage,
                          keys_pol);
            bulk_load(st + kCodeStage, sw + row0, (uint32_t)(mgroups * kSfAtom), k_full + stage);
          }
        } else {
          const int64_t base = gc.base;
          const int32_t blk_lo = pq[u][0], blk_hi = pq[u][1];   // blocks lane, lane + 32
          // scale words into the atoms: row 32 q + r of M-group mg at byte
          // 16 r + 4 q of that group's atom; the slot's block is mg 16 +
          // 4 q + lane / 8, in the first half of the tile for mg < 2
#pragma unroll
          for (int mg = 0; mg < 4; ++mg) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int sl = mg * 128 + 32 * q + lane;     // pool slot of the tile
              const int32_t blk = __shfl_sync(0xffffffffu, mg < 2 ? blk_lo : blk_hi, (sl >> 3) & 31);
              const int64_t row = blk >= 0 ? base + (int64_t)blk * 8 + (sl & 7) : -1;
              const bool live = row >= 0 && row < p.idx_total;
              cp_async4(st + kCodeStage + mg * kSfAtom + lane * 16 + q * 4, sw + (live ? row : 0),
                        live ? 4u : 0u);
            }
          }
          cp_async_arrive_noinc(k_full + stage);
          const uint32_t n_ok = (uint32_t)__popc(__ballot_sync(0xffffffffu, blk_lo >= 0)) +
                                (uint32_t)__popc(__ballot_sync(0xffffffffu, blk_hi >= 0));
          if (lane == 0) mbar_arrive_expect_tx(k_full + stage, n_ok * 512u);
          __syncwarp();
          if (blk_lo >= 0)
            tma_load_2d(st + lane * 512, &tm_kc8, 0, (int32_t)(base + (int64_t)blk_lo * 8),
                        k_full + stage, keys_pol);
          if (blk_hi >= 0)
            tma_load_2d(st + (lane + 32) * 512, &tm_kc8, 0, (int32_t)(base + (int64_t)blk_hi * 8),
                        k_full + stage, keys_pol);
        }
        armed |= 1u << stage;
        armed_ph = (armed_ph & ~(1u << stage)) | (ph << stage);
        if (++stage == kStages) { stage = 0; ph ^= 1; }
        pq[u][0] = load_ids(it + kPf, 0);
        pq[u][1] = load_ids(it + kPf, 1);
      }
    }
    // no bulk copy may still be writing into this CTA's shared memory
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s)
        if (armed & (1u << s)) mbar_wait(k_full + s, (armed_ph >> s) & 1u, p.err, wl);
    }
    __syncwarp();
  } else if (warp >= kPrepBase / 32 && warp < kSfWarp && begin < end) {
    // ------------------------------------------------ query preparation
    const int pt = threadIdx.x - kPrepBase;
    const int qrows = 32 * p.qpg;
    Cursor gc = c0;
    int cur = -1, gi = 0;
    bool ok = true;
    for (int it = begin; it < end && ok; ++it) {
      gc.advance(p, it);
      if (gc.g == cur) continue;
      cur = gc.g;
      const int slot = gi & 1;
      ok = mbar_wait_sleep(b_empty + slot, (uint32_t)(((gi >> 1) & 1) ^ 1), p.err, wl);
      if (!ok) break;
      uint8_t* bc = bslots + slot * kBSlotBytes;
      uint8_t* ba = bc + kBRows * (kIdxDim / 2);
      for (int i = pt; i < kSfAtom / 4; i += kPrepThreads) reinterpret_cast<uint32_t*>(ba)[i] = 0u;
      asm volatile("bar.sync 2, 64;" ::: "memory");   // both warps: zeroed before any scale byte
      for (int item = pt; item < qrows * 4; item += kPrepThreads) {
        const int n = item >> 2, b = item & 3;
        const int q = cur * p.qpg + (n >> 5);
        const bool live = q < p.nq;
        const uint16_t* src = p.q_idx + ((int64_t)q * kIdxHeads + (n & 31)) * kIdxDim + b * 32;
        prep_query_block(src, live, bc, ba, n, b);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_full + slot);
      ++gi;
    }
  } else if (warp == kSfWarp && lane == 0 && sf_warp && begin < end) {
    // ------------------------------------------------ scale copies
    const uint64_t atom_desc0 = sdesc_atom(smem_u32(stages + kCodeStage));
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int it = begin; it < end && ok; ++it) {
      ok = mbar_wait(k_full + stage, ph, p.err, wl);
      if (!ok) break;
      tc_fence_after();
      const uint32_t so = (uint32_t)(stage * kStageBytes) >> 4;
      const uint32_t sfa = tmem_base + kSfaCol + (uint32_t)(stage * 16);
      for (int mg = 0; mg < mgroups; ++mg)
        tmem_cp_atom(sfa + 4 * mg, atom_desc0 + so + (uint32_t)(mg * (kSfAtom >> 4)));
      umma_commit(sf_full + stage);
      if (++stage == kStages) { stage = 0; ph ^= 1; }
    }
    umma_commit(sf_drain);
    mbar_wait(sf_drain, 0, p.err, wl);
  } else if (warp == 1 && lane == 0 && begin < end) {
    // ------------------------------------------------ MMA issuer
    // Shared-memory descriptors built once; a tile's offsets go into the
    // start-address field (16-byte units; shared memory is below 2^18
    // bytes, so the field never carries).  A: 64-byte rows, M-group h 8 KB
    // further, K step ks 32 bytes further.
    const uint64_t a_desc0 = sdesc_sw64(smem_u32(stages));
    const uint32_t a_mg = (uint32_t)(128 * (kIdxDim / 2)) >> 4;
    const uint64_t b_desc0 = sdesc_sw64(smem_u32(bslots));
    const uint64_t atom_desc0 = sdesc_atom(smem_u32(stages + kCodeStage));
    const uint32_t idesc_k0 = idesc_mxf4((uint32_t)N, 0u), idesc_k1 = idesc_mxf4((uint32_t)N, 2u);
    Cursor gc = c0;
    int cur = -1, gi = -1, stage = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int it = begin; it < end && ok; ++it) {
      const bool changed = gc.advance(p, it) || cur < 0;
      if (changed) {
        ++gi;
        cur = gc.g;
        ok = mbar_wait(b_full + (gi & 1), (uint32_t)((gi >> 1) & 1), p.err, wl);
        if (!ok) break;
        tc_fence_after();
        uint8_t* ba = bslots + (gi & 1) * kBSlotBytes + kBRows * (kIdxDim / 2);
        tmem_cp_atom(tmem_base + kSfbCol + 4 * (gi & 1), sdesc_atom(smem_u32(ba)));
      }
      // the tile's codes have landed, its key scales are in tensor memory
      // and its accumulator is free
      ok = mbar_wait(k_full + stage, ph, p.err, wl) &&
           (!sf_warp || mbar_wait(sf_full + stage, ph, p.err, wl)) &&
           mbar_wait(acc_empty + acc, aph ^ 1, p.err, wl);
      if (!ok) break;
      tc_fence_after();
      const uint32_t so = (uint32_t)(stage * kStageBytes) >> 4;   // stage offset, 16-byte units
      const uint32_t sfa = tmem_base + kSfaCol + (uint32_t)(stage * 16);
      if (!sf_warp) {
        // pool mode: the scale words arrived by generic-proxy copies, which
        // tcgen05.cp reads through the async proxy
        if (pool) fence_proxy_async_smem();
        for (int mg = 0; mg < mgroups; ++mg)
          tmem_cp_atom(sfa + 4 * mg, atom_desc0 + so + (uint32_t)(mg * (kSfAtom >> 4)));
      }
      const uint32_t bo = (uint32_t)((gi & 1) * kBSlotBytes) >> 4;
      const uint32_t sfb = tmem_base + kSfbCol + 4 * (gi & 1);
      for (int mg = 0; mg < mgroups; ++mg) {
        const uint32_t d = tmem_base + (uint32_t)(acc * acc_cols + mg * N);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_mxf4(d, a_desc0 + so + (uint32_t)(mg * a_mg + 2 * ks), b_desc0 + bo + (uint32_t)(2 * ks),
                    ks ? idesc_k1 : idesc_k0, sfa + 4 * mg, sfb, ks > 0 ? 1u : 0u);
      }
      umma_commit(k_empty + stage);
      umma_commit(acc_full + acc);
      const bool last_of_group = (it + 1 == end) || (gc.hi <= it + 1);
      if (last_of_group) umma_commit(b_empty + (gi & 1));
      if (++stage == kStages) { stage = 0; ph ^= 1; }
      if (++acc == nacc) { acc = 0; aph ^= 1; }
    }
    umma_commit(drain);
    mbar_wait(drain, 0, p.err, wl);
  } else if (warp >= 2 && warp < 10) {
    // ------------------------------------------------ epilogue
    const int quad = warp & 3;                 // TMEM lane quadrant
    const int et = threadIdx.x - 64;           // 0..255
    // one query: warps 2-5 take the first half of the tile's M-groups, warps
    // 6-9 the second half (one or two M-groups each); four queries: warps
    // 2-5 the queries 0-1, warps 6-9 the queries 2-3 of the one M-group
    const int half = (warp - 2) >> 2;
    const int mgh = p.qpg == 1 ? mgroups / 2 : 1;   // M-groups of one epilogue thread
    const int slot0 = (p.qpg == 1 ? half * mgh * 128 : 0) + quad * 32 + lane;   // its first slot
    const bool use_hist = p.key_hist != nullptr && p.qpg == 1;
    const int qrows = 32 * p.qpg;
    auto esync = [&]() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    auto flush = [&](int qq) {
      esync();
      for (int i = et; i < kKeyHistBins; i += kEpiThreads) {
        const uint32_t v = hs[i];
        if (v) atomicAdd(p.key_hist + (int64_t)qq * kKeyHistBins + i, v);
        hs[i] = 0u;
      }
      esync();
    };
    if (use_hist)
      for (int i = et; i < kKeyHistBins; i += kEpiThreads) hs[i] = 0u;
    Cursor gc = c0;
    int cur = -1, acc = 0, t_first = 0;
    uint32_t aph = 0;
    int nv[2] = {0, 0};   // visible entries of this thread's queries
    for (int it = begin; it < end; ++it) {
      gc.advance(p, it);
      const int g = gc.g;
      if (g != cur) {
        if (use_hist && cur >= 0) flush(cur);
        esync();
        for (int i = et; i < qrows; i += kEpiThreads) {
          const int q = g * p.qpg + (i >> 5);
          wbuf[i] = (q < p.nq) ? __ldg(p.w + (int64_t)q * kIdxHeads + (i & 31)) : 0.0f;
        }
        if (pool) {
          // the block ids of this CTA's tiles of the group, loaded once
          t_first = (begin > gc.lo ? begin : gc.lo) - gc.lo;
          const int t_last = (end < gc.hi ? end : gc.hi) - gc.lo;
          const int i0 = t_first * blocks_per_tile;
          const int i1 = min(t_last * blocks_per_tile, p.pool_blocks);
          const int32_t* src = p.pool + (int64_t)g * p.pool_blocks;
          for (int i = i0 + et; i < i1; i += kEpiThreads) ids_s[i - i0] = __ldg(src + i);
        }
        esync();
        cur = g;
        if (p.qpg == 1) {
          nv[0] = group_nvis_query(p, g, 0);
        } else {
          nv[0] = group_nvis_query(p, g, 2 * half);
          nv[1] = group_nvis_query(p, g, 2 * half + 1);
        }
      }
      if (!mbar_wait_sleep(acc_full + acc, aph, p.err, wl)) break;
      tc_fence_after();
      const int t = it - gc.lo;
      const int lead = lead_of(gc);
      const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * acc_cols);
      // score s of query q at slot `row` of the tile: entry e (pool mode: the
      // pool slot, whose block decides validity)
      auto store = [&](int row, int q, int nvis, float s) {
        const int e = t * tile_e + slot_key(row) - lead;
        if (pool) {
          int32_t blk = -1;
          if (t * blocks_per_tile + (row >> 3) < p.pool_blocks)
            blk = ids_s[(t - t_first) * blocks_per_tile + (row >> 3)];
          const int64_t ent = (int64_t)blk * 8 + (row & 7);
          const float v = (blk >= 0 && ent < nvis) ? s : -INFINITY;
          if (e < p.ld) {
            p.scores[(int64_t)q * p.ld + e] = v;
            if (use_hist) atomicAdd(hs + (score_key(v) >> 21), 1u);
          }
        } else if (q < p.nq && e >= 0 && e < nvis && CSA2_IN_BOUNDS(e < p.ld, p.err)) {
          if (p.score_bf16) {
            const uint32_t bb = float_to_bf16_bits(s);
            reinterpret_cast<uint16_t*>(p.scores)[(int64_t)q * p.ld + e] = (uint16_t)bb;
            if (use_hist) atomicAdd(hs + (score_key(bf16_bits_to_float(bb)) >> 21), 1u);
          } else {
            p.scores[(int64_t)q * p.ld + e] = s;
            if (use_hist) atomicAdd(hs + (score_key(s) >> 21), 1u);
          }
        }
      };
      if (p.qpg == 1 && mgh == 1) {
        uint32_t r[32];
        tmem_ld32(lane_base + (uint32_t)(half * N), r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty + acc);
        store(slot0, g, nv[0], relu_dot32(wbuf, r));
      } else if (p.qpg == 1) {
        // M-groups 2 half and 2 half + 1: columns N apart
        uint32_t ra[32], rb[32];
        const uint32_t c0 = (uint32_t)(2 * half * N);
        tmem_ld32x2(lane_base + c0, lane_base + c0 + (uint32_t)N, ra, rb);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty + acc);
        store(slot0, g, nv[0], relu_dot32(wbuf, ra));
        store(slot0 + 128, g, nv[0], relu_dot32(wbuf, rb));
      } else {
        uint32_t ra[32], rb[32];
        const int j = 2 * half;
        tmem_ld32x2(lane_base + (uint32_t)(j * 32), lane_base + (uint32_t)((j + 1) * 32), ra, rb);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty + acc);
        store(slot0, g * p.qpg + j, nv[0], relu_dot32(wbuf + j * 32, ra));
        store(slot0, g * p.qpg + j + 1, nv[1], relu_dot32(wbuf + (j + 1) * 32, rb));
      }
      if (++acc == nacc) { acc = 0; aph ^= 1; }
    }
    if (use_hist && cur >= 0) flush(cur);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

int index_fp4_smem_bytes() { return smem_layout().total; }

cudaError_t launch_index_fp4(const IndexParams& p, const CUtensorMap& tm_kq,
                             const CUtensorMap& tm_kc8, int grid, cudaStream_t s) {
  if (p.qpg != 1 && p.qpg != kMaxQpg) return cudaErrorInvalidValue;
  const int smem = index_fp4_smem_bytes();
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
  return cudaLaunchKernelEx(&cfg, k_index_fp4, p, tm_kq, tm_kc8);
}

}  // namespace csa2
