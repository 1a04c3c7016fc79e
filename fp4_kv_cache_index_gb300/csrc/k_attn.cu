// k_attn.cu -- CSA2 sparse shared-KV attention over FP4 cache entries plus
// the sliding window, one joint softmax.
//
// Method: the selected compressed entries are both key and value (blog
// reading of the DeepSeek-V4 report, section 4.1, "shared key-value MQA");
// the window rows join the same softmax (same blog, section 4.3; neshdevtech
// article section 3.3.1, "readout concatenates the SWA and the selected main
// KV into a single joint sparse attention"); entries are dequantised from
// FP4 before attention (V4.1 report, section 2.4.4).
//
// One CTA = one query x 64 heads x one share of the candidate tiles of one
// layer (a launch may hold several layers of a group, which share the cache,
// the selection and the window geometry: their CTAs pack the SMs without a
// launch boundary between the layers).  With
// `splits` = 2 (small decode batches) the tiles of a query alternate between
// the two CTAs of a cluster, which merge their unnormalised fp32 states
// (running max, sum, O) exactly through distributed shared memory, each
// finalising one half of the head dimension; with splits = 1 a CTA takes
// every tile.  Candidates come in tiles of 128 rows: the window tile (TMA
// straight into swizzled shared memory) and the top-k tiles (each thread
// loads 64 code bytes of one entry plus their scale bytes into registers,
// one tile ahead; then E2M1 -> bf16 via byte permutes and a bf16 scale
// multiply, written to shared memory in the MMA layout).  With the candidate
// rows as the MMA M dimension:
//     S^T[128 x 64]  = KV[128 x 512] * Q[64 x 512]^T        (K-major A and B)
//     O^T[512 x 64] += KV^T[512 x 128] * P^T[128 x 64]       (MN-major A and B)
// both on tcgen05 with fp32 accumulators in TMEM; the same swizzled KV tile
// serves as the K-major A of the first product and the MN-major A of the
// second, and P^T is written by the softmax one candidate row per thread.  The single KV buffer is refilled in two channel halves: the next
// tile's first half as soon as the O^T products that read it are done (while
// the others run), and S^T of that half while the second half is written.
// Online softmax (base 2) runs across TMEM lanes: each thread holds one
// candidate row; a head's running maximum moves (with a reduce-scatter over
// the rows and a rescale of O^T in TMEM) only when a tile holds a logit more
// than 2^8 above it, and the row sums are kept per thread and reduced once.
#include "csa2_device.cuh"
#include "csa2_kernels.h"

namespace csa2 {
namespace {

constexpr int kThreads = 512;     // 16 warps
constexpr int kHG = 64;               // heads per CTA
constexpr int kRows = 128;            // candidates per tile
constexpr int kMaxTiles = 2048 / kRows + 1;
constexpr float kLazyRescale = 8.0f;  // log2 units

// shared memory map (offsets from a 1024-aligned base)
constexpr int kKvOff = 0;                              // 8 x [128 x 128 B]
constexpr int kQOff = kKvOff + kRows * kHeadDim * 2;   // 8 x [64 x 128 B]
constexpr int kPOff = kQOff + kHG * kHeadDim * 2;      // [128 x 128 B]
constexpr int kIdxOff = kPOff + kHG * kRows * 2;        // the query's top-k row
constexpr int kSmallOff = kIdxOff + 2048 * 4;
struct Small {
  float red_max[4][kHG];
  float red_sum[4][kHG];
  float m[kHG];
  float l[kHG];
  float alpha[kHG];
  int32_t my_list[kMaxTiles];    // this CTA's share
  int32_t tile_any[kMaxTiles];   // top-k tile holds a usable index
  uint8_t row_valid[kRows];
  int32_t n_tiles;
  float rope_c[32], rope_s[32];  // output RoPE(-i): cos, sin of each channel pair
  uint32_t tmem;
  uint64_t bar_q[2], bar_kv[2], bar_mma, bar_o[2];   // [h]: channel half h
};
constexpr int kSmemBytes = kSmallOff + (int)sizeof(Small) + 1024;


// Reduce-scatter over the 32 lanes of a warp: v[0..15] (16 heads) in, lane L
// ends with the reduction for head (L >> 1) in v[0].
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = lane & 16;
    const float send = up ? v[i] : v[i + 8];
    const float keep = up ? v[i + 8] : v[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 16);
    v[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 8;
    const float send = up ? v[i] : v[i + 4];
    const float keep = up ? v[i + 4] : v[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 8);
    v[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 4;
    const float send = up ? v[i] : v[i + 2];
    const float keep = up ? v[i + 2] : v[i];
    const float r = __shfl_xor_sync(0xffffffffu, send, 4);
    v[i] = kMax ? fmaxf(keep, r) : keep + r;
  }
  {
    const bool up = lane & 2;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    const float r = __shfl_xor_sync(0xffffffffu, send, 2);
    v[0] = kMax ? fmaxf(keep, r) : keep + r;
  }
  const float r = __shfl_xor_sync(0xffffffffu, v[0], 1);
  return kMax ? fmaxf(v[0], r) : v[0] + r;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attn(const __grid_constant__ AttnParams p, const __grid_constant__ AttnMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kv = smem + kKvOff;
  uint8_t* qs = smem + kQOff;
  uint8_t* ps = smem + kPOff;
  int32_t* idx_s = reinterpret_cast<int32_t*>(smem + kIdxOff);
  Small& sm = *reinterpret_cast<Small*>(smem + kSmallOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();
  const long long wl = wait_limit(p.wait_cycles);   // bounded-wait limit (cycles)
  const int hgs = p.n_heads / kHG;
  // blocks of one launch: (layer, query, head group, split)
  const int per_layer = p.nq * hgs * p.splits;
  const int layer = (int)blockIdx.x / per_layer;
  const int bid = (int)blockIdx.x - layer * per_layer;
  const int split = bid % p.splits;
  const int qh = bid / p.splits;                   // (query, head group)
  const AttnLayer& ly = p.layer[layer];
  const CUtensorMap* tm_q = &maps.q[layer];
  const CUtensorMap* tm_swa = &maps.swa[layer];
  const int q = qh / hgs, hg = qh % hgs;
  const int n_topk_tiles = p.topk / kRows;
  const int32_t* idx_row = p.topk_idx + (int64_t)q * p.topk;
  // the top-k row decides the first gathers: its loads go out before
  // anything else
  int32_t idx_pre[2048 / kThreads];
#pragma unroll
  for (int j = 0; j < 2048 / kThreads; ++j) {
    const int i = tid + j * kThreads;
    idx_pre[j] = i < p.topk ? idx_row[i] : -1;
  }

  // ---- per-query geometry
  int64_t base;
  int32_t len;
  int32_t swa_row0, swa_count;
  if (p.prefill) {
    base = p.pre_base;
    len = p.pre_len;
    const int64_t pos = p.pos0 + q;
    const int64_t lo = (pos - p.swa + 1 > p.swa_pos0) ? pos - p.swa + 1 : p.swa_pos0;
    swa_row0 = (int32_t)(lo - p.swa_pos0);
    swa_count = (p.swa > 0) ? (int32_t)(pos - lo + 1) : 0;
  } else {
    base = p.q_base[q];
    len = p.q_len[q];
    swa_row0 = q * p.swa;
    int32_t c = p.swa_len ? p.swa_len[q] : p.swa;
    swa_count = c < 0 ? 0 : (c > p.swa ? p.swa : c);
  }

  // The window tile is always first in the tile list: the CTA that owns it
  // (split 0) loads it now, with the query rows, before anything else.  Both
  // come in two channel halves so that S^T of half 0 can start before half 1
  // has arrived.
  const bool swa_first = swa_count > 0 && split == 0;
  if (tid == 0) {
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sm.bar_q[h], 1);
      mbar_init(&sm.bar_kv[h], 1);
      mbar_init(&sm.bar_o[h], 1);
    }
    mbar_init(&sm.bar_mma, 1);
    fence_barrier_init();
    for (int h = 0; h < 2; ++h) {
      mbar_arrive_expect_tx(&sm.bar_q[h], kHG * kHeadDim);
      for (int c = 4 * h; c < 4 * h + 4; ++c)
        tma_load_2d(qs + c * (kHG * 128), tm_q, 64 * c, q * p.n_heads + hg * kHG, &sm.bar_q[h]);
      if (swa_first && !ly.swa_codes) {
        mbar_arrive_expect_tx(&sm.bar_kv[h], kRows * kHeadDim);
        for (int c = 4 * h; c < 4 * h + 4; ++c)
          tma_load_2d(kv + c * (kRows * 128), tm_swa, 64 * c, swa_row0, &sm.bar_kv[h]);
      }
    }
  }
  if (tid < kMaxTiles) sm.tile_any[tid] = 0;
  if (tid < kHG) { sm.m[tid] = -INFINITY; sm.l[tid] = 0.0f; }
  if (warp == 0) { tmem_alloc(&sm.tmem, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  // S^T: two accumulators of 64 columns (even and odd K steps), summed by
  // the softmax; O^T: 4 d-tiles x 64 columns
  const uint32_t s_col = 0, o_col = 128;

  // the top-k row into shared memory (unusable slots become -1), and which
  // tiles hold at least one usable index
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 2048 / kThreads; ++j) {
    const int i = tid + j * kThreads;
    if (i >= p.topk) break;
    int32_t s = idx_pre[j];
    if (s >= 0 && s < len) sm.tile_any[i / kRows] = 1;
    else {
      if (s >= len) bad = true;
      s = -1;
    }
    idx_s[i] = s;
  }
  if (bad) set_error(p.err, kErrIndex);
  __syncthreads();
  if (warp == 0) {
    // position of each tile in the query's list (window first, then the
    // top-k tiles holding a usable index); this CTA takes every splits-th
    const uint32_t any = __ballot_sync(0xffffffffu, lane < n_topk_tiles && sm.tile_any[lane] != 0);
    const int w = swa_count > 0 ? 1 : 0;
    const int n = w + __popc(any);
    if (lane == 0) {
      sm.n_tiles = (n - split + p.splits - 1) / p.splits;
      if (w && split == 0) sm.my_list[0] = -1;
    }
    if ((any >> lane) & 1u) {
      const int pos = w + __popc(any & ((1u << lane) - 1u));
      if (pos % p.splits == split) sm.my_list[pos / p.splits] = lane;
    }
  }
  __syncthreads();
  const int n_tiles = sm.n_tiles;

  // Candidate rows reach the KV buffer in two halves of four 64-channel
  // chunks (16 KB each), so that the next tile's first half is written while
  // the tensor core still reads the second half for O^T, and the first half
  // of S^T is computed while the second half is written.
  //
  // Fill mapping.  Warp 0 issues the MMAs (an issuing thread waits in the
  // issue for about one MMA time) and writes no rows, so its issues never
  // hold back the fill.  The other 15 warps (worker w = tid - 32) fill each
  // half: worker w owns entry 8 (w / 32) + w % 8 (entries 0..119) at chunk
  // quarter (w % 32) / 8, eight pieces of 8 channels; the 32 (entry,
  // quarter) pairs of entries 120..127 are spread as one extra piece over
  // the workers w < 256 (entry 120 + w / 32, quarter (w / 8) % 4, piece
  // w % 8).
  //
  // Gather of one top-k tile into registers: for each half h a worker loads
  // the 32 code bytes of its chunk 4 h + quarter (one 256-bit load, so each
  // 32-byte sector is requested once) and that chunk's scale bytes
  // (two UE8M0 or four E4M3), plus the code word and scale byte of its extra
  // piece.  Issued one tile ahead, so the loads are in flight while the
  // tensor core and the softmax work on the current tile.
  const bool filler = warp > 0;
  const int wkr = tid - 32;
  const int g_e = filler ? (wkr >> 5) * 8 + (lane & 7) : 0, g_q = lane >> 3;
  const bool has_x = filler && wkr < 256;
  const int x_e = 120 + (wkr >> 5), x_q = (wkr >> 3) & 3, x_k = wkr & 7;   // when has_x
  uint4 cw[4];
  uint32_t scw[2], xw[2], xsc[2];
  auto prefetch_tile = [&](int j) {
    if (!filler) return;
    const int32_t s = idx_s[j * kRows + g_e];
    if (s >= 0) {
      const int64_t row = base + s;
      const uint8_t* src = p.codes + row * kCodeBytes + g_q * 32;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ldg_now_v8(src + 128 * h, cw[2 * h], cw[2 * h + 1]);   // 32-byte aligned: 256 B rows
        if (p.layout == 0)
          scw[h] = ldg_now_u16(p.scales + row * 16 + 8 * h + 2 * g_q);
        else
          scw[h] = ldg_now_u32(p.scales + row * 32 + 16 * h + 4 * g_q);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) cw[i] = make_uint4(0u, 0u, 0u, 0u);
      scw[0] = scw[1] = 0u;
    }
    if (has_x) {
      const int32_t sx = idx_s[j * kRows + x_e];
      if (sx >= 0) {
        const int64_t row = base + sx;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          xw[h] = ldg_now_u32(p.codes + row * kCodeBytes + 128 * h + 32 * x_q + 4 * x_k);
          xsc[h] = (p.layout == 0) ? ldg_now_u8(p.scales + row * 16 + 8 * h + 2 * x_q + (x_k >> 2))
                                   : ldg_now_u8(p.scales + row * 32 + 16 * h + 4 * x_q + (x_k >> 1));
        }
      } else {
        xw[0] = xw[1] = xsc[0] = xsc[1] = 0u;
      }
    }
  };
  // the next top-k tile of this CTA's list after position `from`
  auto next_topk_after = [&](int from) {
    int j = from + 1;
    while (j < n_tiles && sm.my_list[j] < 0) ++j;
    return j;
  };
  // L2 prefetch of top-k tile j (one thread per entry: its two 128-byte
  // code lines and its scale line), a tile before the registers load it
  auto prefetch_l2 = [&](int j) {
    const int e = (filler && g_q == 0) ? g_e : (has_x && x_q == 0 && x_k == 0) ? x_e : -1;
    if (e < 0) return;
    const int32_t s = idx_s[j * kRows + e];
    if (s < 0) return;
    const int64_t row = base + s;
    const uint8_t* c = p.codes + row * kCodeBytes;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(c + 128));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.scales + row * (p.layout == 0 ? 16 : 32)));
  };

  // MMA descriptors: bases built once, K steps added to the address field
  // (all of shared memory is below 2^18 bytes, so the 14-bit field never
  // carries).  S^T = KV * Q^T: K-major A and B; O^T += KV^T * P^T: MN-major
  // A and B (P^T is stored one candidate row of 64 heads per 128 bytes, the
  // layout in which each thread writes its own row).
  const uint64_t d_skv = sdesc_sw128(smem_u32(kv), 16, 1024);
  const uint64_t d_sq = sdesc_sw128(smem_u32(qs), 16, 1024);
  const uint64_t d_okv = sdesc_sw128(smem_u32(kv), kRows * 128, 1024);
  const uint64_t d_op = sdesc_sw128(smem_u32(ps), kRows * 128, 1024);
  constexpr uint32_t id_s = idesc_bf16_f32(128, kHG, false, false);
  constexpr uint32_t id_o = idesc_bf16_f32(128, kHG, true, true);
  // S^T K step ks (channels 16 ks .. 16 ks + 15).  Consecutive steps go to
  // two accumulators in turn: an MMA into the accumulator that the previous
  // one still writes waits for it, one into the other does not.
  auto mma_s = [&](int ks) {
    const uint32_t ao = (uint32_t)((ks >> 2) * (kRows * 128) + (ks & 3) * 32);
    const uint32_t bo = (uint32_t)((ks >> 2) * (kHG * 128) + (ks & 3) * 32);
    umma_bf16(tmem + s_col + 64 * (ks & 1), d_skv + (ao >> 4), d_sq + (bo >> 4), id_s,
              ks > 1 ? 1u : 0u);
  };
  // O^T d-block i (reads KV chunks 2 i, 2 i + 1), K step ks (rows 16 ks ..);
  // issued with the two d-blocks of a half in turn, for the same reason
  auto mma_o = [&](int i, int ks, bool first) {
    const uint32_t ao = (uint32_t)((2 * i) * (kRows * 128) + ks * 2048);
    const uint32_t bo = (uint32_t)(ks * 2048);
    umma_bf16(tmem + o_col + 64 * i, d_okv + (ao >> 4), d_op + (bo >> 4), id_o,
              (!first || ks > 0) ? 1u : 0u);
  };

  // Half h of a tile's rows into the KV buffer (the workers; see the fill
  // mapping).  Top-k tiles come from the registers: E2M1 -> bf16 via byte
  // permutes and a bf16 scale multiply.  FP8 window rows come from global
  // memory: E4M3 x 2^scale is a bf16 value; the RoPE channels 448-511 are
  // bf16 already.  Written in the MMA layout (128-byte rows, 16-byte pieces
  // swizzled by row).
  auto piece_at = [&](int e, int c, int k) -> uint4* {
    return reinterpret_cast<uint4*>(kv + c * (kRows * 128) + e * 128 + ((k ^ (e & 7)) << 4));
  };
  auto scale_bf16x2 = [&](uint32_t byte) -> uint32_t {
    const float sc = (p.layout == 0) ? ue8m0_value(byte) : fabsf(e4m3_value(byte));
    const uint32_t s16 = float_to_bf16_bits(sc);
    return s16 | (s16 << 16);
  };
  auto e2m1_piece = [&](uint32_t word, uint32_t s2) -> uint4 {
    uint32_t v[4];
    e2m1x8_to_bf16x8(word, v);
    return make_uint4(bf16x2_mul(v[0], s2), bf16x2_mul(v[1], s2), bf16x2_mul(v[2], s2),
                      bf16x2_mul(v[3], s2));
  };
  // eight E4M3 codes (two words) x sc -> eight bf16
  auto e4m3_piece = [&](uint32_t w0, uint32_t w1, float sc) -> uint4 {
    const uint32_t w[2] = {w0, w1};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
            (__nv_fp8x2_storage_t)((w[i] >> (16 * k)) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const __nv_bfloat162 bb = __floats2bfloat162_rn(f.x * sc, f.y * sc);
        o[2 * i + k] = *reinterpret_cast<const uint32_t*>(&bb);
      }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  // window piece k of row e, chunk c (FP8 codes + scale, or RoPE bf16)
  auto window_piece = [&](int e, int c, int k) -> uint4 {
    const bool live = e < swa_count;
    if (!live) return make_uint4(0u, 0u, 0u, 0u);
    const int64_t row = (int64_t)swa_row0 + e;
    if (c == 7) return __ldg(reinterpret_cast<const uint4*>(ly.swa_rope + row * 64) + k);
    const float sc = ue8m0_value(__ldg(ly.swa_scales + row * 8 + c));
    const uint2 cc = __ldg(reinterpret_cast<const uint2*>(ly.swa_codes + row * 448 + 64 * c + 8 * k));
    return e4m3_piece(cc.x, cc.y, sc);
  };
  auto fill_half = [&](int tile, int h) {
    if (h == 0 && tid < kRows)
      sm.row_valid[tid] = tile >= 0 ? idx_s[tile * kRows + tid] >= 0 : tid < swa_count;
    const int c = 4 * h + g_q;                       // channel chunk of this worker
    if (tile >= 0) {
      if (filler) {
        const uint32_t words[8] = {cw[2 * h].x,     cw[2 * h].y,     cw[2 * h].z,     cw[2 * h].w,
                                   cw[2 * h + 1].x, cw[2 * h + 1].y, cw[2 * h + 1].z, cw[2 * h + 1].w};
        uint32_t s2[4];
        if (p.layout == 0) {                         // one UE8M0 scale per 32 channels
          s2[0] = s2[1] = scale_bf16x2(scw[h] & 0xFFu);
          s2[2] = s2[3] = scale_bf16x2((scw[h] >> 8) & 0xFFu);
        } else {                                     // one E4M3 scale per 16 channels
#pragma unroll
          for (int g = 0; g < 4; ++g) s2[g] = scale_bf16x2((scw[h] >> (8 * g)) & 0xFFu);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) *piece_at(g_e, c, k) = e2m1_piece(words[k], s2[k >> 1]);
      }
      if (has_x) *piece_at(x_e, 4 * h + x_q, x_k) = e2m1_piece(xw[h], scale_bf16x2(xsc[h]));
    } else {
      if (filler) {
#pragma unroll
        for (int k = 0; k < 8; ++k) *piece_at(g_e, c, k) = window_piece(g_e, c, k);
      }
      if (has_x) *piece_at(x_e, 4 * h + x_q, x_k) = window_piece(x_e, 4 * h + x_q, x_k);
    }
  };

  uint32_t ph_s = 0;   // parity of bar_mma (S^T done), once per tile
  bool ok = true;
  float lsum[16];      // partial sums of l: this thread's rows, heads 16 hh .. 16 hh + 15
#pragma unroll
  for (int i = 0; i < 16; ++i) lsum[i] = 0.0f;
  const int quad = warp & 3, hh = warp >> 2;   // TMEM lane quadrant, 16-head slice
  const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;


  // ---- first tile: rows -> KV buffer, then S^T
  int next_topk = next_topk_after(-1);
  if (n_tiles > 0) {
    const int tile = sm.my_list[0];
    if (next_topk < n_tiles) {
      prefetch_tile(sm.my_list[next_topk]);
      const int after = next_topk_after(next_topk);
      if (after < n_tiles) prefetch_l2(sm.my_list[after]);
    }
    if (tile < 0 && !ly.swa_codes) {
      // bf16 window rows: loaded by TMA at kernel entry
      if (tid < kRows) sm.row_valid[tid] = tid < swa_count;
      if (tid == 0) {
        for (int h = 0; h < 2; ++h) {
          ok = mbar_wait(&sm.bar_kv[h], 0, p.err, wl) && ok;
          ok = mbar_wait(&sm.bar_q[h], 0, p.err, wl) && ok;
          tc_fence_after();
          for (int k = 0; k < 16; ++k) mma_s(16 * h + k);
        }
        umma_commit(&sm.bar_mma);
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        fill_half(tile, h);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
          ok = mbar_wait(&sm.bar_q[h], 0, p.err, wl) && ok;
          tc_fence_after();
          for (int k = 0; k < 16; ++k) mma_s(16 * h + k);
          if (h == 1) umma_commit(&sm.bar_mma);
        }
      }
      if (tile >= 0) {
        next_topk = next_topk_after(next_topk);
        if (next_topk < n_tiles) {
          prefetch_tile(sm.my_list[next_topk]);
          const int after = next_topk_after(next_topk);
          if (after < n_tiles) prefetch_l2(sm.my_list[after]);
        }
      }
    }
  }

  for (int ti = 0; ti < n_tiles; ++ti) {
    // one thread polls the mbarrier, the others wait at the CTA barrier
    if (tid == 0) ok = mbar_wait(&sm.bar_mma, ph_s, p.err, wl) && ok;
    ph_s ^= 1;
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc_fence_after();

    // ------------------------------------------------ C: online softmax
    // Each thread holds one candidate row of S^T for 16 heads.  The running
    // maximum m of a head moves only when a tile holds a logit above it by
    // more than 2^8 (log2 units): then the tile maxima are reduced, m is
    // raised to them, and O^T and the partial sums are rescaled (exact: O,
    // l and the probabilities all refer to the same m, and probabilities
    // stay below 256).  Otherwise -- the common case after the first tile --
    // no reduction is needed at all.  Each thread keeps partial sums of l for
    // its 16 heads over the rows it has held; they are reduced once, after
    // the last tile.
    const int row = quad * 32 + lane;
    const bool valid = sm.row_valid[row] != 0;
    float x[16], mh[16];
    bool need = false;
    {
      uint32_t r[16], r2[16];
      tmem_ld16x2(tmem + lane_addr + s_col + 16 * hh, tmem + lane_addr + s_col + 64 + 16 * hh,
                  r, r2);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[i] = valid ? (__uint_as_float(r[i]) + __uint_as_float(r2[i])) * p.scale_log2
                     : -INFINITY;
        mh[i] = sm.m[16 * hh + i];
        need = need || x[i] > mh[i] + kLazyRescale;
      }
    }
    if (__syncthreads_or(need)) {
      {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = x[i];
        const float mx = warp_reduce_scatter16<true>(v, lane);
        if ((lane & 1) == 0) sm.red_max[quad][16 * hh + (lane >> 1)] = mx;
      }
      __syncthreads();
      if (tid < kHG) {
        const float tmax = fmaxf(fmaxf(sm.red_max[0][tid], sm.red_max[1][tid]),
                                 fmaxf(sm.red_max[2][tid], sm.red_max[3][tid]));
        const float mo = sm.m[tid];
        float a = 1.0f;
        if (tmax > mo + kLazyRescale) {
          a = (mo == -INFINITY) ? 0.0f : fast_exp2(mo - tmax);
          sm.m[tid] = tmax;
        }
        sm.alpha[tid] = a;
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        lsum[i] *= sm.alpha[16 * hh + i];
        mh[i] = sm.m[16 * hh + i];
      }
      if (ti > 0) {
        // O^T lanes are head-dim rows, columns are heads: scale column h by alpha[h]
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
          uint32_t r[16];
          const uint32_t ta = tmem + lane_addr + o_col + 64 * i + 16 * hh;
          tmem_ld16(ta, r);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            r[c] = __float_as_uint(__uint_as_float(r[c]) * sm.alpha[16 * hh + c]);
          tmem_st16(ta, r);
        }
        tmem_wait_st();
      }
    }
    {
      // P^T as the MN-major B operand: this thread's candidate row holds its
      // 16 heads in two 16-byte pieces (8 heads each), swizzled by the row
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p0 = (x[2 * i] == -INFINITY) ? 0.0f : fast_exp2(x[2 * i] - mh[2 * i]);
        const float p1 =
            (x[2 * i + 1] == -INFINITY) ? 0.0f : fast_exp2(x[2 * i + 1] - mh[2 * i + 1]);
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);   // .x: head 2i (low half)
        pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
        lsum[2 * i] += __uint_as_float(pk[i] << 16);
        lsum[2 * i + 1] += __uint_as_float(pk[i] & 0xFFFF0000u);
      }
      uint8_t* prow = ps + row * 128;
      *reinterpret_cast<uint4*>(prow + (((2 * hh) ^ (row & 7)) << 4)) =
          make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(prow + (((2 * hh + 1) ^ (row & 7)) << 4)) =
          make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ------------------------------------------------ O^T += KV^T * P^T, next tile
    const bool first = ti == 0;
    const uint32_t ph_o = (uint32_t)(ti & 1);
    if (tid == 0) {
      tc_fence_after();
      for (int k = 0; k < 16; ++k) mma_o(k & 1, k >> 1, first);
      umma_commit(&sm.bar_o[0]);
      for (int k = 0; k < 16; ++k) mma_o(2 + (k & 1), k >> 1, first);
      umma_commit(&sm.bar_o[1]);
    }
    if (ti + 1 < n_tiles) {
      // The next tile (always a top-k tile: the window comes first) replaces
      // the KV buffer half by half: half 0 once O^T d-blocks 0-1 are done
      // (while blocks 2-3 run), half 1 once blocks 2-3 are done (while S^T of
      // half 0 runs).
      const int tile = sm.my_list[ti + 1];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ok = mbar_wait(&sm.bar_o[h], ph_o, p.err, wl) && ok;
        tc_fence_after();
        fill_half(tile, h);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
          tc_fence_after();
          for (int k = 0; k < 16; ++k) mma_s(16 * h + k);
          if (h == 1) umma_commit(&sm.bar_mma);
        }
      }
      next_topk = next_topk_after(next_topk);
      if (next_topk < n_tiles) {
        prefetch_tile(sm.my_list[next_topk]);
        const int after = next_topk_after(next_topk);
        if (after < n_tiles) prefetch_l2(sm.my_list[after]);
      }
    } else {
      if (tid == 0) ok = mbar_wait(&sm.bar_o[1], ph_o, p.err, wl) && ok;
      ok = __syncthreads_and(ok);
      tc_fence_after();
    }
  }

  // l of each head: the partial sums reduced over all rows
  {
    const float sum = warp_reduce_scatter16<false>(lsum, lane);
    if ((lane & 1) == 0) sm.red_sum[quad][16 * hh + (lane >> 1)] = sum;
  }
  __syncthreads();
  if (tid < kHG)
    sm.l[tid] = (sm.red_sum[0][tid] + sm.red_sum[1][tid]) + (sm.red_sum[2][tid] + sm.red_sum[3][tid]);
  __syncthreads();
  // ------------------------------------------------ epilogue
  // Variants of the blog reading of the DeepSeek-V4 report, section 4.3: a
  // per-head sink logit z' whose exp joins the softmax denominator (the sink
  // has no value), and RoPE at position -i on the last 64 output channels
  // (interleaved pairs, frequency base^(-2t/64)), applied before the bf16
  // cast.  The angle -i * theta_t (positions reach 2^20) is formed and
  // reduced modulo 2 pi in fp64, then its sine and cosine are taken in fp32.
  const bool rope = p.rope_out != 0;
  if (rope && tid < 32) {
    const double pos = p.prefill ? (double)(p.pos0 + q) : (double)p.rope_pos[q];
    const double phi = -pos * p.rope_theta[tid];
    const double turns = rint(phi * 0.15915494309189535);       // 1 / (2 pi)
    const float r = (float)fma(-turns, 6.283185307179586, phi);  // in [-pi, pi]
    float sn, cs;
    sincosf(r, &sn, &cs);
    sm.rope_c[tid] = cs;
    sm.rope_s[tid] = sn;
  }
  __syncthreads();
  const int64_t out_row = (int64_t)q * p.n_heads + hg * kHG;   // first head of this CTA
  // sink logit of head h in log2 units (-inf: none)
  auto sink_log2 = [&](int h) -> float {
    return ly.sink ? ly.sink[hg * kHG + h] * 1.4426950408889634f : -INFINITY;
  };
  // output channel d of head slot c, rotated when it is a RoPE channel
  // (channel pairs sit in adjacent lanes: every lane of the warp calls this)
  auto finish = [&](int i, float o) -> float {
    if (rope && i == 3 && quad >= 2) {
      const float other = __shfl_xor_sync(0xffffffffu, o, 1);
      const int t = ((quad - 2) * 32 + lane) >> 1;
      const float cs = sm.rope_c[t], sn = sm.rope_s[t];
      o = (lane & 1) ? fmaf(other, sn, o * cs) : fmaf(-other, sn, o * cs);
    }
    return o;
  };
  // Output rows go through shared memory: bf16 [64 heads][dw] in the Q
  // buffer (free after the last S product), then 16-byte stores of each
  // head's d range [d0, d0 + dw).
  uint16_t* out_s = reinterpret_cast<uint16_t*>(qs);   // free after the last S^T
  auto store_rows = [&](int d0, int dw) {
    const int per_row = dw / 8;
    for (int k = tid; k < kHG * per_row; k += kThreads) {
      const int h = k / per_row, c = k % per_row;
      *reinterpret_cast<uint4*>(ly.out + (out_row + h) * kHeadDim + d0 + 8 * c) =
          *reinterpret_cast<const uint4*>(out_s + h * dw + 8 * c);
    }
  };
  const bool have = ok && n_tiles > 0;
  if (p.splits == 1) {
    if (have) {
      if (tid < kHG) {
        const float l = sm.l[tid], m = sm.m[tid], z = sink_log2(tid);
        const float M = fmaxf(m, z);
        const float am = (m == -INFINITY) ? 0.0f : fast_exp2(m - M);
        const float L = l * am + ((z == -INFINITY) ? 0.0f : fast_exp2(z - M));
        sm.alpha[tid] = L > 0.0f ? am / L : 0.0f;
        if (ly.lse)
          ly.lse[out_row + tid] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      }
      __syncthreads();
      float w_me[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) w_me[c] = sm.alpha[16 * hh + c];
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_addr + o_col + 64 * i + 16 * hh, r);
        const int d = 128 * i + quad * 32 + lane;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float o = finish(i, __uint_as_float(r[c]) * w_me[c]);
          out_s[(16 * hh + c) * kHeadDim + d] = (uint16_t)float_to_bf16_bits(o);
        }
      }
      __syncthreads();
      store_rows(0, kHeadDim);
    } else if (n_tiles == 0) {
      // no candidate at all: output 0, lse = the sink alone (or -inf)
      for (int i = tid; i < kHG * kHeadDim; i += kThreads) ly.out[out_row * kHeadDim + i] = 0;
      if (ly.lse && tid < kHG)
        ly.lse[out_row + tid] = ly.sink ? ly.sink[hg * kHG + tid] : -INFINITY;
    }
  } else {
    // ---- split-KV over a cluster of two CTAs (cluster rank = split).  Each
    //      stages, in its free KV buffer, its unnormalised O^T for the d half
    //      that the partner finalises; after a cluster barrier each finalises
    //      its own half d in [256 split, 256 split + 256) from its TMEM and
    //      the partner's staged copy, with the partner's (m, l) read through
    //      distributed shared memory:
    //        out = (a0 * O_0 + a1 * O_1) / (a0 * l0 + a1 * l1),
    //      operands in split order.  Staging layout [half][warp][4][lane][4
    //      floats]: a warp's 16-byte accesses are contiguous.
    const uint32_t peer = (uint32_t)(split ^ 1);
    float* stage = reinterpret_cast<float*>(kv);
    if (tid < kHG && !have) { sm.m[tid] = -INFINITY; sm.l[tid] = 0.0f; }
    if (have) {
#pragma unroll 1
      for (int ii = 0; ii < 2; ++ii) {
        const int i = 2 * (int)peer + ii;
        uint32_t r[16];
        tmem_ld16(tmem + lane_addr + o_col + 64 * i + 16 * hh, r);
        float4* dst = reinterpret_cast<float4*>(stage) + ((ii * 16 + warp) * 4) * 32 + lane;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[32 * v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                    __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      }
    }
    cluster_arrive();
    cluster_wait();
    if (tid < kHG) {
      const float m_ot = ld_dsmem_f32(dsmem_addr(smem_u32(&sm.m[tid]), peer));
      const float l_ot = ld_dsmem_f32(dsmem_addr(smem_u32(&sm.l[tid]), peer));
      const float m_me = sm.m[tid], l_me = sm.l[tid];
      const float m0 = split == 0 ? m_me : m_ot, m1 = split == 0 ? m_ot : m_me;
      const float l0 = split == 0 ? l_me : l_ot, l1 = split == 0 ? l_ot : l_me;
      const float z = sink_log2(tid);
      const float M = fmaxf(fmaxf(m0, m1), z);
      const float a0 = (m0 == -INFINITY) ? 0.0f : fast_exp2(m0 - M);
      const float a1 = (m1 == -INFINITY) ? 0.0f : fast_exp2(m1 - M);
      const float L = a0 * l0 + a1 * l1 + ((z == -INFINITY) ? 0.0f : fast_exp2(z - M));
      const float c_me = L > 0.0f ? (split == 0 ? a0 : a1) / L : 0.0f;
      const float c_ot = L > 0.0f ? (split == 0 ? a1 : a0) / L : 0.0f;
      sm.alpha[tid] = have ? c_me : 0.0f;               // weight of this CTA's O
      sm.red_max[0][tid] = (l_ot > 0.0f) ? c_ot : 0.0f;  // weight of the partner's O
      if (ly.lse && split == 0)
        ly.lse[out_row + tid] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    __syncthreads();
    // this CTA's O^T first (warp-collective TMEM loads), then all eight
    // 16-byte reads of the partner's staged half in flight at once, with no
    // warp-synchronising instruction until they are used
    uint32_t ro[2][16];
    if (have) {
      tmem_ld16(tmem + lane_addr + o_col + 64 * (2 * split) + 16 * hh, ro[0]);
      tmem_ld16(tmem + lane_addr + o_col + 64 * (2 * split + 1) + 16 * hh, ro[1]);
    }
    float w_me[16], w_pt[16];   // the weights of this thread's 16 heads, read once
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      w_me[c] = sm.alpha[16 * hh + c];
      w_pt[c] = sm.red_max[0][16 * hh + c];
    }
    const uint32_t peer_stage = dsmem_addr(smem_u32(stage), peer);
    float4 pv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      pv[k] = ld_dsmem_v4(peer_stage +
                          (uint32_t)(((((k >> 2) * 16 + warp) * 4 + (k & 3)) * 32 + lane) * 16));
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const int i = 2 * split + ii;
      const int d = 128 * i + quad * 32 + lane;
      const float po[16] = {pv[4 * ii].x,     pv[4 * ii].y,     pv[4 * ii].z,     pv[4 * ii].w,
                            pv[4 * ii + 1].x, pv[4 * ii + 1].y, pv[4 * ii + 1].z, pv[4 * ii + 1].w,
                            pv[4 * ii + 2].x, pv[4 * ii + 2].y, pv[4 * ii + 2].z, pv[4 * ii + 2].w,
                            pv[4 * ii + 3].x, pv[4 * ii + 3].y, pv[4 * ii + 3].z, pv[4 * ii + 3].w};
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int h = 16 * hh + c;
        const float o_me = have ? w_me[c] * __uint_as_float(ro[ii][c]) : 0.0f;
        const float o_ot = w_pt[c] != 0.0f ? w_pt[c] * po[c] : 0.0f;
        // fixed order: split 0's term first
        const float o = finish(i, split == 0 ? o_me + o_ot : o_ot + o_me);
        out_s[h * 256 + (d - 256 * split)] = (uint16_t)float_to_bf16_bits(o);
      }
    }
    // the partner's shared memory is read no more: it may exit once it waits
    cluster_arrive();
    __syncthreads();
    store_rows(256 * split, 256);
    cluster_wait();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int attn_smem_bytes() { return kSmemBytes; }
cudaError_t launch_attn(const AttnParams& p, const AttnMaps& maps, cudaStream_t s) {
  if (p.n_layers < 1 || p.n_layers > kAttnMaxLayers) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k_attn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.n_layers * p.nq * (p.n_heads / kHG) * p.splits;
  if (blocks <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2] = {pdl_attribute(), {}};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.splits == 2) {
    // the two CTAs of a (query, head group) form a cluster
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, k_attn, p, maps);
}

}  // namespace csa2
