// csa2_kernels.h -- host-side launch interface between the C ABI layer
// (csa2_api.cu) and the kernel translation units.  Internal to the library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace csa2 {

// Sticky device error word bits (see csa2_get_device_error).
constexpr uint32_t kErrTimeoutBit = 1u;
constexpr uint32_t kErrIndexBit = 2u;

// Launch attribute: programmatic stream serialisation (the kernel's launch
// overlaps the end of the previous kernel in the stream; the kernel waits for
// it with griddepcontrol.wait before its first global memory access).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

constexpr int kHeadDim = 512;     // main-KV latent / attention head dim
constexpr int kIdxDim = 128;      // indexer head dim
constexpr int kIdxHeads = 32;     // indexer heads
constexpr int kCodeBytes = kHeadDim / 2;
constexpr int kKeyHistBinsHost = 2048;   // score-key histogram bins (top 11 key bits)

// ---------------------------------------------------------------- append
constexpr int kMaxAppendSegs = 64;
struct AppendSeg {
  int64_t first;     // first output row of this segment within the launch
  int64_t src_row;   // first input entry row (entries mode) or entry-block row
  int64_t dst_row;   // first cache row
  int32_t seq;
  int32_t new_len;   // sequence length after the append
};
struct AppendParams {
  int32_t mode;      // 0 compress only, 1 append entries, 2 append tokens
  int32_t ratio;
  int32_t layout;    // 0 = L32_UE8M0, 1 = L16_E4M3
  int32_t dim;       // channels (compress-only may differ from kHeadDim)
  int32_t n_segs;
  int64_t rows;      // output rows in this launch
  AppendSeg seg[kMaxAppendSegs];
  const float* entries;
  const uint16_t* c_tok;
  const float* z_tok;
  const uint16_t* idx_k;
  float* entries_out;
  uint8_t* codes;
  uint8_t* scales;
  uint16_t* cache_idxk;
  int32_t idx_mxfp4;         // 1: indexer keys quantised to MXFP4 (codes + scales below)
  uint8_t* idx_codes;
  uint8_t* idx_scales;
  int32_t* d_len;
  int64_t total;             // cache rows (bounds checks of the debug build)
  uint32_t* err;             // nullable device error word
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);

// ---------------------------------------------------------------- indexer
constexpr int kMaxIdxGroups = 1024;
// Fault injection for tests of the timeout path: the indexer's producer
// issues no key loads, so the MMA and epilogue waits run out with nothing in
// flight (no copy, no MMA).
constexpr int32_t kInjectNoKeyLoads = 1;
struct IndexParams {
  const float* w;          // [nq, 32]
  float* scores;           // [nq, ld]
  int64_t ld;
  uint32_t* key_hist;      // nullable [nq, 2048] score-key histogram (qpg == 1 only)
  int32_t score_bf16;      // 1: scores are stored as bf16 (uint16 [nq, ld], nearest even)
  const uint16_t* q_idx;     // MXFP4 keys (k_index_fp4): bf16 queries [nq, 32, 128]
  const uint8_t* idx_codes;  // MXFP4 keys (k_index_fp4): E2M1 codes [idx_total, 64]
  const uint8_t* idx_scales; // MXFP4 keys: UE8M0 scales [idx_total, 4]
  int64_t idx_total;         // MXFP4 keys: rows in the cache
  const int32_t* pool;     // nullable: pool mode, [nq, pool_blocks] block ids (-1 unused)
  int32_t pool_blocks;     // blocks per pool row (multiple of 16)
  uint32_t* err;
  int32_t nq;
  int32_t qpg;             // queries per group (1 decode, 8 prefill; MXFP4 keys: 4)
  int32_t n_groups;
  int32_t prefill;         // 1: visibility from positions
  int64_t pre_base;        // prefill: entry offset of the sequence
  int64_t pos0;            // prefill: position of query 0
  int32_t pre_len;         // prefill: entries in the sequence
  int32_t ratio;
  int64_t wait_cycles;     // bounded-wait limit in cycles (0: the default, ~2^31)
  int32_t inject;          // kInjectNoKeyLoads: the producer issues no key loads (tests)
  int32_t tile_prefix[kMaxIdxGroups + 1];  // cumulative tiles per group (128 entries; the
                                           // MXFP4 kernel: 256 for one query per group)
  int64_t entry_base[kMaxIdxGroups];       // decode: entry offset of the group's sequence
  int32_t nvis[kMaxIdxGroups];             // decode: visible entries of the group's query
};
int index_smem_bytes(int qpg);
cudaError_t launch_index(const IndexParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_q,
                         int grid, cudaStream_t s);
// MXFP4 keys (codes [idx_rows, 64], scales [idx_rows, 4], idx_rows a
// multiple of 512): tm_kq views the codes as aligned 128-key tiles in the
// permuted row order of the kernel (key 4 r + q of a tile in shared-memory
// row 32 q + r, 64-byte rows, 64-byte swizzle), tm_kc8 as [idx_total, 64]
// in boxes of 8 rows (pool blocks, 64-byte swizzle).  qpg is 1 (decode,
// pool mode) or 4 (prefill).  Decode tiles (no pool) are the aligned 512-key
// chunks: a sequence at key row off has ceil((n + off % 512) / 512) tiles;
// prefill tiles the aligned 128-key chunks, ceil((n + off % 128) / 128) per
// group.
int index_fp4_smem_bytes();
cudaError_t launch_index_fp4(const IndexParams& p, const CUtensorMap& tm_kq,
                             const CUtensorMap& tm_kc8, int grid, cudaStream_t s);

// ---------------------------------------------------------------- HSI
constexpr int kHsiBlock = 8;   // positions per block of the candidate pool
struct HsiParams {
  int32_t rows;              // <= kHsiTab
  // block max: bmax[r, b] = max of scores[r, 8 b .. 8 b + 7] over the row's
  // n[r] positions, for b < ceil(n[r] / 8)
  const float* scores;
  int64_t ld;
  float* bmax;
  int64_t ld_b;
  // pool map: out[r, j] = pool[r, s / 8] * 8 + s % 8 for s = sel[r, j];
  // -1 for unused slots and for entries >= n[r]
  const int32_t* sel;
  int32_t k;
  const int32_t* pool;
  int32_t pool_blocks;
  int32_t* out;
  float* score_out;          // nullable: zeroed where out is -1
  uint32_t* err;             // nullable device error word (debug-build checks)
  int64_t n[1024];
};
constexpr int kHsiTab = 1024;
cudaError_t launch_block_max(const HsiParams& p, cudaStream_t s);
cudaError_t launch_pool_map(const HsiParams& p, cudaStream_t s);

// ---------------------------------------------------------------- top-k
constexpr int kTopkMaxRowsPerLaunch = 65535;
constexpr int kTopkTab = 1024;
struct TopkParams {
  const float* scores;       // row r at scores + r * ld
  int64_t ld;
  int32_t rows;
  int32_t k;
  const uint32_t* key_hist;  // nullable [rows, 2048] score-key histogram
  int32_t* idx_out;          // [rows, k]
  float* score_out;          // nullable [rows, k]
  int32_t formula;           // 1: n_valid(r) = min(len, (pos0 + r + 1) / ratio)
  int32_t pre_len;
  int32_t ratio;
  int64_t pos0;
  int32_t score_bf16;        // 1: scores are bf16 (uint16 [rows, ld])
  uint32_t* seg_ws;          // nullable: per-segment candidate buffers (see topk_seg_bytes)
  int32_t n_seg;             // segments per row when seg_ws is set
  uint32_t* err;             // nullable device error word (debug-build checks)
  int64_t n_valid[kTopkTab]; // formula == 0: per-row valid counts
};
// Segmented candidate compaction (rows with a score-key histogram): scratch
// bytes for `rows` rows of up to `max_valid` scores, and its segment count.
constexpr int kTopkSegLen = 8192;
int topk_segments(int64_t max_valid);
size_t topk_seg_bytes(int32_t rows, int64_t max_valid);
cudaError_t launch_topk(const TopkParams& p, cudaStream_t s);

// ---------------------------------------------------------------- attention
constexpr int kAttnTab = 1024;
constexpr int kAttnMaxLayers = 8;
// What differs between the layers of one readout launch (the layers of a
// group share the cache, the selection and the windows' geometry).
struct AttnLayer {
  uint16_t* out;             // bf16 [nq, n_heads, 512]
  float* lse;                // nullable [nq, n_heads]
  const float* sink;         // nullable [n_heads]: per-head sink logit z' (units of scale * q.kv)
  const uint8_t* swa_codes;  // FP8 window rows (nullable): E4M3 codes [rows, 448]
  const uint16_t* swa_rope;  //   bf16 RoPE channels [rows, 64]
  const uint8_t* swa_scales; //   UE8M0 scales [rows, 8]
};
// The layers' query rows and bf16 window rows as TMA tensor maps.
struct AttnMaps {
  CUtensorMap q[kAttnMaxLayers];
  CUtensorMap swa[kAttnMaxLayers];
};
struct AttnParams {
  const int32_t* topk_idx;   // [nq, topk]
  const int32_t* swa_len;    // decode: nullable [nq]
  const uint8_t* codes;
  const uint8_t* scales;
  int32_t n_layers;          // layers of the launch; blocks are (layer, query, head group, split)
  int32_t splits;            // CTAs per (query, 64-head group): 1, or 2 (a cluster)
  uint32_t* err;
  int32_t nq;
  int32_t n_heads;
  int32_t topk;
  int32_t swa;               // window size W
  int32_t layout;
  float scale_log2;          // scale * log2(e)
  float scale;
  int32_t prefill;
  int64_t pre_base;          // prefill: entry offset of the sequence
  int32_t pre_len;           // prefill: entries in the sequence
  int64_t pos0;              // prefill: position of query 0
  int64_t swa_pos0;          // prefill: position of swa row 0
  const int64_t* rope_pos;   // decode: [nq] query positions for the output RoPE(-i)
  int32_t rope_out;          // 1: rotate the last 64 output channels by -position
  double rope_theta[32];     // RoPE frequencies base^(-2t/64) of the 32 channel pairs
  int64_t wait_cycles;       // bounded-wait limit in cycles (0: the default, ~2^31)
  AttnLayer layer[kAttnMaxLayers];
  int64_t q_base[kAttnTab];  // decode: entry offset of each query's sequence
  int32_t q_len[kAttnTab];   // decode: entries of each query's sequence
};
cudaError_t launch_swa_fp8(const uint16_t* rows, int64_t n, uint8_t* codes, uint16_t* rope,
                           uint8_t* scales, cudaStream_t s);
int attn_smem_bytes();
constexpr int kAttnHeadGroup = 64;
// The two-CTA decode split needs no scratch memory: a caller opts in by
// passing a workspace of at least this many bytes.
constexpr size_t kAttnSplitToken = 16;
cudaError_t launch_attn(const AttnParams& p, const AttnMaps& maps, cudaStream_t s);

}  // namespace csa2
