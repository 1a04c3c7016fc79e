// csa2_api.cu -- the C ABI declared in include/csa2.h: argument checks, the
// cache layout in caller memory, TMA tensor maps, and launch scheduling of
// the kernels in k_append.cu, k_index.cu, k_topk.cu and k_attn.cu.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "csa2.h"
#include "csa2_kernels.h"

namespace {
// One NVTX range per C call, named after the call (shows in Nsight
// timelines; without an attached tool the push and pop return at once).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace
#define CSA2_RANGE() NvtxRange csa2_nvtx_range_(__func__)

// Scratch of csa2_index_topk_decode_static, for callers that cannot allocate:
// a fixed array in the library's device image (one per GPU that loads it).
static __device__ __align__(256) uint8_t g_static_scratch[CSA2_STATIC_SCRATCH_BYTES];

using namespace csa2;

struct csa2_cache {
  csa2_config_t cfg;
  int32_t batch;
  int32_t group;       // channels per scale
  int32_t scale_bytes; // per entry
  std::vector<int64_t> cap, off, len;
  int64_t total;
  int64_t max_cap;
  uint8_t* base;
  size_t bytes;
  int32_t* d_len;
  uint32_t* d_err;
  uint8_t* codes;
  uint8_t* scales;
  uint16_t* idxk;       // CSA2_IDX_BF16 keys
  uint8_t* idx_codes;   // CSA2_IDX_MXFP4 keys: codes [idx_rows, 64], scales [idx_rows, 4]
  uint8_t* idx_scales;
  int64_t idx_rows;     // total rounded up to whole 512-key chunks (MXFP4 keys)
  CUtensorMap tm_k;    // indexer keys, 128-row boxes (contiguous tiles)
  CUtensorMap tm_k8;   // indexer keys, one 8-key block per box (pool mode)
  CUtensorMap tm_kq;   // MXFP4 key codes, 128-key tiles in the permuted row order
  CUtensorMap tm_kc8;  // MXFP4 key codes, one 8-key block per box (pool mode)
  int num_sms;
  int index_sms;       // SMs the indexer's persistent grid may occupy
  int64_t wait_cycles; // bounded-wait limit of the kernels (0: their default)
  int32_t inject;      // fault injection for tests (kInjectNoKeyLoads)
};

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa2_status_t check_cfg(const csa2_config_t* c) {
  if (!c) return CSA2_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->idx_dim != kIdxDim || c->idx_heads != kIdxHeads)
    return CSA2_ERR_UNSUPPORTED;
  if (c->n_heads <= 0 || c->n_heads % kAttnHeadGroup != 0 || c->n_heads > 128)
    return CSA2_ERR_UNSUPPORTED;
  if (c->topk <= 0 || c->topk % 128 != 0 || c->topk > 2048) return CSA2_ERR_UNSUPPORTED;
  if (c->swa < 0 || c->swa > 128) return CSA2_ERR_UNSUPPORTED;
  if (c->ratio < 1 || c->ratio > 16) return CSA2_ERR_UNSUPPORTED;
  if (c->layout != CSA2_KV_L32_UE8M0 && c->layout != CSA2_KV_L16_E4M3) return CSA2_ERR_UNSUPPORTED;
  if (c->idx_layout != CSA2_IDX_BF16 && c->idx_layout != CSA2_IDX_MXFP4) return CSA2_ERR_UNSUPPORTED;
  return CSA2_OK;
}

struct Layout {
  size_t len_off, err_off, codes_off, scales_off, idxk_off, idxs_off, total;
};

static_assert(CSA2_MAX_ATTN_LAYERS == kAttnMaxLayers, "layers of one readout launch");

// Rows of the MXFP4 key arrays: the entries rounded up to 512-key chunks.
int64_t mxfp4_rows(int64_t total) { return (total + 511) / 512 * 512; }

Layout layout_for(const csa2_config_t* c, int64_t total) {
  Layout L;
  const int g = c->layout == CSA2_KV_L16_E4M3 ? 16 : 32;
  L.len_off = 0;
  L.err_off = 0;  // filled below
  L.codes_off = 0;
  size_t o = 0;
  L.len_off = o;
  o = align_up(o + 4096 * sizeof(int32_t), kAlign);  // up to 4096 sequences of lengths
  L.err_off = o;
  o = align_up(o + sizeof(uint32_t), kAlign);
  L.codes_off = o;
  o = align_up(o + (size_t)total * (kHeadDim / 2), kAlign);
  L.scales_off = o;
  o = align_up(o + (size_t)total * (kHeadDim / g), kAlign);
  L.idxk_off = o;
  if (c->idx_layout == CSA2_IDX_MXFP4) {
    // E2M1 codes and UE8M0 scales, each holding whole 512-key chunks (the
    // indexer reads keys in aligned tiles of up to 512 keys; rows past
    // `total` are never valid entries)
    const size_t rows = (size_t)mxfp4_rows(total);
    o = align_up(o + rows * (kIdxDim / 2), kAlign);
    L.idxs_off = o;
    o = align_up(o + rows * (kIdxDim / 32), kAlign);
  } else {
    o = align_up(o + (size_t)total * kIdxDim * 2, kAlign);
    L.idxs_off = 0;
  }
  L.total = o;
  return L;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows, cols] (row stride cols * 2 bytes), 128B-swizzled
// boxes of [box_rows, box_cols]; out-of-range rows read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
              uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t gdim[2] = {cols, rows};
  cuuint64_t gstride[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP4 key codes as bytes [rows, row_bytes] (64: one key per row, 64-byte
// swizzle; 128: two keys per row, 128-byte swizzle), boxes of box_rows rows:
// the K-major layouts of the block-scaled MMA's operands.
bool make_code_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t row_bytes,
                   uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t gdim[2] = {row_bytes, rows};
  cuuint64_t gstride[1] = {row_bytes};
  cuuint32_t box[2] = {row_bytes, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP4 key codes in aligned 128-key tiles with their rows permuted: key
// 4 r + q of a tile (r < 32, q < 4) lands in shared-memory row 32 q + r (64-
// byte rows, the 64-byte swizzle).  With the keys in that order, the tile's
// UE8M0 scale words in their natural order are exactly the scale atom of
// the block-scaled MMA (row 32 q + r at byte 16 r + 4 q), so a tile's scales
// are one contiguous copy.  The view is (64 bytes, r, q, tile) with strides
// (1, 256, 64, 8192); rows must be a multiple of 128.  (The box's rows are
// exactly one swizzle span wide: with a wider swizzle than the row, the TMA
// would lay each row out at the swizzle span.)
bool make_perm_map(CUtensorMap* m, const void* base, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0 || rows % 128 != 0) return false;
  cuuint64_t gdim[4] = {64, 32, 4, (cuuint64_t)(rows / 128)};
  cuuint64_t gstride[3] = {256, 64, 8192};
  cuuint32_t box[4] = {64, 32, 4, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), gdim, gstride, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Indexer keys [rows, 128] bf16 seen as (64 columns, rows, 2 halves): one
// box of (64, 8, 2) is a whole block of 8 keys, landing in shared memory as
// two 1 KB 128B-swizzled atoms (columns 0-63, then 64-127).
bool make_block_map(CUtensorMap* m, const void* base, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t gdim[3] = {64, rows, 2};
  cuuint64_t gstride[2] = {kIdxDim * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)kHsiBlock, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaStream_t S(csa2_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

csa2_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

int64_t score_ld(int64_t n) { return std::max<int64_t>(4, (n + 3) / 4 * 4); }

// The indexer kernel for the cache's key storage: bf16 keys (TMA, kind::f16
// MMAs), or MXFP4 keys (E2M1 codes by TMA, block-scaled kind::mxf4 MMAs,
// queries rounded to MXFP4 on chip from q_idx).  `pool` selects the
// pool-mode tensor map of bf16 keys.
cudaError_t launch_index_any(const csa2_cache* c, IndexParams& ip, const CUtensorMap& tm_q,
                             const void* q_idx, int grid, cudaStream_t s, bool pool = false) {
  if (c->cfg.idx_layout == CSA2_IDX_MXFP4) {
    ip.idx_codes = c->idx_codes;
    ip.idx_scales = c->idx_scales;
    ip.idx_total = c->total;
    ip.q_idx = static_cast<const uint16_t*>(q_idx);
    return launch_index_fp4(ip, c->tm_kq, c->tm_kc8, grid, s);
  }
  return launch_index(ip, pool ? c->tm_k8 : c->tm_k, tm_q, grid, s);
}

// Append / compress segments: rows of one launch grouped by sequence.
csa2_status_t run_append(csa2_cache* c, int mode, int32_t n_seqs, const int32_t* seq_ids,
                         const int32_t* n_rows_in, const float* entries, const void* c_tok,
                         const float* z_tok, const void* idx_k, float* entries_out,
                         csa2_stream_t stream) {
  if (!c || n_seqs < 0 || (n_seqs > 0 && (!seq_ids || !n_rows_in))) return CSA2_ERR_INVALID_ARG;
  const int m = c->cfg.ratio;
  std::vector<int64_t> new_len(c->len);
  int64_t total_rows = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const int32_t s = seq_ids[i];
    const int32_t n = n_rows_in[i];
    if (s < 0 || s >= c->batch || n < 0) return CSA2_ERR_INVALID_ARG;
    if (mode == 2 && n % m != 0) return CSA2_ERR_INVALID_ARG;
    const int64_t ne = mode == 2 ? n / m : n;
    new_len[s] += ne;
    if (new_len[s] > c->cap[s]) return CSA2_ERR_CAPACITY;
    total_rows += ne;
  }
  if (total_rows == 0) return CSA2_OK;
  if (!idx_k || !aligned16(idx_k)) return CSA2_ERR_INVALID_ARG;
  if (mode == 1 && (!entries || !aligned16(entries))) return CSA2_ERR_INVALID_ARG;
  if (mode == 2 && (!c_tok || !z_tok || !aligned16(c_tok) || !aligned16(z_tok)))
    return CSA2_ERR_INVALID_ARG;
  if (entries_out && !aligned16(entries_out)) return CSA2_ERR_INVALID_ARG;

  std::vector<int64_t> cur(c->len);
  int64_t src = 0;
  int i = 0;
  while (i < n_seqs) {
    AppendParams p;
    std::memset(&p, 0, sizeof(p));
    p.mode = mode;
    p.ratio = m;
    p.layout = c->cfg.layout;
    p.dim = kHeadDim;
    p.entries = entries;
    p.c_tok = static_cast<const uint16_t*>(c_tok);
    p.z_tok = z_tok;
    p.idx_k = static_cast<const uint16_t*>(idx_k);
    p.entries_out = entries_out;
    p.codes = c->codes;
    p.scales = c->scales;
    p.cache_idxk = c->idxk;
    p.idx_mxfp4 = c->cfg.idx_layout == CSA2_IDX_MXFP4 ? 1 : 0;
    p.idx_codes = c->idx_codes;
    p.idx_scales = c->idx_scales;
    p.d_len = c->d_len;
    p.total = c->total;
    p.err = c->d_err;
    int64_t rows = 0;
    while (i < n_seqs && p.n_segs < kMaxAppendSegs) {
      const int32_t s = seq_ids[i];
      const int64_t ne = mode == 2 ? n_rows_in[i] / m : n_rows_in[i];
      AppendSeg& g = p.seg[p.n_segs++];
      g.first = rows;
      g.src_row = src;
      g.dst_row = c->off[s] + cur[s];
      g.seq = s;
      cur[s] += ne;
      g.new_len = (int32_t)cur[s];
      rows += ne;
      src += ne;
      ++i;
    }
    p.rows = rows;
    cudaError_t e = launch_append(p, S(stream));
    if (e != cudaSuccess) return CSA2_ERR_CUDA;
  }
  c->len = new_len;
  return CSA2_OK;
}

}  // namespace

extern "C" {

int32_t csa2_version(void) { return 1; }

const char* csa2_status_string(csa2_status_t s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSA2_ERR_CAPACITY: return "capacity exceeded";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_OOM: return "out of memory";
    case CSA2_ERR_TIMEOUT: return "device wait timed out";
    case CSA2_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

size_t csa2_cache_bytes(const csa2_config_t* cfg, int32_t batch, const int64_t* capacity) {
  if (check_cfg(cfg) != CSA2_OK || batch <= 0 || batch > 4096 || !capacity) return 0;
  int64_t total = 0;
  for (int i = 0; i < batch; ++i) {
    if (capacity[i] < 0 || capacity[i] > (int64_t)INT32_MAX) return 0;
    total += capacity[i];
  }
  if (total <= 0) return 0;
  return layout_for(cfg, total).total;
}

csa2_status_t csa2_cache_create(const csa2_config_t* cfg, int32_t batch, const int64_t* capacity,
                                void* dev_mem, size_t bytes, csa2_stream_t stream,
                                csa2_cache_t** out) {
  CSA2_RANGE();
  if (!out) return CSA2_ERR_INVALID_ARG;
  *out = nullptr;
  csa2_status_t st = check_cfg(cfg);
  if (st != CSA2_OK) return st;
  if (batch <= 0 || batch > 4096 || !capacity || !dev_mem) return CSA2_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_mem) & (kAlign - 1)) != 0) return CSA2_ERR_INVALID_ARG;
  const size_t need = csa2_cache_bytes(cfg, batch, capacity);
  if (need == 0) return CSA2_ERR_INVALID_ARG;
  if (bytes < need) return CSA2_ERR_CAPACITY;

  csa2_cache* c = new (std::nothrow) csa2_cache();
  if (!c) return CSA2_ERR_OOM;
  c->cfg = *cfg;
  c->batch = batch;
  c->group = cfg->layout == CSA2_KV_L16_E4M3 ? 16 : 32;
  c->scale_bytes = kHeadDim / c->group;
  c->cap.assign(capacity, capacity + batch);
  c->off.resize(batch + 1);
  c->len.assign(batch, 0);
  c->off[0] = 0;
  c->max_cap = 0;
  for (int i = 0; i < batch; ++i) {
    c->off[i + 1] = c->off[i] + capacity[i];
    c->max_cap = std::max(c->max_cap, capacity[i]);
  }
  c->total = c->off[batch];
  const Layout L = layout_for(cfg, c->total);
  c->base = static_cast<uint8_t*>(dev_mem);
  c->bytes = bytes;
  c->d_len = reinterpret_cast<int32_t*>(c->base + L.len_off);
  c->d_err = reinterpret_cast<uint32_t*>(c->base + L.err_off);
  c->codes = c->base + L.codes_off;
  c->scales = c->base + L.scales_off;
  const bool mx = cfg->idx_layout == CSA2_IDX_MXFP4;
  c->idxk = mx ? nullptr : reinterpret_cast<uint16_t*>(c->base + L.idxk_off);
  c->idx_codes = mx ? c->base + L.idxk_off : nullptr;
  c->idx_scales = mx ? c->base + L.idxs_off : nullptr;
  c->idx_rows = mx ? mxfp4_rows(c->total) : 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete c;
    return CSA2_ERR_CUDA;
  }
  c->index_sms = c->num_sms;
  c->wait_cycles = 0;
  c->inject = 0;
  if (!mx && (!make_map(&c->tm_k, c->idxk, (uint64_t)c->total, kIdxDim, 64, 128) ||
              !make_block_map(&c->tm_k8, c->idxk, (uint64_t)c->total))) {
    delete c;
    return CSA2_ERR_CUDA;
  }
  if (mx && (!make_perm_map(&c->tm_kq, c->idx_codes, c->idx_rows) ||
             !make_code_map(&c->tm_kc8, c->idx_codes, (uint64_t)c->total, kIdxDim / 2, kHsiBlock))) {
    delete c;
    return CSA2_ERR_CUDA;
  }
  if (cudaMemsetAsync(c->base, 0, L.codes_off, S(stream)) != cudaSuccess) {
    delete c;
    return CSA2_ERR_CUDA;
  }
  *out = c;
  return CSA2_OK;
}

csa2_status_t csa2_cache_destroy(csa2_cache_t* c) {
  CSA2_RANGE();
  if (!c) return CSA2_ERR_INVALID_ARG;
  delete c;
  return CSA2_OK;
}

csa2_status_t csa2_cache_set_index_sms(csa2_cache_t* c, int32_t n_sms) {
  CSA2_RANGE();
  if (!c || n_sms < 0) return CSA2_ERR_INVALID_ARG;
  c->index_sms = (n_sms == 0 || n_sms > c->num_sms) ? c->num_sms : n_sms;
  return CSA2_OK;
}

csa2_status_t csa2_cache_set_wait_limit(csa2_cache_t* c, int64_t cycles) {
  CSA2_RANGE();
  if (!c || cycles < 0) return CSA2_ERR_INVALID_ARG;
  c->wait_cycles = cycles;
  return CSA2_OK;
}

csa2_status_t csa2_cache_inject_fault(csa2_cache_t* c, int32_t fault) {
  CSA2_RANGE();
  if (!c || (fault != CSA2_FAULT_NONE && fault != CSA2_FAULT_INDEX_NO_KEY_LOADS))
    return CSA2_ERR_INVALID_ARG;
  c->inject = fault == CSA2_FAULT_INDEX_NO_KEY_LOADS ? kInjectNoKeyLoads : 0;
  return CSA2_OK;
}

csa2_status_t csa2_cache_reset(csa2_cache_t* c, csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c) return CSA2_ERR_INVALID_ARG;
  std::fill(c->len.begin(), c->len.end(), 0);
  return cuda_status(cudaMemsetAsync(c->d_len, 0, sizeof(int32_t) * c->batch, S(stream)));
}

csa2_status_t csa2_cache_length(const csa2_cache_t* c, int32_t seq, int64_t* n) {
  CSA2_RANGE();
  if (!c || !n || seq < 0 || seq >= c->batch) return CSA2_ERR_INVALID_ARG;
  *n = c->len[seq];
  return CSA2_OK;
}

csa2_status_t csa2_cache_views(const csa2_cache_t* c, csa2_cache_views_t* v) {
  CSA2_RANGE();
  if (!c || !v) return CSA2_ERR_INVALID_ARG;
  v->codes = c->codes;
  v->scales = c->scales;
  v->idx_k = c->idxk;
  v->idx_codes = c->idx_codes;
  v->idx_scales = c->idx_scales;
  v->lengths = c->d_len;
  v->entry_offset = c->off.data();
  v->total = c->total;
  v->batch = c->batch;
  v->group = c->group;
  return CSA2_OK;
}

csa2_status_t csa2_compress(int32_t ratio, int64_t n_out, int32_t dim, const void* c_tok,
                            const float* z_tok, float* out, csa2_stream_t stream) {
  CSA2_RANGE();
  if (ratio < 1 || ratio > 16 || n_out < 0 || dim <= 0 || dim % 16 != 0 || dim > kHeadDim)
    return ratio > 16 || dim > kHeadDim ? CSA2_ERR_UNSUPPORTED : CSA2_ERR_INVALID_ARG;
  if (n_out == 0) return CSA2_OK;
  if (!c_tok || !z_tok || !out || !aligned16(c_tok) || !aligned16(z_tok) || !aligned16(out))
    return CSA2_ERR_INVALID_ARG;
  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  p.mode = 0;
  p.ratio = ratio;
  p.dim = dim;
  p.n_segs = 1;
  p.rows = n_out;
  p.seg[0].first = 0;
  p.c_tok = static_cast<const uint16_t*>(c_tok);
  p.z_tok = z_tok;
  p.entries_out = out;
  return cuda_status(launch_append(p, S(stream)));
}

csa2_status_t csa2_append_entries(csa2_cache_t* c, int32_t n_seqs, const int32_t* seq_ids,
                                  const int32_t* n_new, const float* entries, const void* idx_k,
                                  csa2_stream_t stream) {
  CSA2_RANGE();
  return run_append(c, 1, n_seqs, seq_ids, n_new, entries, nullptr, nullptr, idx_k, nullptr,
                    stream);
}

csa2_status_t csa2_append_tokens(csa2_cache_t* c, int32_t n_seqs, const int32_t* seq_ids,
                                 const int32_t* n_tok, const void* c_tok, const float* z_tok,
                                 const void* idx_k, float* entries_out, csa2_stream_t stream) {
  CSA2_RANGE();
  return run_append(c, 2, n_seqs, seq_ids, n_tok, nullptr, c_tok, z_tok, idx_k, entries_out,
                    stream);
}

size_t csa2_index_workspace_bytes(const csa2_cache_t* c, int32_t n_queries) {
  if (!c || n_queries < 0) return 0;
  return (size_t)n_queries * ((size_t)score_ld(c->max_cap) * sizeof(float) +
                              kKeyHistBinsHost * sizeof(uint32_t)) +
         topk_seg_bytes(n_queries, c->max_cap);
}

size_t csa2_index_prefill_workspace_bytes(const csa2_cache_t* c, int32_t seq, int32_t n_queries) {
  if (!c || seq < 0 || seq >= c->batch || n_queries < 0) return 0;
  size_t b = (size_t)n_queries * (size_t)score_ld(c->cap[seq]) * sizeof(float);
  if (c->cfg.idx_layout == CSA2_IDX_BF16) b += (size_t)n_queries * kKeyHistBinsHost * sizeof(uint32_t);
  return b;
}

size_t csa2_topk_workspace_bytes(int32_t n_rows, int64_t max_valid) {
  if (n_rows < 0 || max_valid < 0) return 0;
  return topk_seg_bytes(n_rows, max_valid);
}

}  // extern "C"

namespace {
csa2_status_t topk_impl(int32_t n_rows, const void* scores, int64_t ld, const int64_t* n_valid,
                        int32_t k, const uint32_t* key_hist, int32_t* idx_out, float* score_out,
                        void* workspace, size_t ws_bytes, csa2_stream_t stream, bool bf16) {
  if (n_rows < 0 || k <= 0 || k > 4096) return CSA2_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (!scores || !n_valid || !idx_out || ld < 0) return CSA2_ERR_INVALID_ARG;
  const size_t esz = bf16 ? 2 : 4;
  int64_t max_valid = 0;
  for (int r = 0; r < n_rows; ++r) {
    if (n_valid[r] < 0 || n_valid[r] > ld || n_valid[r] > (int64_t)INT32_MAX)
      return CSA2_ERR_INVALID_ARG;
    max_valid = std::max(max_valid, n_valid[r]);
  }
  const bool seg = key_hist && workspace && aligned16(workspace) && topk_segments(max_valid) > 2 &&
                   ws_bytes >= topk_seg_bytes(n_rows, max_valid) &&
                   topk_segments(max_valid) <= 1024;
  const int n_seg = topk_segments(max_valid);
  for (int r0 = 0; r0 < n_rows; r0 += kTopkTab) {
    const int nr = std::min(kTopkTab, n_rows - r0);
    TopkParams* p = new (std::nothrow) TopkParams();
    if (!p) return CSA2_ERR_OOM;
    p->scores = reinterpret_cast<const float*>(static_cast<const uint8_t*>(scores) +
                                               (size_t)r0 * ld * esz);
    p->score_bf16 = bf16 ? 1 : 0;
    p->ld = ld;
    p->rows = nr;
    p->k = k;
    p->idx_out = idx_out + (int64_t)r0 * k;
    p->score_out = score_out ? score_out + (int64_t)r0 * k : nullptr;
    p->key_hist = key_hist ? key_hist + (int64_t)r0 * kKeyHistBinsHost : nullptr;
    p->seg_ws = seg ? static_cast<uint32_t*>(workspace) +
                          (size_t)r0 * topk_seg_bytes(1, max_valid) / sizeof(uint32_t)
                    : nullptr;
    p->n_seg = seg ? n_seg : 0;
    p->formula = 0;
    for (int r = 0; r < nr; ++r) p->n_valid[r] = n_valid[r0 + r];
    cudaError_t e = launch_topk(*p, S(stream));
    delete p;
    if (e != cudaSuccess) return CSA2_ERR_CUDA;
  }
  return CSA2_OK;
}
}  // namespace

extern "C" {

csa2_status_t csa2_topk(int32_t n_rows, const float* scores, int64_t ld, const int64_t* n_valid,
                        int32_t k, const uint32_t* key_hist, int32_t* idx_out, float* score_out,
                        void* workspace, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_RANGE();
  return topk_impl(n_rows, scores, ld, n_valid, k, key_hist, idx_out, score_out, workspace,
                   ws_bytes, stream, false);
}

csa2_status_t csa2_topk_bf16(int32_t n_rows, const uint16_t* scores, int64_t ld,
                             const int64_t* n_valid, int32_t k, const uint32_t* key_hist,
                             int32_t* idx_out, float* score_out, void* workspace, size_t ws_bytes,
                             csa2_stream_t stream) {
  CSA2_RANGE();
  return topk_impl(n_rows, scores, ld, n_valid, k, key_hist, idx_out, score_out, workspace,
                   ws_bytes, stream, true);
}

}  // extern "C"

namespace {

// Scores of decode queries [q0, q0 + n) into scores (row stride ld): one
// indexer launch per chunk of up to kMaxIdxGroups queries.
// Entries query i sees: its sequence's appended entries, or with a token
// position those causally visible there, (s + 1) * ratio - 1 <= pos.
int64_t visible_of(const csa2_cache_t* c, int32_t s, const int64_t* q_pos, int i) {
  const int64_t len = c->len[s];
  if (!q_pos) return len;
  return std::min<int64_t>(len, (q_pos[i] + 1) / c->cfg.ratio);
}

csa2_status_t run_index_decode(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                               const float* w, const int32_t* seq_ids, void* scores, int64_t ld,
                               uint32_t* key_hist, csa2_stream_t stream, IndexParams* ip,
                               bool bf16 = false, const int64_t* q_pos = nullptr) {
  const size_t esz = bf16 ? 2 : 4;
  const uint16_t* qb = static_cast<const uint16_t*>(q_idx);
  if (key_hist &&
      cudaMemsetAsync(key_hist, 0, (size_t)nq * kKeyHistBinsHost * sizeof(uint32_t), S(stream)) !=
          cudaSuccess)
    return CSA2_ERR_CUDA;
  // keys per decode tile: 512 for MXFP4 keys, 256 for bf16 keys
  const bool mx = c->cfg.idx_layout == CSA2_IDX_MXFP4;
  const int64_t tile_e = mx ? 512 : 256;
  for (int q0 = 0; q0 < nq; q0 += kMaxIdxGroups) {
    const int n = std::min(kMaxIdxGroups, nq - q0);
    std::memset(ip, 0, sizeof(IndexParams));
    ip->w = w + (int64_t)q0 * kIdxHeads;
    ip->scores = reinterpret_cast<float*>(static_cast<uint8_t*>(scores) + (size_t)q0 * ld * esz);
    ip->score_bf16 = bf16 ? 1 : 0;
    ip->ld = ld;
    ip->key_hist = key_hist ? key_hist + (int64_t)q0 * kKeyHistBinsHost : nullptr;
    ip->err = c->d_err;
    ip->nq = n;
    ip->qpg = 1;
    ip->n_groups = n;
    ip->prefill = 0;
    ip->ratio = c->cfg.ratio;
    ip->wait_cycles = c->wait_cycles;
    ip->inject = c->inject;
    ip->tile_prefix[0] = 0;
    for (int i = 0; i < n; ++i) {
      const int s = seq_ids ? seq_ids[q0 + i] : q0 + i;
      const int64_t nv = visible_of(c, s, q_pos, q0 + i);
      ip->entry_base[i] = c->off[s];
      ip->nvis[i] = (int32_t)nv;
      // MXFP4 decode tiles are aligned 512-key chunks: a sequence starting
      // inside one begins `lead` keys into its first tile
      const int64_t lead = (mx && nv > 0) ? (c->off[s] & 511) : 0;
      ip->tile_prefix[i + 1] = ip->tile_prefix[i] + (int32_t)((nv + lead + tile_e - 1) / tile_e);
    }
    CUtensorMap tm_q;
    const uint16_t* qn = qb + (int64_t)q0 * kIdxHeads * kIdxDim;
    if (!make_map(&tm_q, qn, (uint64_t)n * kIdxHeads, kIdxDim, 64, 32)) return CSA2_ERR_CUDA;
    const int tiles = ip->tile_prefix[n];
    if (tiles > 0) {
      const int grid = std::min(c->index_sms, tiles);
      if (launch_index_any(c, *ip, tm_q, qn, grid, S(stream)) != cudaSuccess) return CSA2_ERR_CUDA;
    }
  }
  return CSA2_OK;
}

csa2_status_t check_decode_queries(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                   const float* w, const int32_t* seq_ids) {
  if (!q_idx || !w || !aligned16(q_idx) || !aligned16(w)) return CSA2_ERR_INVALID_ARG;
  if (seq_ids) {
    for (int i = 0; i < nq; ++i)
      if (seq_ids[i] < 0 || seq_ids[i] >= c->batch) return CSA2_ERR_INVALID_ARG;
  } else if (nq > c->batch) {
    return CSA2_ERR_INVALID_ARG;
  }
  return CSA2_OK;
}

}  // namespace

extern "C" {

csa2_status_t csa2_index_scores_decode(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                       const float* w, const int32_t* seq_ids, float* scores,
                                       int64_t ld, uint32_t* key_hist, csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  csa2_status_t st = check_decode_queries(c, nq, q_idx, w, seq_ids);
  if (st != CSA2_OK) return st;
  if (!scores || !aligned16(scores) || ld % 4 != 0) return CSA2_ERR_INVALID_ARG;
  for (int i = 0; i < nq; ++i)
    if (c->len[seq_ids ? seq_ids[i] : i] > ld) return CSA2_ERR_CAPACITY;
  IndexParams* ip = new (std::nothrow) IndexParams();
  if (!ip) return CSA2_ERR_OOM;
  if (key_hist && !aligned16(key_hist)) { delete ip; return CSA2_ERR_INVALID_ARG; }
  st = run_index_decode(c, nq, q_idx, w, seq_ids, scores, ld, key_hist, stream, ip);
  delete ip;
  return st;
}

}  // extern "C"

namespace {
csa2_status_t index_topk_decode_impl(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                     const float* w, const int32_t* seq_ids, int32_t* topk_idx,
                                     float* topk_score, void* workspace, size_t ws_bytes,
                                     csa2_stream_t stream, bool bf16,
                                     const int64_t* q_pos = nullptr) {
  if (!c || nq < 0) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  csa2_status_t st = check_decode_queries(c, nq, q_idx, w, seq_ids);
  if (st != CSA2_OK) return st;
  if (q_pos)
    for (int i = 0; i < nq; ++i)
      if (q_pos[i] < 0) return CSA2_ERR_INVALID_ARG;
  if (!topk_idx || !workspace || !aligned16(workspace)) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < csa2_index_workspace_bytes(c, nq)) return CSA2_ERR_CAPACITY;
  // bf16 rows: a multiple of 8 scores keeps every row 16-byte aligned (and
  // the bf16 layout never needs more bytes than the fp32 one)
  const int64_t ld = bf16 ? (c->max_cap + 7) / 8 * 8 : score_ld(c->max_cap);
  const size_t esz = bf16 ? 2 : 4;
  uint8_t* scores = static_cast<uint8_t*>(workspace);
  uint32_t* key_hist = reinterpret_cast<uint32_t*>(scores + (size_t)nq * ld * esz);
  uint32_t* seg_ws = key_hist + (int64_t)nq * kKeyHistBinsHost;
  IndexParams* ip = new (std::nothrow) IndexParams();
  TopkParams* tp = new (std::nothrow) TopkParams();
  if (!ip || !tp) { delete ip; delete tp; return CSA2_ERR_OOM; }
  st = run_index_decode(c, nq, q_idx, w, seq_ids, scores, ld, key_hist, stream, ip, bf16, q_pos);
  const int k = c->cfg.topk;
  for (int q0 = 0; q0 < nq && st == CSA2_OK; q0 += kTopkTab) {
    const int n = std::min(kTopkTab, nq - q0);
    std::memset(tp, 0, sizeof(TopkParams));
    tp->scores = reinterpret_cast<const float*>(scores + (size_t)q0 * ld * esz);
    tp->score_bf16 = bf16 ? 1 : 0;
    tp->ld = ld;
    tp->rows = n;
    tp->k = k;
    tp->idx_out = topk_idx + (int64_t)q0 * k;
    tp->score_out = topk_score ? topk_score + (int64_t)q0 * k : nullptr;
    tp->key_hist = key_hist + (int64_t)q0 * kKeyHistBinsHost;
    // segments pay from three on: rows of up to two (16384 scores) are
    // compacted by the row kernel in one block-wide pass, one launch
    const bool use_seg = topk_segments(c->max_cap) <= 1024 && topk_segments(c->max_cap) > 2;
    tp->seg_ws = use_seg ? seg_ws + (size_t)q0 * topk_seg_bytes(1, c->max_cap) / sizeof(uint32_t)
                         : nullptr;
    tp->n_seg = use_seg ? topk_segments(c->max_cap) : 0;
    tp->formula = 0;
    tp->err = c->d_err;
    for (int i = 0; i < n; ++i)
      tp->n_valid[i] = visible_of(c, seq_ids ? seq_ids[q0 + i] : q0 + i, q_pos, q0 + i);
    if (launch_topk(*tp, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
  }
  delete ip;
  delete tp;
  return st;
}
}  // namespace

extern "C" {

csa2_status_t csa2_index_topk_decode(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                     const float* w, const int32_t* seq_ids, int32_t* topk_idx,
                                     float* topk_score, void* workspace, size_t ws_bytes,
                                     csa2_stream_t stream) {
  CSA2_RANGE();
  return index_topk_decode_impl(c, nq, q_idx, w, seq_ids, topk_idx, topk_score, workspace,
                                ws_bytes, stream, false);
}

csa2_status_t csa2_index_topk(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                              const float* w, const int32_t* seq_of_q, const int64_t* q_pos,
                              int32_t* topk_idx, float* topk_score, void* workspace,
                              size_t ws_bytes, csa2_stream_t stream) {
  CSA2_RANGE();
  if (!q_pos) return CSA2_ERR_INVALID_ARG;
  return index_topk_decode_impl(c, nq, q_idx, w, seq_of_q, topk_idx, topk_score, workspace,
                                ws_bytes, stream, false, q_pos);
}

csa2_status_t csa2_index_topk_decode_bf16(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                          const float* w, const int32_t* seq_ids,
                                          int32_t* topk_idx, float* topk_score, void* workspace,
                                          size_t ws_bytes, csa2_stream_t stream) {
  CSA2_RANGE();
  return index_topk_decode_impl(c, nq, q_idx, w, seq_ids, topk_idx, topk_score, workspace,
                                ws_bytes, stream, true);
}

csa2_status_t csa2_index_scores_decode_bf16(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                            const float* w, const int32_t* seq_ids,
                                            uint16_t* scores, int64_t ld, uint32_t* key_hist,
                                            csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  csa2_status_t st = check_decode_queries(c, nq, q_idx, w, seq_ids);
  if (st != CSA2_OK) return st;
  if (!scores || !aligned16(scores) || ld % 8 != 0) return CSA2_ERR_INVALID_ARG;
  for (int i = 0; i < nq; ++i)
    if (c->len[seq_ids ? seq_ids[i] : i] > ld) return CSA2_ERR_CAPACITY;
  if (key_hist && !aligned16(key_hist)) return CSA2_ERR_INVALID_ARG;
  IndexParams* ip = new (std::nothrow) IndexParams();
  if (!ip) return CSA2_ERR_OOM;
  st = run_index_decode(c, nq, q_idx, w, seq_ids, scores, ld, key_hist, stream, ip, true);
  delete ip;
  return st;
}

csa2_status_t csa2_index_scores_prefill(const csa2_cache_t* c, int32_t seq, int32_t nq,
                                        int64_t pos0, const void* q_idx, const float* w,
                                        float* scores, int64_t ld, uint32_t* key_hist,
                                        csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0 || seq < 0 || seq >= c->batch || pos0 < 0) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  if (!q_idx || !w || !scores || !aligned16(q_idx) || !aligned16(w) || !aligned16(scores) ||
      ld % 4 != 0 || (key_hist && !aligned16(key_hist)))
    return CSA2_ERR_INVALID_ARG;
  if (ld < c->len[seq]) return CSA2_ERR_CAPACITY;
  // queries sharing one tile of keys in the MMA: 8 (N = 256) on bf16 keys,
  // 4 (N = 128) on MXFP4 keys, whose tensor memory also holds the scales
  const bool mx = c->cfg.idx_layout == CSA2_IDX_MXFP4;
  // the score-key histograms come from the bf16 indexer's epilogue (the
  // MXFP4 kernel's shared memory has no room for eight of them)
  if (key_hist && mx) return CSA2_ERR_UNSUPPORTED;
  if (key_hist &&
      cudaMemsetAsync(key_hist, 0, (size_t)nq * kKeyHistBinsHost * sizeof(uint32_t), S(stream)) !=
          cudaSuccess)
    return CSA2_ERR_CUDA;
  const int kQpg = mx ? 4 : 8;
  const int m = c->cfg.ratio;
  const int64_t len = c->len[seq];
  const uint16_t* qb = static_cast<const uint16_t*>(q_idx);
  IndexParams* ip = new (std::nothrow) IndexParams();
  if (!ip) return CSA2_ERR_OOM;
  csa2_status_t st = CSA2_OK;
  const int per_launch = kMaxIdxGroups * kQpg;
  for (int q0 = 0; q0 < nq && st == CSA2_OK; q0 += per_launch) {
    const int n = std::min(per_launch, nq - q0);
    const int groups = (n + kQpg - 1) / kQpg;
    std::memset(ip, 0, sizeof(IndexParams));
    ip->w = w + (int64_t)q0 * kIdxHeads;
    ip->scores = scores + (int64_t)q0 * ld;
    ip->ld = ld;
    ip->key_hist = key_hist ? key_hist + (int64_t)q0 * kKeyHistBinsHost : nullptr;
    ip->err = c->d_err;
    ip->nq = n;
    ip->qpg = kQpg;
    ip->n_groups = groups;
    ip->prefill = 1;
    ip->pre_base = c->off[seq];
    ip->pos0 = pos0 + q0;
    ip->pre_len = (int32_t)len;
    ip->ratio = m;
    ip->wait_cycles = c->wait_cycles;
    ip->inject = c->inject;
    ip->tile_prefix[0] = 0;
    for (int g = 0; g < groups; ++g) {
      const int64_t last = std::min<int64_t>((int64_t)g * kQpg + kQpg, n) - 1;
      const int64_t nv = std::min<int64_t>(len, (ip->pos0 + last + 1) / m);
      // MXFP4 tiles are aligned 128-key chunks (the first one `lead` keys
      // before the sequence start)
      const int64_t lead = (mx && nv > 0) ? (c->off[seq] & 127) : 0;
      ip->tile_prefix[g + 1] = ip->tile_prefix[g] + (int32_t)((nv + lead + 127) / 128);
    }
    CUtensorMap tm_q;
    const uint16_t* qn = qb + (int64_t)q0 * kIdxHeads * kIdxDim;
    if (!make_map(&tm_q, qn, (uint64_t)n * kIdxHeads, kIdxDim, 64, 32 * kQpg)) {
      st = CSA2_ERR_CUDA;
      break;
    }
    const int tiles = ip->tile_prefix[groups];
    if (tiles > 0) {
      const int grid = std::min(c->index_sms, tiles);
      if (launch_index_any(c, *ip, tm_q, qn, grid, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
    }
  }
  delete ip;
  return st;
}

csa2_status_t csa2_index_topk_prefill(const csa2_cache_t* c, int32_t seq, int32_t nq, int64_t pos0,
                                      const void* q_idx, const float* w, int32_t* topk_idx,
                                      float* topk_score, void* workspace, size_t ws_bytes,
                                      csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0 || seq < 0 || seq >= c->batch || pos0 < 0) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  if (!topk_idx || !workspace || !aligned16(workspace)) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < csa2_index_prefill_workspace_bytes(c, seq, nq)) return CSA2_ERR_CAPACITY;
  const int64_t ld = score_ld(c->cap[seq]);
  // workspace: scores [nq, ld], then (bf16 keys) the score-key histograms
  // [nq, 2048] that the indexer builds for the top-k's first digit
  float* scores = static_cast<float*>(workspace);
  uint32_t* key_hist = c->cfg.idx_layout == CSA2_IDX_BF16
                           ? reinterpret_cast<uint32_t*>(scores + (size_t)nq * ld)
                           : nullptr;
  csa2_status_t st =
      csa2_index_scores_prefill(c, seq, nq, pos0, q_idx, w, scores, ld, key_hist, stream);
  if (st != CSA2_OK) return st;
  TopkParams* tp = new (std::nothrow) TopkParams();
  if (!tp) return CSA2_ERR_OOM;
  tp->scores = scores;
  tp->key_hist = key_hist;
  tp->ld = ld;
  tp->rows = nq;
  tp->k = c->cfg.topk;
  tp->idx_out = topk_idx;
  tp->score_out = topk_score;
  tp->formula = 1;
  tp->err = c->d_err;
  tp->pre_len = (int32_t)c->len[seq];
  tp->ratio = c->cfg.ratio;
  tp->pos0 = pos0;
  if (launch_topk(*tp, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
  delete tp;
  return st;
}

size_t csa2_sparse_attn_workspace_bytes(const csa2_cache_t* c, int32_t n_queries) {
  if (!c || n_queries < 0) return 0;
  return kAttnSplitToken;
}

}  // extern "C"

namespace {
// Epilogue options into the launch parameters; false when they are invalid.
// Epilogue options of layer `ly` of a launch (sink, FP8 window rows), and
// the launch's output RoPE (shared by its layers); false when they are
// invalid.
bool apply_opts(AttnParams* p, AttnLayer* ly, const csa2_attn_opts_t* opts, bool decode,
                int32_t q0, int64_t row0) {
  if (!opts) return true;
  ly->sink = opts->sink;
  const bool f8 = opts->swa_codes || opts->swa_rope || opts->swa_scales;
  if (f8) {
    if (!opts->swa_codes || !opts->swa_rope || !opts->swa_scales || !aligned16(opts->swa_codes) ||
        !aligned16(opts->swa_rope) || (reinterpret_cast<uintptr_t>(opts->swa_scales) & 7u))
      return false;
    ly->swa_codes = opts->swa_codes + row0 * 448;
    ly->swa_rope = static_cast<const uint16_t*>(opts->swa_rope) + row0 * 64;
    ly->swa_scales = opts->swa_scales + row0 * 8;
  }
  if (opts->rope_out) {
    if (decode && !opts->rope_pos) return false;
    if (opts->rope_base < 0.0 || opts->rope_base != opts->rope_base) return false;
    p->rope_out = 1;
    p->rope_pos = decode ? opts->rope_pos + q0 : nullptr;
    const double base = opts->rope_base > 0.0 ? opts->rope_base : 10000.0;
    for (int t = 0; t < 32; ++t) p->rope_theta[t] = std::pow(base, -(double)t / 32.0);
  }
  return true;
}
}  // namespace

extern "C" {

csa2_status_t csa2_sparse_attn_decode(const csa2_cache_t* c, int32_t nq, const int32_t* seq_ids,
                                      const void* q, const void* swa_kv, const int32_t* swa_len,
                                      const int32_t* topk_idx, float scale, void* out, float* lse,
                                      void* workspace, size_t ws_bytes, csa2_stream_t stream) {
  CSA2_RANGE();
  return csa2_sparse_attn_decode_ex(c, nq, seq_ids, q, swa_kv, swa_len, topk_idx, scale, out, lse,
                                    workspace, ws_bytes, nullptr, stream);
}

csa2_status_t csa2_sparse_attn_decode_ex(const csa2_cache_t* c, int32_t nq,
                                         const int32_t* seq_ids, const void* q,
                                         const void* swa_kv, const int32_t* swa_len,
                                         const int32_t* topk_idx, float scale, void* out,
                                         float* lse, void* workspace, size_t ws_bytes,
                                         const csa2_attn_opts_t* opts, csa2_stream_t stream) {
  CSA2_RANGE();
  return csa2_sparse_attn_decode_layers(c, 1, nq, seq_ids, &q, &swa_kv, swa_len, topk_idx, scale,
                                        &out, &lse, workspace, ws_bytes, &opts, stream);
}

csa2_status_t csa2_sparse_attn_decode_layers(const csa2_cache_t* c, int32_t n_layers, int32_t nq,
                                             const int32_t* seq_ids, const void* const* q,
                                             const void* const* swa_kv, const int32_t* swa_len,
                                             const int32_t* topk_idx, float scale,
                                             void* const* out, float* const* lse,
                                             void* workspace, size_t ws_bytes,
                                             const csa2_attn_opts_t* const* opts,
                                             csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0 || n_layers < 1 || n_layers > CSA2_MAX_ATTN_LAYERS || !q || !out)
    return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  const int W = c->cfg.swa;
  if (!topk_idx || !aligned16(topk_idx)) return CSA2_ERR_INVALID_ARG;
  const csa2_attn_opts_t* o0 = opts ? opts[0] : nullptr;
  for (int l = 0; l < n_layers; ++l) {
    const csa2_attn_opts_t* ol = opts ? opts[l] : nullptr;
    if (!q[l] || !out[l] || !aligned16(q[l]) || !aligned16(out[l])) return CSA2_ERR_INVALID_ARG;
    const bool f8 = ol && ol->swa_codes;
    const void* sw = swa_kv ? swa_kv[l] : nullptr;
    if (W > 0 && !f8 && (!sw || !aligned16(sw))) return CSA2_ERR_INVALID_ARG;
    if (lse && lse[l] && !aligned16(lse[l])) return CSA2_ERR_INVALID_ARG;
    // the output RoPE is one setting for the launch: every layer the same
    const bool r0 = o0 && o0->rope_out, rl = ol && ol->rope_out;
    if (r0 != rl || (rl && (ol->rope_pos != o0->rope_pos || ol->rope_base != o0->rope_base)))
      return CSA2_ERR_INVALID_ARG;
  }
  if (workspace && !aligned16(workspace)) return CSA2_ERR_INVALID_ARG;
  if (seq_ids)
    for (int i = 0; i < nq; ++i)
      if (seq_ids[i] < 0 || seq_ids[i] >= c->batch) return CSA2_ERR_INVALID_ARG;
  if (!seq_ids && nq > c->batch) return CSA2_ERR_INVALID_ARG;
  const int H = c->cfg.n_heads, k = c->cfg.topk, G = H / kAttnHeadGroup;
  AttnParams* p = new (std::nothrow) AttnParams();
  AttnMaps* maps = new (std::nothrow) AttnMaps();
  if (!p || !maps) { delete p; delete maps; return CSA2_ERR_OOM; }
  csa2_status_t st = CSA2_OK;
  for (int q0 = 0; q0 < nq && st == CSA2_OK; q0 += kAttnTab) {
    const int n = std::min(kAttnTab, nq - q0);
    // two CTAs per (query, head group) when the pairs still fit the SMs in
    // one wave: a second wave of split CTAs costs more than unsplit CTAs
    // leaving some SMs idle
    const bool split = workspace && ws_bytes >= kAttnSplitToken &&
                       2 * (int64_t)n_layers * n * G <= c->num_sms;
    std::memset(p, 0, sizeof(AttnParams));
    p->topk_idx = topk_idx + (int64_t)q0 * k;
    p->swa_len = swa_len ? swa_len + q0 : nullptr;
    p->codes = c->codes;
    p->scales = c->scales;
    p->n_layers = n_layers;
    p->err = c->d_err;
    p->nq = n;
    p->n_heads = H;
    p->topk = k;
    p->swa = W;
    p->layout = c->cfg.layout;
    p->scale = scale;
    p->scale_log2 = scale * 1.4426950408889634f;
    p->prefill = 0;
    p->splits = split ? 2 : 1;
    p->wait_cycles = c->wait_cycles;
    for (int i = 0; i < n; ++i) {
      const int s = seq_ids ? seq_ids[q0 + i] : q0 + i;
      p->q_base[i] = c->off[s];
      p->q_len[i] = (int32_t)c->len[s];
    }
    for (int l = 0; l < n_layers && st == CSA2_OK; ++l) {
      AttnLayer& ly = p->layer[l];
      const csa2_attn_opts_t* ol = opts ? opts[l] : nullptr;
      ly.out = static_cast<uint16_t*>(out[l]) + (int64_t)q0 * H * kHeadDim;
      ly.lse = (lse && lse[l]) ? lse[l] + (int64_t)q0 * H : nullptr;
      if (!apply_opts(p, &ly, ol, true, q0, (int64_t)q0 * W)) { st = CSA2_ERR_INVALID_ARG; break; }
      const uint16_t* qb = static_cast<const uint16_t*>(q[l]) + (int64_t)q0 * H * kHeadDim;
      if (!make_map(&maps->q[l], qb, (uint64_t)n * H, kHeadDim, 64, kAttnHeadGroup)) {
        st = CSA2_ERR_CUDA;
        break;
      }
      if (W > 0 && !(ol && ol->swa_codes)) {
        const uint16_t* sb = static_cast<const uint16_t*>(swa_kv[l]) + (int64_t)q0 * W * kHeadDim;
        if (!make_map(&maps->swa[l], sb, (uint64_t)n * W, kHeadDim, 64, 128)) { st = CSA2_ERR_CUDA; break; }
      } else {
        maps->swa[l] = maps->q[l];
      }
    }
    if (st == CSA2_OK && launch_attn(*p, *maps, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
  }
  delete p;
  delete maps;
  return st;
}

csa2_status_t csa2_sparse_attn_prefill(const csa2_cache_t* c, int32_t seq, int32_t nq,
                                       int64_t pos0, const void* q, const void* swa_kv,
                                       int64_t swa_pos0, int64_t n_swa_rows,
                                       const int32_t* topk_idx, float scale, void* out, float* lse,
                                       csa2_stream_t stream) {
  CSA2_RANGE();
  return csa2_sparse_attn_prefill_ex(c, seq, nq, pos0, q, swa_kv, swa_pos0, n_swa_rows, topk_idx,
                                     scale, out, lse, nullptr, stream);
}

csa2_status_t csa2_sparse_attn_prefill_ex(const csa2_cache_t* c, int32_t seq, int32_t nq,
                                          int64_t pos0, const void* q, const void* swa_kv,
                                          int64_t swa_pos0, int64_t n_swa_rows,
                                          const int32_t* topk_idx, float scale, void* out,
                                          float* lse, const csa2_attn_opts_t* opts,
                                          csa2_stream_t stream) {
  CSA2_RANGE();
  return csa2_sparse_attn_prefill_layers(c, seq, 1, nq, pos0, &q, &swa_kv, swa_pos0, n_swa_rows,
                                         topk_idx, scale, &out, &lse, &opts, stream);
}

csa2_status_t csa2_sparse_attn_prefill_layers(const csa2_cache_t* c, int32_t seq, int32_t n_layers,
                                              int32_t nq, int64_t pos0, const void* const* q,
                                              const void* const* swa_kv, int64_t swa_pos0,
                                              int64_t n_swa_rows, const int32_t* topk_idx,
                                              float scale, void* const* out, float* const* lse,
                                              const csa2_attn_opts_t* const* opts,
                                              csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0 || seq < 0 || seq >= c->batch || pos0 < 0 || n_layers < 1 ||
      n_layers > CSA2_MAX_ATTN_LAYERS || !q || !out)
    return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  const int W = c->cfg.swa;
  if (!topk_idx || !aligned16(topk_idx)) return CSA2_ERR_INVALID_ARG;
  if (W > 0 && (swa_pos0 < 0 || swa_pos0 > pos0 || n_swa_rows <= 0 ||
                pos0 + nq - 1 - swa_pos0 >= n_swa_rows))
    return CSA2_ERR_INVALID_ARG;
  const csa2_attn_opts_t* o0 = opts ? opts[0] : nullptr;
  for (int l = 0; l < n_layers; ++l) {
    const csa2_attn_opts_t* ol = opts ? opts[l] : nullptr;
    if (!q[l] || !out[l] || !aligned16(q[l]) || !aligned16(out[l])) return CSA2_ERR_INVALID_ARG;
    if (lse && lse[l] && !aligned16(lse[l])) return CSA2_ERR_INVALID_ARG;
    const bool f8 = ol && ol->swa_codes;
    const void* sw = swa_kv ? swa_kv[l] : nullptr;
    if (W > 0 && !f8 && (!sw || !aligned16(sw))) return CSA2_ERR_INVALID_ARG;
    const bool r0 = o0 && o0->rope_out, rl = ol && ol->rope_out;
    if (r0 != rl || (rl && ol->rope_base != o0->rope_base)) return CSA2_ERR_INVALID_ARG;
  }
  const int H = c->cfg.n_heads, k = c->cfg.topk;
  AttnParams* p = new (std::nothrow) AttnParams();
  AttnMaps* maps = new (std::nothrow) AttnMaps();
  if (!p || !maps) { delete p; delete maps; return CSA2_ERR_OOM; }
  std::memset(p, 0, sizeof(AttnParams));
  p->topk_idx = topk_idx;
  p->codes = c->codes;
  p->scales = c->scales;
  p->n_layers = n_layers;
  p->err = c->d_err;
  p->nq = nq;
  p->n_heads = H;
  p->topk = k;
  p->swa = W;
  p->layout = c->cfg.layout;
  p->scale = scale;
  p->scale_log2 = scale * 1.4426950408889634f;
  p->prefill = 1;
  p->pre_base = c->off[seq];
  p->pre_len = (int32_t)c->len[seq];
  p->pos0 = pos0;
  p->swa_pos0 = swa_pos0;
  p->splits = 1;
  p->wait_cycles = c->wait_cycles;
  csa2_status_t st = CSA2_OK;
  for (int l = 0; l < n_layers && st == CSA2_OK; ++l) {
    AttnLayer& ly = p->layer[l];
    const csa2_attn_opts_t* ol = opts ? opts[l] : nullptr;
    ly.out = static_cast<uint16_t*>(out[l]);
    ly.lse = lse ? lse[l] : nullptr;
    if (!apply_opts(p, &ly, ol, false, 0, 0)) { st = CSA2_ERR_INVALID_ARG; break; }
    if (!make_map(&maps->q[l], q[l], (uint64_t)nq * H, kHeadDim, 64, kAttnHeadGroup)) {
      st = CSA2_ERR_CUDA;
      break;
    }
    if (W > 0 && !(ol && ol->swa_codes)) {
      if (!make_map(&maps->swa[l], swa_kv[l], (uint64_t)n_swa_rows, kHeadDim, 64, 128)) {
        st = CSA2_ERR_CUDA;
        break;
      }
    } else {
      maps->swa[l] = maps->q[l];
    }
  }
  if (st == CSA2_OK && launch_attn(*p, *maps, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
  delete p;
  delete maps;
  return st;
}

// Device address of g_static_scratch for the current device (host code
// cannot use the symbol itself as a device pointer).  It is looked up again
// on every call made while `stream` is not being captured, so a new context
// (after a device reset) gets its own address; a call during a capture uses
// the address the last uncaptured call found and is refused with
// CSA2_ERR_UNSUPPORTED when there is none (the lookup may load the module,
// which a capture must not contain).
static csa2_status_t static_scratch_ptr(cudaStream_t stream, void** out) {
  static std::mutex mu;
  static void* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CSA2_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return CSA2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return CSA2_ERR_CUDA;
    ptrs[dev] = p;
  } else if (!ptrs[dev]) {
    return CSA2_ERR_UNSUPPORTED;
  }
  *out = ptrs[dev];
  return CSA2_OK;
}

csa2_status_t csa2_index_topk_decode_static(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                            const float* w, const int32_t* seq_ids,
                                            int32_t* topk_idx, float* topk_score,
                                            csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0) return CSA2_ERR_INVALID_ARG;
  if (nq == 0) return CSA2_OK;
  csa2_status_t st = check_decode_queries(c, nq, q_idx, w, seq_ids);
  if (st != CSA2_OK) return st;
  if (!topk_idx) return CSA2_ERR_INVALID_ARG;
  const int64_t ld = score_ld(c->max_cap);
  const size_t need = (size_t)nq * ((size_t)ld * sizeof(float) + kKeyHistBinsHost * sizeof(uint32_t));
  if (need > CSA2_STATIC_SCRATCH_BYTES) return CSA2_ERR_CAPACITY;
  void* scratch = nullptr;
  st = static_scratch_ptr(S(stream), &scratch);
  if (st != CSA2_OK) return st;
  float* scores = static_cast<float*>(scratch);
  uint32_t* key_hist = reinterpret_cast<uint32_t*>(scores + (int64_t)nq * ld);
  // parameter blocks on the stack: this path touches no heap
  IndexParams ip;
  st = run_index_decode(c, nq, q_idx, w, seq_ids, scores, ld, key_hist, stream, &ip);
  const int k = c->cfg.topk;
  TopkParams tp;
  for (int q0 = 0; q0 < nq && st == CSA2_OK; q0 += kTopkTab) {
    const int n = std::min(kTopkTab, nq - q0);
    std::memset(&tp, 0, sizeof(TopkParams));
    tp.scores = scores + (int64_t)q0 * ld;
    tp.ld = ld;
    tp.rows = n;
    tp.k = k;
    tp.idx_out = topk_idx + (int64_t)q0 * k;
    tp.score_out = topk_score ? topk_score + (int64_t)q0 * k : nullptr;
    tp.key_hist = key_hist + (int64_t)q0 * kKeyHistBinsHost;
    tp.seg_ws = nullptr;   // one CTA per row: no segment scratch
    tp.n_seg = 0;
    tp.formula = 0;
    tp.err = c->d_err;
    for (int i = 0; i < n; ++i) tp.n_valid[i] = c->len[seq_ids ? seq_ids[q0 + i] : q0 + i];
    if (launch_topk(tp, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
  }
  return st;
}

// ---------------------------------------------------------------- HSI
static int64_t hsi_ld_b(int64_t max_valid) {
  return score_ld((max_valid + kHsiBlock - 1) / kHsiBlock);
}

size_t csa2_hsi_pool_workspace_bytes(int32_t n_rows, int64_t max_valid) {
  if (n_rows < 0 || max_valid < 0) return 0;
  return (size_t)n_rows * (size_t)hsi_ld_b(max_valid) * sizeof(float);
}

csa2_status_t csa2_hsi_pool(int32_t n_rows, const float* scores, int64_t ld,
                            const int64_t* n_valid, int32_t block, int32_t max_blocks,
                            int32_t* pool_blocks, void* workspace, size_t ws_bytes,
                            csa2_stream_t stream) {
  CSA2_RANGE();
  if (n_rows < 0 || ld < 0) return CSA2_ERR_INVALID_ARG;
  if (block != kHsiBlock || max_blocks <= 0 || max_blocks % 16 != 0 || max_blocks > 4096)
    return CSA2_ERR_UNSUPPORTED;
  if (n_rows == 0) return CSA2_OK;
  if (!scores || !n_valid || !pool_blocks || !workspace || !aligned16(workspace))
    return CSA2_ERR_INVALID_ARG;
  int64_t max_valid = 0;
  for (int r = 0; r < n_rows; ++r) {
    if (n_valid[r] < 0 || n_valid[r] > ld) return CSA2_ERR_INVALID_ARG;
    max_valid = std::max(max_valid, n_valid[r]);
  }
  if (ws_bytes < csa2_hsi_pool_workspace_bytes(n_rows, max_valid)) return CSA2_ERR_CAPACITY;
  const int64_t ld_b = hsi_ld_b(max_valid);
  float* bmax = static_cast<float*>(workspace);
  HsiParams* hp = new (std::nothrow) HsiParams();
  TopkParams* tp = new (std::nothrow) TopkParams();
  if (!hp || !tp) { delete hp; delete tp; return CSA2_ERR_OOM; }
  csa2_status_t st = CSA2_OK;
  for (int r0 = 0; r0 < n_rows && st == CSA2_OK; r0 += kHsiTab) {
    const int n = std::min(kHsiTab, n_rows - r0);
    std::memset(hp, 0, sizeof(HsiParams));
    hp->rows = n;
    hp->scores = scores + (int64_t)r0 * ld;
    hp->ld = ld;
    hp->bmax = bmax + (int64_t)r0 * ld_b;
    hp->ld_b = ld_b;
    for (int i = 0; i < n; ++i) hp->n[i] = n_valid[r0 + i];
    if (launch_block_max(*hp, S(stream)) != cudaSuccess) { st = CSA2_ERR_CUDA; break; }
    // the blocks with the highest block scores, ties to the lower block
    std::memset(tp, 0, sizeof(TopkParams));
    tp->scores = hp->bmax;
    tp->ld = ld_b;
    tp->rows = n;
    tp->k = max_blocks;
    tp->idx_out = pool_blocks + (int64_t)r0 * max_blocks;
    tp->formula = 0;
    for (int i = 0; i < n; ++i) tp->n_valid[i] = (n_valid[r0 + i] + kHsiBlock - 1) / kHsiBlock;
    if (launch_topk(*tp, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
  }
  delete hp;
  delete tp;
  return st;
}

size_t csa2_index_reindex_workspace_bytes(const csa2_cache_t* c, int32_t n_queries,
                                          int32_t max_blocks) {
  if (!c || n_queries < 0 || max_blocks <= 0) return 0;
  const int64_t slots = (int64_t)max_blocks * kHsiBlock;
  return (size_t)n_queries * ((size_t)slots * sizeof(float) + kKeyHistBinsHost * 4 +
                              (size_t)c->cfg.topk * 4) +
         topk_seg_bytes(n_queries, slots);
}

csa2_status_t csa2_index_topk_reindex_decode(const csa2_cache_t* c, int32_t nq, const void* q_idx,
                                             const float* w, const int32_t* seq_ids,
                                             const int32_t* pool_blocks, int32_t max_blocks,
                                             int32_t* topk_idx, float* topk_score,
                                             void* workspace, size_t ws_bytes,
                                             csa2_stream_t stream) {
  CSA2_RANGE();
  if (!c || nq < 0) return CSA2_ERR_INVALID_ARG;
  if (max_blocks <= 0 || max_blocks % 16 != 0 || max_blocks > 4096) return CSA2_ERR_UNSUPPORTED;
  if (nq == 0) return CSA2_OK;
  csa2_status_t st = check_decode_queries(c, nq, q_idx, w, seq_ids);
  if (st != CSA2_OK) return st;
  if (!pool_blocks || !topk_idx || !workspace || !aligned16(workspace)) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < csa2_index_reindex_workspace_bytes(c, nq, max_blocks)) return CSA2_ERR_CAPACITY;
  const int64_t slots = (int64_t)max_blocks * kHsiBlock;
  float* pscores = static_cast<float*>(workspace);
  uint32_t* key_hist = reinterpret_cast<uint32_t*>(pscores + (int64_t)nq * slots);
  int32_t* sel = reinterpret_cast<int32_t*>(key_hist + (int64_t)nq * kKeyHistBinsHost);
  uint32_t* seg_ws = reinterpret_cast<uint32_t*>(sel + (int64_t)nq * c->cfg.topk);
  const int k = c->cfg.topk;
  IndexParams* ip = new (std::nothrow) IndexParams();
  TopkParams* tp = new (std::nothrow) TopkParams();
  HsiParams* hp = new (std::nothrow) HsiParams();
  if (!ip || !tp || !hp) { delete ip; delete tp; delete hp; return CSA2_ERR_OOM; }
  const uint16_t* qb = static_cast<const uint16_t*>(q_idx);
  if (cudaMemsetAsync(key_hist, 0, (size_t)nq * kKeyHistBinsHost * 4, S(stream)) != cudaSuccess)
    st = CSA2_ERR_CUDA;
  // tiles of 32 blocks (256 slots) over bf16 keys, of 64 blocks (512 slots)
  // over MXFP4 keys; a last tile holds what remains of max_blocks (a
  // multiple of 16)
  const int blocks_per_tile = c->cfg.idx_layout == CSA2_IDX_MXFP4 ? 64 : 32;
  const int pool_tiles = (max_blocks + blocks_per_tile - 1) / blocks_per_tile;
  for (int q0 = 0; q0 < nq && st == CSA2_OK; q0 += kMaxIdxGroups) {
    const int n = std::min(kMaxIdxGroups, nq - q0);
    // ---- the pool positions' scores (indexer in pool mode)
    std::memset(ip, 0, sizeof(IndexParams));
    ip->w = w + (int64_t)q0 * kIdxHeads;
    ip->scores = pscores + (int64_t)q0 * slots;
    ip->ld = slots;
    ip->key_hist = key_hist + (int64_t)q0 * kKeyHistBinsHost;
    ip->pool = pool_blocks + (int64_t)q0 * max_blocks;
    ip->pool_blocks = max_blocks;
    ip->err = c->d_err;
    ip->nq = n;
    ip->qpg = 1;
    ip->n_groups = n;
    ip->ratio = c->cfg.ratio;
    ip->wait_cycles = c->wait_cycles;
    ip->inject = c->inject;
    ip->tile_prefix[0] = 0;
    for (int i = 0; i < n; ++i) {
      const int s = seq_ids ? seq_ids[q0 + i] : q0 + i;
      ip->entry_base[i] = c->off[s];
      ip->nvis[i] = (int32_t)c->len[s];
      ip->tile_prefix[i + 1] = ip->tile_prefix[i] + pool_tiles;
    }
    CUtensorMap tm_q;
    const uint16_t* qn = qb + (int64_t)q0 * kIdxHeads * kIdxDim;
    if (!make_map(&tm_q, qn, (uint64_t)n * kIdxHeads, kIdxDim, 64, 32)) {
      st = CSA2_ERR_CUDA;
      break;
    }
    const int grid = std::min(c->index_sms, ip->tile_prefix[n]);
    if (launch_index_any(c, *ip, tm_q, qn, grid, S(stream), true) != cudaSuccess) {
      st = CSA2_ERR_CUDA;
      break;
    }
    // ---- top-k over the pool slots (ties to the lower slot = lower entry)
    std::memset(tp, 0, sizeof(TopkParams));
    tp->scores = ip->scores;
    tp->ld = slots;
    tp->rows = n;
    tp->k = k;
    tp->idx_out = sel + (int64_t)q0 * k;
    tp->score_out = topk_score ? topk_score + (int64_t)q0 * k : nullptr;
    tp->key_hist = ip->key_hist;
    // a pool of at most two segments (16384 slots) is compacted by the row
    // kernel itself in one block-wide pass: one launch instead of two
    const bool use_seg = topk_segments(slots) > 2;
    tp->seg_ws = use_seg ? seg_ws + (size_t)q0 * topk_seg_bytes(1, slots) / sizeof(uint32_t)
                         : nullptr;
    tp->n_seg = use_seg ? topk_segments(slots) : 0;
    tp->formula = 0;
    tp->err = c->d_err;
    for (int i = 0; i < n; ++i) tp->n_valid[i] = slots;
    if (launch_topk(*tp, S(stream)) != cudaSuccess) { st = CSA2_ERR_CUDA; break; }
    // ---- pool slots back to entry indices
    std::memset(hp, 0, sizeof(HsiParams));
    hp->rows = n;
    hp->sel = tp->idx_out;
    hp->k = k;
    hp->pool = ip->pool;
    hp->pool_blocks = max_blocks;
    hp->out = topk_idx + (int64_t)q0 * k;
    hp->score_out = tp->score_out;
    hp->err = c->d_err;
    for (int i = 0; i < n; ++i) hp->n[i] = ip->nvis[i];
    if (launch_pool_map(*hp, S(stream)) != cudaSuccess) st = CSA2_ERR_CUDA;
  }
  delete ip;
  delete tp;
  delete hp;
  return st;
}

csa2_status_t csa2_swa_fp8_quantise(int64_t n_rows, const void* rows, uint8_t* codes, void* rope,
                                    uint8_t* scales, csa2_stream_t stream) {
  CSA2_RANGE();
  if (n_rows < 0) return CSA2_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (!rows || !codes || !rope || !scales || !aligned16(rows) || !aligned16(codes) ||
      !aligned16(rope) || (reinterpret_cast<uintptr_t>(scales) & 7u))
    return CSA2_ERR_INVALID_ARG;
  return cuda_status(launch_swa_fp8(static_cast<const uint16_t*>(rows), n_rows, codes,
                                    static_cast<uint16_t*>(rope), scales, S(stream)));
}

csa2_status_t csa2_get_device_error(const csa2_cache_t* c, csa2_stream_t stream,
                                    int32_t* device_status) {
  CSA2_RANGE();
  if (!c || !device_status) return CSA2_ERR_INVALID_ARG;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, c->d_err, sizeof(word), cudaMemcpyDeviceToHost, S(stream)) !=
          cudaSuccess ||
      cudaStreamSynchronize(S(stream)) != cudaSuccess)
    return CSA2_ERR_CUDA;
  if (word && cudaMemsetAsync(c->d_err, 0, sizeof(uint32_t), S(stream)) != cudaSuccess)
    return CSA2_ERR_CUDA;
  *device_status = (word & kErrTimeoutBit) ? CSA2_ERR_TIMEOUT
                   : (word & kErrIndexBit) ? CSA2_ERR_DEVICE
                                           : CSA2_OK;
  return CSA2_OK;
}

}  // extern "C"
