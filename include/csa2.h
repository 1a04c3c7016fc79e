/*
 * csa2.h -- C ABI of the CSA2 (Compressed Sparse Attention 2) attention step
 * over an FP4 global KV cache, for one GB300 (sm_103a) GPU.
 *
 * The method (sources are web pages; each declaration cites the passage that
 * defines the operation):
 *   [V41] "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *         (technical report, PaperTrace mirror)
 *   [V4B] blog reading of the DeepSeek-V4 report (gzher.com)
 *   [NDT] neshdevtech article on DeepSeek-V4.1-Flash
 *
 * One CSA2 group (a Full layer and the Reuse layers that follow it) owns one
 * global cache: per sequence, compressed main-KV entries (FP4 E2M1 codes plus
 * per-block scales) and indexer keys ([V41 sec 2.3.1], [NDT sec 3.1]).
 * Sliding-window (SWA) KV is per layer and is passed in by the caller.
 *
 * Conventions (every call):
 *   - "dev" pointers are CUDA device pointers owned by the caller; "host"
 *     pointers are host memory read before the call returns.  Device
 *     tensors are dense row-major and 16-byte aligned, else the call
 *     returns CSA2_ERR_INVALID_ARG.
 *   - bf16 tensors are passed as void* to raw 16-bit bf16 values.
 *   - Calls are stream-ordered on `stream` (a cudaStream_t; NULL = legacy
 *     default stream), never synchronise the device and never allocate
 *     device memory.  Scratch memory comes from the caller (`workspace`).
 *     The indexers, top-k and readout kernels are launched with programmatic
 *     stream serialisation: a launch may begin while the previous kernel in
 *     the stream finishes, but each waits for that kernel to complete before
 *     its first global memory access, so every read and write keeps its
 *     stream order (also inside captured CUDA graphs).
 *   - Errors found on the host return a status before anything is
 *     launched.  Errors found inside a kernel (a bounded wait that ran out,
 *     an index out of range) set a sticky device error word that
 *     csa2_get_device_error() reads.
 *   - Entry indices are positions in a sequence's list of compressed
 *     entries (not token positions).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* csa2_stream_t; /* a cudaStream_t */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned tensor      */
  CSA2_ERR_UNSUPPORTED = 2, /* configuration outside what the kernels support */
  CSA2_ERR_CAPACITY = 3,    /* append beyond a sequence's capacity, or a too  */
                            /* small workspace / cache buffer                 */
  CSA2_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed           */
  CSA2_ERR_OOM = 5,         /* reserved: the library itself never allocates   */
  CSA2_ERR_TIMEOUT = 6,     /* device error word: a bounded wait ran out      */
  CSA2_ERR_DEVICE = 7       /* device error word: bad index seen by a kernel  */
} csa2_status_t;

/* FP4 main-KV layouts.  [V41 sec 2.4.4] names both the OCP MXFP4 format
 * (E2M1 + one power-of-two UE8M0 scale per 32 channels) and the format it
 * selects for the main KV (E2M1 + one E4M3 scale per 16 channels, no global
 * scale; largest magnitude 448 * 6 = 2688).
 *   L32_UE8M0: scale byte = floor(log2(amax)) - 2 + 127 (OCP MX rule,
 *              clamped to [0, 254]); 256 B codes + 16 B scales per entry.
 *   L16_E4M3 : scale = E4M3(amax / 6), round to nearest even, saturating at
 *              448; 256 B codes + 32 B scales per entry.
 * Codes are E2M1 of x / scale, round to nearest even, saturating at 6, the
 * sign kept; two per byte, the even channel in the low nibble.             */
typedef enum { CSA2_KV_L32_UE8M0 = 0, CSA2_KV_L16_E4M3 = 1 } csa2_kv_layout_t;

/* Shapes of one CSA2 layer.  [V41 sec 4.2.1]: 64 query heads of dim 512,
 * 32 indexer heads of dim 128, top-k 512, window 128, ratio m = 2 (encoder)
 * or 1 (decoder).  Supported: head_dim 512, idx_dim 128, idx_heads 32,
 * n_heads 64 or 128, topk a multiple of 128 up to 2048,
 * 0 <= swa <= 128, 1 <= ratio <= 16.                                      */
typedef struct {
  int32_t n_heads;
  int32_t head_dim;
  int32_t idx_heads;
  int32_t idx_dim;
  int32_t topk;
  int32_t swa;
  int32_t ratio;
  int32_t layout; /* csa2_kv_layout_t */
  int32_t idx_layout; /* csa2_idx_layout_t */
} csa2_config_t;

/* Indexer-key storage.  CSA2_IDX_BF16: 128 bf16 channels (256 B/entry).
 * CSA2_IDX_MXFP4 ([V41 sec 2.4.4]: FP4 indexer queries and keys in OCP
 * MXFP4; the 68 B per key of [NDT sec 3.1]): E2M1 codes (64 B, even channel
 * in the low nibble) + one UE8M0 scale per 32 channels (4 B), the scale
 * rule of CSA2_KV_L32_UE8M0; the indexer then also rounds each query head
 * to the MXFP4 grid before scoring.  The tensor cores take the codes and
 * scales as they are (block-scaled MXFP4 MMAs, fp32 accumulation).        */
typedef enum { CSA2_IDX_BF16 = 0, CSA2_IDX_MXFP4 = 1 } csa2_idx_layout_t;

typedef struct csa2_cache csa2_cache_t; /* opaque host handle, one per group */

/* Device views of a cache, for inspection.  Entry e of sequence b is row
 * entry_offset[b] + e of every array.                                       */
typedef struct {
  uint8_t* codes;        /* dev [total, head_dim / 2]                         */
  uint8_t* scales;       /* dev [total, head_dim / group]                     */
  void* idx_k;           /* CSA2_IDX_BF16: dev bf16 [total, idx_dim], else NULL */
  int32_t* lengths;      /* dev [batch]: entries appended so far              */
  const int64_t* entry_offset; /* host [batch + 1]                           */
  int64_t total;         /* sum of capacities                                 */
  int32_t batch;
  int32_t group;         /* 32 or 16 channels per scale                       */
  uint8_t* idx_codes;    /* CSA2_IDX_MXFP4: dev [total, idx_dim / 2], else NULL */
  uint8_t* idx_scales;   /* CSA2_IDX_MXFP4: dev [total, idx_dim / 32], else NULL */
} csa2_cache_views_t;

int32_t csa2_version(void);
const char* csa2_status_string(csa2_status_t status);

/* ---- cache ------------------------------------------------------------- */

/* Bytes of device memory a cache for `batch` sequences with the given
 * per-sequence capacities (in compressed entries, host [batch]) needs.
 * Returns 0 for an invalid or unsupported configuration.                    */
size_t csa2_cache_bytes(const csa2_config_t* cfg, int32_t batch,
                        const int64_t* capacity);

/* Lays a cache out in caller-owned device memory `dev_mem` (`bytes` long,
 * 256-byte aligned) and zeroes its lengths on `stream`.  The handle (host
 * memory) is returned in *out.  The caller keeps dev_mem alive until
 * csa2_cache_destroy.  [V41 sec 2.3.1]: main KV and indexer K are shared by
 * every layer of the group, so one cache serves all of them.              */
csa2_status_t csa2_cache_create(const csa2_config_t* cfg, int32_t batch,
                                const int64_t* capacity, void* dev_mem,
                                size_t bytes, csa2_stream_t stream,
                                csa2_cache_t** out);

/* Frees the host handle only; the device memory stays the caller's. */
csa2_status_t csa2_cache_destroy(csa2_cache_t* cache);

/* Upper bound on the SMs that the indexer's persistent grid occupies for
 * this cache (n_sms = 0 or more than the GPU has: all of them, the default).
 * A caller that splits a decode batch into micro-batches on separate streams
 * leaves the other SMs to the latency-bound top-k and attention kernels of
 * the other micro-batch, which then run concurrently with the bandwidth-
 * bound indexer (the results do not depend on the setting).  Applies to
 * indexer launches made after it returns.  CSA2_ERR_INVALID_ARG for a NULL
 * cache or n_sms < 0.  The pages have no counterpart: this is a scheduling
 * knob of this implementation, not part of the method.                    */
csa2_status_t csa2_cache_set_index_sms(csa2_cache_t* cache, int32_t n_sms);

/* Upper bound, in SM clock cycles, on every bounded wait inside the
 * indexer and readout kernels launched for this cache after the call
 * (cycles = 0 restores the default of 2^31, about one second).  A wait that
 * runs out records CSA2_ERR_TIMEOUT in the device error word, waits (within
 * the same bound) for the copies its CTA has in flight, frees its tensor
 * memory and ends the kernel, so the context stays usable.
 * CSA2_ERR_INVALID_ARG for a NULL cache or cycles < 0.  The pages have no
 * counterpart: this is a watchdog of this implementation.                 */
csa2_status_t csa2_cache_set_wait_limit(csa2_cache_t* cache, int64_t cycles);

/* Fault injection for tests of the timeout path (the pages have no
 * counterpart).  CSA2_FAULT_INDEX_NO_KEY_LOADS: the indexers' producer warp
 * issues no key loads, so their MMA and epilogue waits run out with no copy
 * and no MMA in flight; the scores are then not written and the device
 * error word reads CSA2_ERR_TIMEOUT.  CSA2_FAULT_NONE switches it off.
 * Applies to launches made after the call.                                */
typedef enum { CSA2_FAULT_NONE = 0, CSA2_FAULT_INDEX_NO_KEY_LOADS = 1 } csa2_fault_t;
csa2_status_t csa2_cache_inject_fault(csa2_cache_t* cache, int32_t fault);

/* Empties every sequence (host lengths and, on `stream`, device lengths). */
csa2_status_t csa2_cache_reset(csa2_cache_t* cache, csa2_stream_t stream);

/* Entries appended so far to sequence `seq` (host-side count). */
csa2_status_t csa2_cache_length(const csa2_cache_t* cache, int32_t seq,
                                int64_t* n_entries);

csa2_status_t csa2_cache_views(const csa2_cache_t* cache,
                               csa2_cache_views_t* out);

/* ---- compress / append ------------------------------------------------- */

/* CSA2 compressor ([V41 sec 2.3]: no overlap between blocks, no positional
 * bias; pooling form of [V4B sec 4.2]): out[i, c] = sum_j softmax_j(z[j, c])
 * * c_tok[j, c] over the `ratio` tokens j of block i, in fp32 with a fixed
 * order.  At ratio 1 it is the identity ([NDT sec 3.3.2]).
 *   c_tok: dev bf16 [n_out * ratio, dim];  z_tok: dev fp32 [n_out * ratio,
 *   dim];  out: dev fp32 [n_out, dim].  dim must be a multiple of 16.     */
csa2_status_t csa2_compress(int32_t ratio, int64_t n_out, int32_t dim,
                            const void* c_tok, const float* z_tok, float* out,
                            csa2_stream_t stream);

/* Quantises compressed entries to the cache's FP4 layout and appends them
 * with their indexer keys ([V41 sec 2.4.4]: FP4 main KV cache, quantised
 * after RoPE; [V41 sec 2.3]: indexer K is projected from the main KV by the
 * caller).  Rows of `entries` / `idx_k` are grouped by sequence in the order
 * of seq_ids: n_new[i] rows for sequence seq_ids[i].
 *   seq_ids, n_new: host [n_seqs];  entries: dev fp32 [sum n_new, head_dim];
 *   idx_k: dev bf16 [sum n_new, idx_dim].
 * Returns CSA2_ERR_CAPACITY (nothing written) if a sequence would overflow. */
csa2_status_t csa2_append_entries(csa2_cache_t* cache, int32_t n_seqs,
                                  const int32_t* seq_ids, const int32_t* n_new,
                                  const float* entries, const void* idx_k,
                                  csa2_stream_t stream);

/* Fused compress + quantise + append of whole blocks of tokens: n_tok[i] (a
 * multiple of the ratio) tokens of sequence seq_ids[i] become n_tok[i] /
 * ratio entries, bit-identical to csa2_compress followed by
 * csa2_append_entries.  The unfinished tail of a block stays with the caller
 * (it is not yet causally visible, [V4B sec 4.3]).
 *   c_tok: dev bf16 [sum n_tok, head_dim];  z_tok: dev fp32 [sum n_tok,
 *   head_dim];  idx_k: dev bf16 [sum n_tok / ratio, idx_dim];
 *   entries_out: nullable dev fp32 [sum n_tok / ratio, head_dim].          */
csa2_status_t csa2_append_tokens(csa2_cache_t* cache, int32_t n_seqs,
                                 const int32_t* seq_ids, const int32_t* n_tok,
                                 const void* c_tok, const float* z_tok,
                                 const void* idx_k, float* entries_out,
                                 csa2_stream_t stream);

/* ---- indexer + top-k --------------------------------------------------- */

/* Workspace bytes csa2_index_topk_decode / _prefill need for n_queries
 * queries against this cache (fp32 scores for every visible entry of every
 * query plus selection state).                                            */
size_t csa2_index_workspace_bytes(const csa2_cache_t* cache, int32_t n_queries);

/* Score-key histogram.  Scores are ordered through a 32-bit key: the fp32
 * bit pattern with the sign bit set for non-negative values and all bits
 * inverted for negative ones (-0 counts as +0), so that keys compare like
 * the scores.  key_hist[r, b] (uint32, 2048 bins per row) counts the valid
 * scores of row r whose key has b in its top 11 bits.  csa2_index_scores_*
 * can produce it while scoring; csa2_topk then skips its own first pass.    */

/* Index scores only (the scoring step of csa2_index_topk_decode, for callers
 * that select on their own or time the steps apart): for decode query q,
 * scores[q * ld + s] = sum_h w[q, h] * ReLU(q_idx[q, h] . K_I[s]) for every
 * entry s of its sequence ([V4B sec 4.1]); entries past a sequence's length
 * are left untouched.
 *   scores: dev fp32 [n_queries, ld], ld >= the longest sequence's length
 *   and a multiple of 4;  key_hist: nullable dev uint32 [n_queries, 2048],
 *   overwritten with the score-key histogram of each row;  other arguments
 *   as for csa2_index_topk_decode.                                         */
csa2_status_t csa2_index_scores_decode(const csa2_cache_t* cache,
                                       int32_t n_queries, const void* q_idx,
                                       const float* w, const int32_t* seq_ids,
                                       float* scores, int64_t ld,
                                       uint32_t* key_hist, csa2_stream_t stream);

/* Full-mode selection for decode queries, one query per sequence, each the
 * newest token of its sequence so every appended entry is visible.
 * Index score ([V4B sec 4.1]):  I[q, s] = sum_h w[q, h] * ReLU(q_idx[q, h] .
 * K_I[s]), fp32; then the top-k entries ([V41 sec 4.2.1]: k = 512) with
 * ties to the lower index, listed in ascending index order, padded with -1
 * when fewer than k entries exist.
 *   q_idx: dev bf16 [n_queries, idx_heads, idx_dim];  w: dev fp32
 *   [n_queries, idx_heads];  seq_ids: host [n_queries] (NULL: query i reads
 *   sequence i);  topk_idx: dev int32 [n_queries, topk];  topk_score:
 *   nullable dev fp32 [n_queries, topk] (the scores of topk_idx, 0 for -1).
 * A Reuse layer ([V41 sec 2.3.1]) calls nothing here: it passes the Full
 * layer's topk_idx to csa2_sparse_attn_decode unchanged.                  */
csa2_status_t csa2_index_topk_decode(const csa2_cache_t* cache,
                                     int32_t n_queries, const void* q_idx,
                                     const float* w, const int32_t* seq_ids,
                                     int32_t* topk_idx, float* topk_score,
                                     void* workspace, size_t workspace_bytes,
                                     csa2_stream_t stream);

/* Full-mode selection for queries at any token positions of any sequences
 * (decode queries and prefill chunks of several sequences in one call):
 * query i belongs to sequence seq_of_q[i] and sits at absolute token
 * position q_pos[i]; it sees entry s iff (s + 1) * ratio - 1 <= q_pos[i]
 * and s is appended ([V41 sec 2.3.2] "causally visible"; [V4B sec 4.3]).
 * Same score, top-k and output rules as csa2_index_topk_decode (a decode
 * query is q_pos = its sequence's last token, seeing every entry).
 *   seq_of_q: host [n_queries] (NULL: query i reads sequence i);  q_pos:
 *   host int64 [n_queries], >= 0;  other arguments and the workspace as for
 *   csa2_index_topk_decode.  One query per tile of the tensor-core indexer:
 *   a long chunk of consecutive positions of one sequence is scored faster
 *   by csa2_index_topk_prefill (eight queries per tile).                   */
csa2_status_t csa2_index_topk(const csa2_cache_t* cache, int32_t n_queries,
                              const void* q_idx, const float* w, const int32_t* seq_of_q,
                              const int64_t* q_pos, int32_t* topk_idx, float* topk_score,
                              void* workspace, size_t workspace_bytes, csa2_stream_t stream);

/* The same selection as csa2_index_topk_decode for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is an
 * integration entry point, not part of the method.
 *
 * Some callers cannot call cudaMalloc or hand over a workspace: serving
 * runtimes that own every byte of device memory through their own pool and
 * hand kernels no scratch (so that the memory budget is fixed and nothing
 * fragments it), latency-critical loops in which an allocation, which may
 * synchronise the device, is not acceptable, and plain C hosts that want a
 * single call with nothing to size or free.  This entry point keeps its
 * scratch (fp32 scores and score-key histograms) in a fixed array inside
 * the library, CSA2_STATIC_SCRATCH_BYTES long.  A GPU holds that array from
 * the first use of the library's device code on it (at the latest the first
 * call of this entry point) until the process exits.
 *   - Requests needing more than the array (n_queries * (4 * ld + 8192)
 *     bytes, ld = the longest capacity rounded up to a multiple of 4) return
 *     CSA2_ERR_CAPACITY and launch nothing.
 *   - A call made while `stream` is not being captured looks the array's
 *     device address up (cudaGetSymbolAddress) with the current device; the
 *     first call on a device does this set-up, so make it before any stream
 *     capture: a first call during a capture returns CSA2_ERR_UNSUPPORTED
 *     and launches nothing.
 *   - Every call uses the same array, which keeps what the last call left
 *     there (each call first zeroes the histograms it accumulates into, on
 *     `stream`); two calls that overlap on the GPU (different streams
 *     without ordering between them) race, calls on one stream are safe.
 *   - Allocates nothing: no cudaMalloc / cudaFree, no host heap.
 * Arguments and outputs as for csa2_index_topk_decode.                     */
#define CSA2_STATIC_SCRATCH_BYTES ((size_t)48 << 20)
csa2_status_t csa2_index_topk_decode_static(const csa2_cache_t* cache,
                                            int32_t n_queries,
                                            const void* q_idx, const float* w,
                                            const int32_t* seq_ids,
                                            int32_t* topk_idx,
                                            float* topk_score,
                                            csa2_stream_t stream);

/* Full-mode selection for a prefill chunk of one sequence: query i is the
 * token at absolute position pos0 + i and sees entry s iff its block is
 * complete, (s + 1) * ratio - 1 <= pos0 + i ([V41 sec 2.3.2] "causally
 * visible"; [V4B sec 4.3]).  Same score, top-k and output rules as decode.
 *   q_idx: dev bf16 [n_queries, idx_heads, idx_dim];  w: dev fp32
 *   [n_queries, idx_heads];  topk_idx: dev int32 [n_queries, topk];
 *   workspace: dev, 16-byte aligned, at least
 *   csa2_index_prefill_workspace_bytes(cache, seq, n_queries) bytes (else
 *   CSA2_ERR_CAPACITY): the scores, and with bf16 indexer keys the score-key
 *   histograms the indexer builds for the top-k.                           */
csa2_status_t csa2_index_topk_prefill(const csa2_cache_t* cache, int32_t seq,
                                      int32_t n_queries, int64_t pos0,
                                      const void* q_idx, const float* w,
                                      int32_t* topk_idx, float* topk_score,
                                      void* workspace, size_t workspace_bytes,
                                      csa2_stream_t stream);

/* Workspace bytes of csa2_index_topk_prefill for n_queries queries of
 * sequence seq: n_queries * 4 * ld (ld = the sequence's capacity rounded up
 * to a multiple of 4), plus n_queries * 8192 with bf16 indexer keys.  0 for
 * invalid arguments.                                                       */
size_t csa2_index_prefill_workspace_bytes(const csa2_cache_t* cache, int32_t seq,
                                          int32_t n_queries);

/* Index scores only for a prefill chunk (the scoring step of
 * csa2_index_topk_prefill): query i at position pos0 + i, scores[i * ld + s]
 * for every entry s visible to it ((s + 1) * ratio - 1 <= pos0 + i);
 * other entries are left untouched.  Eight consecutive queries share each
 * tile of indexer keys on the tensor cores (four with MXFP4 keys).
 *   scores: dev fp32 [n_queries, ld], ld >= the sequence's length and a
 *   multiple of 4;  key_hist: NULL or dev uint32 [n_queries, 2048], 16-byte
 *   aligned: zeroed, then query i's row counts its visible scores by the
 *   top 11 bits of their order-preserving key (the histogram csa2_topk
 *   takes); bf16 indexer keys only (MXFP4 keys: CSA2_ERR_UNSUPPORTED);
 *   other arguments as for csa2_index_topk_prefill.                        */
csa2_status_t csa2_index_scores_prefill(const csa2_cache_t* cache, int32_t seq,
                                        int32_t n_queries, int64_t pos0,
                                        const void* q_idx, const float* w,
                                        float* scores, int64_t ld,
                                        uint32_t* key_hist, csa2_stream_t stream);

/* ---- Hierarchical Sparse Indexer and Reindex mode ([V41 sec 2.3.2]) -----
 * The first Full layer of the decoder also picks a candidate pool: every
 * block of 8 consecutive entries gets the maximum of its entries' index
 * scores, and the max_blocks blocks with the highest block scores are kept
 * (ties to the lower block index); [V41 sec 4.2.1]: 2048 blocks x 8 =
 * 16384 candidates.  A later Reindex layer scores only the pool with its
 * own indexer query and selects its own top-k inside it.                  */

/* Workspace bytes of csa2_hsi_pool. */
size_t csa2_hsi_pool_workspace_bytes(int32_t n_rows, int64_t max_valid);

/* Candidate pool from a Full layer's scores: row r has n_valid[r] scores at
 * scores + r * ld (the scores csa2_index_scores_decode writes).
 *   block: must be 8;  max_blocks: a multiple of 16, at most 4096;
 *   pool_blocks: dev int32 [n_rows, max_blocks], the kept block indices in
 *   ascending order, -1 padded;  n_valid: host int64 [n_rows].            */
csa2_status_t csa2_hsi_pool(int32_t n_rows, const float* scores, int64_t ld,
                            const int64_t* n_valid, int32_t block,
                            int32_t max_blocks, int32_t* pool_blocks,
                            void* workspace, size_t workspace_bytes,
                            csa2_stream_t stream);

/* Workspace bytes of csa2_index_topk_reindex_decode. */
size_t csa2_index_reindex_workspace_bytes(const csa2_cache_t* cache,
                                          int32_t n_queries, int32_t max_blocks);

/* Reindex-mode selection for decode queries: the index score of [V4B sec
 * 4.1] with this layer's q_idx / w, over the entries of the query's pool
 * blocks only (blocks of 8, entries past the sequence excluded), then the
 * top-k of those with ties to the lower entry, ascending, -1 padded.
 *   pool_blocks: dev int32 [n_queries, max_blocks] from csa2_hsi_pool;
 *   other arguments as for csa2_index_topk_decode.                          */
csa2_status_t csa2_index_topk_reindex_decode(const csa2_cache_t* cache,
                                             int32_t n_queries, const void* q_idx,
                                             const float* w, const int32_t* seq_ids,
                                             const int32_t* pool_blocks,
                                             int32_t max_blocks, int32_t* topk_idx,
                                             float* topk_score, void* workspace,
                                             size_t workspace_bytes,
                                             csa2_stream_t stream);

/* Workspace bytes with which csa2_topk splits each row's candidate search
 * over several CTAs (used when key_hist is given and rows hold more than
 * 16384 scores), for n_rows rows of at most max_valid scores.  A smaller
 * workspace (or none) is allowed: the selection is the same, one CTA per
 * row.                                                                      */
size_t csa2_topk_workspace_bytes(int32_t n_rows, int64_t max_valid);

/* Stand-alone top-k over caller scores (the selection step of the indexer):
 * row r has n_valid[r] fp32 scores at scores + r * ld; the k largest are
 * returned, ties to the lower index, ascending index order, -1 padded.  -0
 * and +0 compare equal (a selected -0 is reported as +0); NaN is not
 * allowed.
 *   scores: dev fp32;  n_valid: host int64 [n_rows];  key_hist: nullable
 *   dev uint32 [n_rows, 2048], the score-key histogram of each row if the
 *   caller has it (see above), which saves one pass over the scores;
 *   idx_out: dev int32 [n_rows, k];  score_out: nullable dev fp32
 *   [n_rows, k].  k <= 4096.                                                */
csa2_status_t csa2_topk(int32_t n_rows, const float* scores, int64_t ld,
                        const int64_t* n_valid, int32_t k,
                        const uint32_t* key_hist, int32_t* idx_out,
                        float* score_out, void* workspace,
                        size_t workspace_bytes, csa2_stream_t stream);

/* ---- bf16-rounded index scores ([V4B sec 7]: the index scores are
 * quantised from FP32 to BF16 so that the top-k selector runs faster, with
 * a reported recall of 99.7% of the KV entries the FP32 selection keeps).
 * A score is the fp32 score of csa2_index_scores_decode rounded to the
 * nearest bf16 value (ties to even); the selection rule is unchanged (the
 * k largest, ties -- now frequent -- to the lower index).                  */

/* Scores as bf16: scores is dev uint16 [n_queries, ld] (bf16 bits), ld a
 * multiple of 8; key_hist (nullable) is the histogram of the rounded
 * scores' keys.  Other arguments as for csa2_index_scores_decode.          */
csa2_status_t csa2_index_scores_decode_bf16(const csa2_cache_t* cache,
                                            int32_t n_queries, const void* q_idx,
                                            const float* w, const int32_t* seq_ids,
                                            uint16_t* scores, int64_t ld,
                                            uint32_t* key_hist, csa2_stream_t stream);

/* csa2_topk over bf16 scores (dev uint16 [n_rows, ld]); score_out (nullable
 * dev fp32) receives the selected bf16 values.  Same workspace.           */
csa2_status_t csa2_topk_bf16(int32_t n_rows, const uint16_t* scores, int64_t ld,
                             const int64_t* n_valid, int32_t k,
                             const uint32_t* key_hist, int32_t* idx_out,
                             float* score_out, void* workspace,
                             size_t workspace_bytes, csa2_stream_t stream);

/* csa2_index_topk_decode on bf16-rounded scores; the same workspace size
 * (csa2_index_workspace_bytes) suffices.                                   */
csa2_status_t csa2_index_topk_decode_bf16(const csa2_cache_t* cache,
                                          int32_t n_queries, const void* q_idx,
                                          const float* w, const int32_t* seq_ids,
                                          int32_t* topk_idx, float* topk_score,
                                          void* workspace, size_t workspace_bytes,
                                          csa2_stream_t stream);

/* ---- sparse attention -------------------------------------------------- */

/* Workspace bytes of csa2_sparse_attn_decode for n_queries queries: a small
 * constant, since the two-CTA split keeps its partial states on chip and a
 * workspace only opts in to it. */
size_t csa2_sparse_attn_workspace_bytes(const csa2_cache_t* cache,
                                        int32_t n_queries);

/* Decode readout of one layer ([V4B sec 4.1] shared-KV MQA: the selected
 * compressed entries are both key and value; [V4B sec 4.3] and [NDT sec
 * 3.3.1]: the window rows join the same softmax): for query q and head h,
 *   l_j = scale * q[q, h] . kv_j   over j in {selected entries} U {window},
 *   out[q, h] = sum_j softmax(l)_j kv_j,   lse[q, h] = ln sum_j exp(l_j),
 * with the selected entries dequantised from FP4 on chip.  Full and Reuse
 * layers make the same call; a Reuse layer passes its group's topk_idx.
 *   q: dev bf16 [n_queries, n_heads, head_dim];  swa_kv: dev bf16
 *   [n_queries, swa, head_dim], the first swa_len[q] rows of query q are its
 *   window;  swa_len: nullable dev int32 [n_queries] (NULL: all swa rows);
 *   topk_idx: dev int32 [n_queries, topk] (-1 = unused slot);  seq_ids: host
 *   [n_queries] or NULL (query i reads sequence i);  out: dev bf16
 *   [n_queries, n_heads, head_dim];  lse: nullable dev fp32 [n_queries,
 *   n_heads];  workspace: nullable dev buffer of at least
 *   csa2_sparse_attn_workspace_bytes(cache, n_queries) bytes (not written)
 *   -- with it a small batch spreads each query's candidates over a cluster
 *   of two CTAs whose partial softmax states are merged exactly on chip (the
 *   output is the same function; without it one CTA per query does all the
 *   work).  An index >= the
 *   sequence's length is skipped and sets CSA2_ERR_DEVICE in the device
 *   error word.                                                             */
csa2_status_t csa2_sparse_attn_decode(const csa2_cache_t* cache,
                                      int32_t n_queries, const int32_t* seq_ids,
                                      const void* q, const void* swa_kv,
                                      const int32_t* swa_len,
                                      const int32_t* topk_idx, float scale,
                                      void* out, float* lse, void* workspace,
                                      size_t workspace_bytes,
                                      csa2_stream_t stream);

/* Prefill readout of one layer for a chunk of sequence `seq`: query i sits
 * at absolute position p = pos0 + i and its window is the token rows of
 * positions [max(swa_pos0, p - swa + 1), p] ([V41 sec 3.2.2]: a replay that
 * starts at swa_pos0 truncates the window there).
 *   q: dev bf16 [n_queries, n_heads, head_dim];  swa_kv: dev bf16
 *   [n_swa_rows, head_dim], row r holds the token at position swa_pos0 + r
 *   (requires pos0 + n_queries - 1 - swa_pos0 < n_swa_rows and
 *   swa_pos0 <= pos0);  topk_idx: dev int32 [n_queries, topk];  out, lse as
 *   for decode.                                                            */
csa2_status_t csa2_sparse_attn_prefill(const csa2_cache_t* cache, int32_t seq,
                                       int32_t n_queries, int64_t pos0,
                                       const void* q, const void* swa_kv,
                                       int64_t swa_pos0, int64_t n_swa_rows,
                                       const int32_t* topk_idx, float scale,
                                       void* out, float* lse,
                                       csa2_stream_t stream);

/* ---- readout epilogue variants ([V4B sec 4.3]) --------------------------
 * Both are off when the options pointer is NULL or the struct is zeroed.
 *   sink: nullable dev fp32 [n_heads], a per-head logit z'_h in the units of
 *     l_j (scale * q . kv); exp(z'_h) joins the softmax denominator, so a
 *     head's weights sum to less than 1 (the sink has no value):
 *     out = sum_j exp(l_j) kv_j / (sum_j exp(l_j) + exp(z'_h)), and lse is
 *     the log of that whole denominator (z'_h alone when nothing is
 *     selected).
 *   rope_out: 1 rotates the last 64 channels of each output row by the
 *     RoPE angle of position -i (channel pairs (448 + 2t, 449 + 2t), angle
 *     -i * rope_base^(-2t / 64)), so that the output carries relative
 *     position; i is rope_pos[q] (decode: dev int64 [n_queries], required)
 *     or pos0 + q (prefill).  rope_base: 0 means 10000.                    */
typedef struct {
  const float* sink;
  const int64_t* rope_pos;
  int32_t rope_out;
  double rope_base;
  /* FP8 window rows (all three set, or none): the rows of swa_kv in the
   * format of csa2_swa_fp8_quantise -- E4M3 codes [rows, 448], bf16 RoPE
   * channels [rows, 64], UE8M0 scales [rows, 8], the same row order as
   * swa_kv (which is then ignored and may be NULL).                       */
  const uint8_t* swa_codes;
  const void* swa_rope;
  const uint8_t* swa_scales;
} csa2_attn_opts_t;

/* FP8 window rows ([V41 sec 2.4.4]: the SWA KV cache stays FP8; the row is
 * the V4 FP8 entry of [NDT sec 3.1]: 448 + 128 + 8 = 584 bytes): for each
 * bf16 row of 512 channels, channels 0-447 as E4M3 codes with one UE8M0
 * scale per 64 channels (OCP MX rule for E4M3 elements: exponent of the
 * block's largest magnitude minus 8; codes of x / scale, nearest even,
 * saturating at 448), channels 448-511 (RoPE) kept as bf16, scale byte 7
 * zero.
 *   rows: dev bf16 [n_rows, 512];  codes: dev u8 [n_rows, 448];  rope: dev
 *   bf16 [n_rows, 64];  scales: dev u8 [n_rows, 8].  All 16-byte aligned
 *   (scales: 8).                                                           */
csa2_status_t csa2_swa_fp8_quantise(int64_t n_rows, const void* rows, uint8_t* codes,
                                    void* rope, uint8_t* scales, csa2_stream_t stream);

/* csa2_sparse_attn_decode with epilogue options (NULL: none).           */
csa2_status_t csa2_sparse_attn_decode_ex(const csa2_cache_t* cache,
                                         int32_t n_queries, const int32_t* seq_ids,
                                         const void* q, const void* swa_kv,
                                         const int32_t* swa_len,
                                         const int32_t* topk_idx, float scale,
                                         void* out, float* lse, void* workspace,
                                         size_t workspace_bytes,
                                         const csa2_attn_opts_t* opts,
                                         csa2_stream_t stream);

/* Decode readout of n_layers layers of one group in one launch: the
 * layers share the cache, the queries' sequences and windows' geometry
 * (seq_ids, swa_len) and the selection (topk_idx, e.g. a Full layer and its
 * Reuse layers, [V41 sec 2.3.1]), each has its own queries, window rows,
 * outputs and epilogue options.  Layer l's out / lse are those of
 * csa2_sparse_attn_decode_ex with q[l], swa_kv[l], out[l], lse[l], opts[l]
 * -- bit for bit when both launches split a query's candidates over the
 * same number of CTAs (with a workspace the two-CTA split follows the
 * launch's CTA count, so a launch of several layers may not split where one
 * of a single layer does, and then differ in the last bits); one launch lets the
 * layers' CTAs fill the SMs without a kernel boundary between the layers.
 *   n_layers: 1 .. CSA2_MAX_ATTN_LAYERS;  q, out: host arrays of n_layers
 *   device pointers;  swa_kv: host array of n_layers device pointers
 *   (entries NULL for FP8 windows), or NULL when there is no window;  lse:
 *   host array of n_layers nullable device pointers, or NULL;  opts: host
 *   array of n_layers nullable option pointers, or NULL -- the output RoPE
 *   settings (rope_out, rope_pos, rope_base) must be the same in every
 *   layer, else CSA2_ERR_INVALID_ARG;  other arguments as for
 *   csa2_sparse_attn_decode (the workspace's two-CTA split counts the CTAs
 *   of all layers).                                                        */
#define CSA2_MAX_ATTN_LAYERS 8
csa2_status_t csa2_sparse_attn_decode_layers(const csa2_cache_t* cache, int32_t n_layers,
                                             int32_t n_queries, const int32_t* seq_ids,
                                             const void* const* q,
                                             const void* const* swa_kv,
                                             const int32_t* swa_len,
                                             const int32_t* topk_idx, float scale,
                                             void* const* out, float* const* lse,
                                             void* workspace, size_t workspace_bytes,
                                             const csa2_attn_opts_t* const* opts,
                                             csa2_stream_t stream);

/* csa2_sparse_attn_prefill with epilogue options (NULL: none).          */
csa2_status_t csa2_sparse_attn_prefill_ex(const csa2_cache_t* cache, int32_t seq,
                                          int32_t n_queries, int64_t pos0,
                                          const void* q, const void* swa_kv,
                                          int64_t swa_pos0, int64_t n_swa_rows,
                                          const int32_t* topk_idx, float scale,
                                          void* out, float* lse,
                                          const csa2_attn_opts_t* opts,
                                          csa2_stream_t stream);

/* Prefill readout of n_layers layers of one group in one launch, as
 * csa2_sparse_attn_decode_layers is for decode: layer l's out / lse are
 * exactly those of csa2_sparse_attn_prefill_ex with q[l], swa_kv[l], out[l],
 * lse[l], opts[l]; the chunk (seq, pos0, n_queries), the window rows'
 * geometry (swa_pos0, n_swa_rows) and topk_idx are shared; the layers'
 * CTAs fill the SMs without a launch boundary between the layers.  Arrays
 * as for csa2_sparse_attn_decode_layers (the output RoPE base the same in
 * every layer).                                                           */
csa2_status_t csa2_sparse_attn_prefill_layers(const csa2_cache_t* cache, int32_t seq,
                                              int32_t n_layers, int32_t n_queries,
                                              int64_t pos0, const void* const* q,
                                              const void* const* swa_kv, int64_t swa_pos0,
                                              int64_t n_swa_rows, const int32_t* topk_idx,
                                              float scale, void* const* out,
                                              float* const* lse,
                                              const csa2_attn_opts_t* const* opts,
                                              csa2_stream_t stream);

/* ---- errors ------------------------------------------------------------ */

/* Reads and clears the cache's sticky device error word (synchronises
 * `stream`).  *device_status receives CSA2_OK, CSA2_ERR_TIMEOUT or
 * CSA2_ERR_DEVICE.                                                          */
csa2_status_t csa2_get_device_error(const csa2_cache_t* cache,
                                    csa2_stream_t stream,
                                    int32_t* device_status);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
