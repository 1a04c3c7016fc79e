/*
 * csa2_oracle.h -- CPU oracle of the CSA2 attention step over an FP4 global
 * KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path and is deliberately slow: plain loops, no blocking, fp64
 * accumulation for real-valued results, and fp32 exactly where a floating
 * point value decides an integer (a quantised code, a top-k index set).
 *
 * Citations name the page and the section / equation they follow:
 *  [V41]  "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
 *         (PaperTrace mirror of the technical report)
 *  [V4B]  blog reading of the DeepSeek-V4 report (gzher.com), section 4
 *  [NDT]  neshdevtech article on DeepSeek-V4.1-Flash
 *
 * Layout codes (independent of the CUDA library's enum, same meaning):
 *   0 = E2M1 codes + one UE8M0 (power-of-two) scale per 32 channels
 *   1 = E2M1 codes + one E4M3 scale per 16 channels
 * Codes are packed two per byte, even channel in the low nibble; the scales
 * of an entry are stored in a separate array [n, dim / group].
 *
 * bf16 tensors are passed as their uint16 bit patterns.
 *
 * Parity unpinned: the E4M3 / UE8M0 scale-selection rules (the pages name the
 * formats, not how a block's scale is chosen; the rules here are the NVFP4 /
 * OCP-MX readings).
 */
#ifndef CSA2_ORACLE_H
#define CSA2_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int    orc_num_threads(void);

/* ---- FP4 / FP8 codec  [V41 sec 2.4.4] ---------------------------------- */
float  orc_e2m1_value(int code);          /* code 0..15                        */
int    orc_e2m1_encode(float v);          /* nearest, ties to even, saturating */
float  orc_e4m3_value(int byte);          /* NaN for 0x7f / 0xff               */
int    orc_e4m3_encode(float v);          /* v >= 0: nearest, ties even, <=448 */
float  orc_ue8m0_value(int byte);         /* 2^(byte-127), NaN for 0xff        */
int    orc_ue8m0_for_amax(float amax);    /* OCP MX shared-exponent rule       */
int    orc_group(int layout);
int    orc_ue8m0_for_amax_e4m3(float amax);
void   orc_swa_fp8_quantise(int64_t n, const uint16_t* rows, uint8_t* codes, uint16_t* rope,
                            uint8_t* scales);
void   orc_swa_fp8_dequantise(int64_t n, const uint8_t* codes, const uint16_t* rope,
                              const uint8_t* scales, float* out);             /* 32 or 16                          */
void   orc_quantise(int64_t n, int dim, int layout, const float* x,
                    uint8_t* codes, uint8_t* scales);
void   orc_dequantise(int64_t n, int dim, int layout, const uint8_t* codes,
                      const uint8_t* scales, float* out);
double orc_entry_bytes(int dim, int layout); /* payload + scale bytes        */
double orc_bytes_per_token(int n_layers, const int* ratio,
                           const double* bytes_per_entry);

/* ---- compressor  [V41 sec 2.3], [V4B sec 4.2 pooling form] -------------- */
float  orc_expf(float x);
void   orc_compress(int64_t n_out, int m, int dim, const uint16_t* c_bf16,
                    const float* z, float* out);

/* ---- indexer and top-k  [V4B sec 4.1 index score], [V41 sec 4.2.1] ------- */
void   orc_index_scores(int64_t n, int heads, int d, const uint16_t* k_bf16,
                        const uint16_t* q_bf16, const float* w, double* out);
float  orc_bf16_round(float x);
void   orc_bf16_round_n(int64_t n, const float* in, float* out);
int    orc_topk(int64_t n, const float* scores, int k, int32_t* idx_out);

/* ---- sparse shared-KV attention with SWA  [V4B sec 4.1/4.3], [NDT 3.3.1] - */
void   orc_sparse_attention(int heads, int dim, int layout,
                            const uint16_t* q_bf16,
                            const uint8_t* codes, const uint8_t* scales,
                            int64_t n_ent, int n_idx, const int32_t* idx,
                            int n_swa, const uint16_t* swa_bf16, float scale,
                            uint16_t* out_bf16, double* out_f64, double* lse);

#ifdef __cplusplus
}
#endif
#endif
