/*
 * csa2_oracle.c -- CPU oracle of the CSA2 attention step over an FP4 global
 * KV cache.  TEST INFRASTRUCTURE ONLY (see csa2_oracle.h): the product path
 * never loads it.  Build with -ffp-contract=off so that every fp32 operation
 * below is rounded exactly where it is written.
 */
#include "csa2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* FP4 / FP8 codec.  [V41 sec 2.4.4]: main KV is E2M1 with a per-block scale,
 * no second-level global scale; largest magnitude 448 * 6 = 2688 (E4M3
 * scale).  The OCP MX variant (E2M1 + UE8M0 per 32) is the "MXFP4" the same
 * section names.                                                             */

/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal (0, 0.5).                                                        */
float orc_e2m1_value(int code) {
  int e = (code >> 1) & 3, m = code & 1;
  float mag = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
  return (code & 8) ? -mag : mag;
}

/* Nearest representable magnitude by exhaustive search; an exact tie goes to
 * the even code; magnitudes above 6 saturate to 6.  Sign is carried over.    */
int orc_e2m1_encode(float v) {
  double a = fabs((double)v);
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(a - (double)orc_e2m1_value(c));
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) { bd = d; best = c; }
  }
  if (a > 6.0) best = 7;
  return best | (signbit(v) ? 8 : 0);
}

/* E4M3 (OCP FP8): 4 exponent bits (bias 7), 3 mantissa bits, exponent 0 is
 * subnormal, 0x7f / 0xff are NaN, no infinities.                             */
float orc_e4m3_value(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  float mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexpf((float)m, -9);
  else mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return s ? -mag : mag;
}

/* Non-negative v only (a scale): nearest finite E4M3 value by search, ties to
 * the even code, saturating at 448.                                          */
int orc_e4m3_encode(float v) {
  double a = (double)v;
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c <= 0x7e; ++c) {
    double d = fabs(a - (double)orc_e4m3_value(c));
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) { bd = d; best = c; }
  }
  if (a > 448.0) best = 0x7e;
  return best;
}

float orc_ue8m0_value(int byte) {
  if (byte == 255) return NAN;
  return ldexpf(1.0f, byte - 127);
}

/* OCP MX: shared exponent = floor(log2(amax)) - emax(E2M1) with emax = 2,
 * stored biased by 127 and clamped to the finite UE8M0 range.  amax = 0 takes
 * the smallest scale.                                                         */
int orc_ue8m0_for_amax(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e2;
  frexp((double)amax, &e2);          /* amax = f * 2^e2, f in [0.5, 1) */
  int b = (e2 - 1) - 2 + 127;
  if (b < 0) b = 0;
  if (b > 254) b = 254;
  return b;
}

/* FP8 window rows [V41 sec 2.4.4: the SWA KV cache stays FP8; the V4 FP8
 * row of the cache breakdown (NDT sec 3.1, the PaperTrace reading of V4):
 * 448 non-RoPE channels in FP8, 64 RoPE channels in bf16, 8 bytes of
 * scale].  Reading: E4M3 codes with one UE8M0 scale per 64 channels by the
 * OCP MX rule for E4M3 elements (shared exponent floor(log2 amax) - 8; a
 * quotient above 448 saturates), byte 7 of the scales unused; the RoPE
 * channels keep their bf16 bits.  584 bytes per row.                       */
int orc_ue8m0_for_amax_e4m3(float amax) {
  if (!(amax > 0.0f)) return 0;
  int e2;
  frexp((double)amax, &e2);          /* amax = f * 2^e2, f in [0.5, 1) */
  int b = (e2 - 1) - 8 + 127;
  if (b < 0) b = 0;
  if (b > 254) b = 254;
  return b;
}

static float bf16_bits_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

void orc_swa_fp8_quantise(int64_t n, const uint16_t* rows, uint8_t* codes, uint16_t* rope,
                          uint8_t* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    const uint16_t* x = rows + r * 512;
    for (int blk = 0; blk < 7; ++blk) {
      float amax = 0.0f;
      for (int c = 64 * blk; c < 64 * blk + 64; ++c) {
        const float a = fabsf(bf16_bits_value(x[c]));
        if (a > amax) amax = a;
      }
      const int b = orc_ue8m0_for_amax_e4m3(amax);
      const float s = orc_ue8m0_value(b);
      scales[r * 8 + blk] = (uint8_t)b;
      for (int c = 64 * blk; c < 64 * blk + 64; ++c) {
        const float v = bf16_bits_value(x[c]) / s;
        const int code = orc_e4m3_encode(fabsf(v));
        codes[r * 448 + c] = (uint8_t)(code | (signbit(v) ? 0x80 : 0));
      }
    }
    scales[r * 8 + 7] = 0;
    for (int c = 0; c < 64; ++c) rope[r * 64 + c] = x[448 + c];
  }
}

void orc_swa_fp8_dequantise(int64_t n, const uint8_t* codes, const uint16_t* rope,
                            const uint8_t* scales, float* out) {
  for (int64_t r = 0; r < n; ++r) {
    for (int c = 0; c < 448; ++c)
      out[r * 512 + c] = orc_e4m3_value(codes[r * 448 + c]) * orc_ue8m0_value(scales[r * 8 + c / 64]);
    for (int c = 0; c < 64; ++c) out[r * 512 + 448 + c] = bf16_bits_value(rope[r * 64 + c]);
  }
}

int orc_group(int layout) { return layout == 1 ? 16 : 32; }

static float block_scale(int layout, float amax, uint8_t* byte) {
  if (layout == 1) {
    int b = orc_e4m3_encode(amax / 6.0f);
    *byte = (uint8_t)b;
    return orc_e4m3_value(b);
  }
  int b = orc_ue8m0_for_amax(amax);
  *byte = (uint8_t)b;
  return orc_ue8m0_value(b);
}

void orc_quantise(int64_t n, int dim, int layout, const float* x, uint8_t* codes,
                  uint8_t* scales) {
  const int g = orc_group(layout), nb = dim / g;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    const float* xr = x + r * dim;
    uint8_t* cr = codes + r * (dim / 2);
    for (int b = 0; b < nb; ++b) {
      float amax = 0.0f;
      for (int i = 0; i < g; ++i) {
        float a = fabsf(xr[b * g + i]);
        if (a > amax) amax = a;
      }
      uint8_t sb;
      float s = block_scale(layout, amax, &sb);
      scales[r * nb + b] = sb;
      for (int i = 0; i < g; ++i) {
        int ch = b * g + i;
        int code = (s == 0.0f) ? 0 : orc_e2m1_encode(xr[ch] / s);
        if (ch & 1) cr[ch >> 1] = (uint8_t)(cr[ch >> 1] | (code << 4));
        else cr[ch >> 1] = (uint8_t)code;
      }
    }
  }
}

void orc_dequantise(int64_t n, int dim, int layout, const uint8_t* codes,
                    const uint8_t* scales, float* out) {
  const int g = orc_group(layout), nb = dim / g;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int ch = 0; ch < dim; ++ch) {
      uint8_t byte = codes[r * (dim / 2) + ch / 2];
      int code = (ch & 1) ? (byte >> 4) : (byte & 15);
      int sb = scales[r * nb + ch / g];
      float s = layout == 1 ? orc_e4m3_value(sb) : orc_ue8m0_value(sb);
      out[r * dim + ch] = orc_e2m1_value(code) * s;
    }
}

/* One entry: 4 bits per channel plus one scale byte per block.               */
double orc_entry_bytes(int dim, int layout) {
  return dim * 0.5 + (double)(dim / orc_group(layout));
}

/* Global KV bytes per token: every layer that owns a cache stores one entry
 * per `ratio` tokens.  [NDT sec 3.1], [V41 abstract: 890 bytes / token].     */
double orc_bytes_per_token(int n_layers, const int* ratio, const double* bpe) {
  double t = 0.0;
  for (int i = 0; i < n_layers; ++i) t += bpe[i] / (double)ratio[i];
  return t;
}

/* ------------------------------------------------------------------------ */
/* exp for the compressor's softmax weights.  Cody-Waite range reduction
 * (ln 2 split as 0.693359375 - 2.12194440e-4, the split used by Cephes'
 * expf) followed by the degree-7 Taylor polynomial in Horner form with fused
 * multiply-adds, then an exact scaling by 2^n.  Defined on [-87, 88]; returns
 * 0 below (the compressor only evaluates it at x <= 0).                      */
float orc_expf(float x) {
  if (x != x) return x;
  if (x < -87.0f) return 0.0f;
  if (x > 88.0f) return INFINITY;
  float t = x * 1.44269504088896341f;
  float n = rintf(t);
  float r = fmaf(-n, 0.693359375f, x);
  r = fmaf(-n, -2.12194440e-4f, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n;
  float two_n;
  if (ni < -126) {              /* only reachable at x just above -87 */
    two_n = ldexpf(1.0f, ni);
  } else {
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    memcpy(&two_n, &bits, 4);
  }
  return p * two_n;
}

static float bf16f(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint16_t f32_bf16_rne(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((b >> 16) | 0x40);
  return (uint16_t)((b + 0x7fffu + ((b >> 16) & 1u)) >> 16);
}

/* CSA2 compressor ([V41 sec 2.3]: no overlap, no positional bias; pooling
 * form of [V4B sec 4.2]): entry i, channel c is sum_j softmax_j(Z[j,c]) *
 * C[j,c] over the m tokens j of block i.  fp32, fixed order j = 0..m-1, IEEE
 * division; the sum starts from the j = 0 term so that m = 1 is the identity
 * ([NDT sec 3.3.2]: the pooling degenerates to a per-token projection).    */
void orc_compress(int64_t n_out, int m, int dim, const uint16_t* c_bf16,
                  const float* z, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_out; ++i) {
    float e[64];
    for (int c = 0; c < dim; ++c) {
      float mx = z[(i * m) * dim + c];
      for (int j = 1; j < m; ++j) {
        float v = z[(i * m + j) * dim + c];
        if (v > mx) mx = v;
      }
      float sum = 0.0f;
      for (int j = 0; j < m; ++j) {
        e[j] = orc_expf(z[(i * m + j) * dim + c] - mx);
        sum = (j == 0) ? e[j] : sum + e[j];
      }
      float acc = 0.0f;
      for (int j = 0; j < m; ++j) {
        float w = e[j] / sum;
        float term = w * bf16f(c_bf16[(i * m + j) * dim + c]);
        acc = (j == 0) ? term : acc + term;
      }
      out[i * dim + c] = acc;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Index score [V4B sec 4.1]: I[s] = sum_h w[h] * ReLU(q[h] . K[s]), q and K
 * taken at their bf16 values, fp64 throughout, no extra scale.               */
void orc_index_scores(int64_t n, int heads, int d, const uint16_t* k_bf16,
                      const uint16_t* q_bf16, const float* w, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t s = 0; s < n; ++s) {
    double tot = 0.0;
    for (int h = 0; h < heads; ++h) {
      double dot = 0.0;
      for (int i = 0; i < d; ++i)
        dot += (double)bf16f(q_bf16[h * d + i]) * (double)bf16f(k_bf16[s * d + i]);
      tot += (double)w[h] * (dot > 0.0 ? dot : 0.0);
    }
    out[s] = tot;
  }
}

typedef struct { float v; int32_t i; } scored_t;

static int cmp_score(const void* a, const void* b) {
  const scored_t* x = (const scored_t*)a;
  const scored_t* y = (const scored_t*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

static int cmp_int(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* bf16 rounding of index scores [V4B sec 7: the scores are quantised from
 * FP32 to BF16 for the selector]: the nearest value whose low 16 fp32 bits
 * are zero, found by comparing the two neighbours' distances in double; an
 * exact tie goes to the neighbour whose last kept bit is 0 (IEEE
 * round-to-nearest-even on the 8-bit significand).  Finite inputs.          */
float orc_bf16_round(float x) {
  if (x != x || isinf(x)) return x;
  uint32_t b;
  memcpy(&b, &x, 4);
  const uint32_t lo_b = b & 0xFFFF0000u;    /* toward zero */
  if (lo_b == b) return x;
  const uint32_t hi_b = lo_b + 0x10000u;    /* away from zero */
  float lo, hi;
  memcpy(&lo, &lo_b, 4);
  memcpy(&hi, &hi_b, 4);
  const double dl = fabs((double)x - (double)lo), dh = fabs((double)hi - (double)x);
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return ((lo_b >> 16) & 1u) ? hi : lo;
}

void orc_bf16_round_n(int64_t n, const float* in, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(in[i]);
}

/* Top-k [V4B sec 4.1, V41 sec 4.2.1: k = 512]: full sort by (score desc,
 * index asc); keep min(k, n); report them in ascending index order, pad -1.  */
int orc_topk(int64_t n, const float* scores, int k, int32_t* idx_out) {
  int keff = (int)(n < k ? n : k);
  if (n > 0) {
    scored_t* all = (scored_t*)malloc(sizeof(scored_t) * (size_t)n);
    for (int64_t s = 0; s < n; ++s) { all[s].v = scores[s]; all[s].i = (int32_t)s; }
    qsort(all, (size_t)n, sizeof(scored_t), cmp_score);
    for (int t = 0; t < keff; ++t) idx_out[t] = all[t].i;
    free(all);
    qsort(idx_out, (size_t)keff, sizeof(int32_t), cmp_int);
  }
  for (int t = keff; t < k; ++t) idx_out[t] = -1;
  return keff;
}

/* ------------------------------------------------------------------------ */
/* Shared-KV MQA over the selected entries plus the sliding window, one joint
 * softmax ([V4B sec 4.1 core attention with key = value], [V4B sec 4.3 SWA
 * branch], [NDT sec 3.3.1: readout concatenates the SWA and the selected main
 * KV]).  For each head h and candidate j: l_j = scale * q_h . kv_j,
 * o_h = sum_j softmax(l)_j kv_j, lse_h = log sum_j exp(l_j).  Entries with a
 * negative index are padding and are skipped.  fp64 throughout; the bf16
 * output is the fp64 result rounded to fp32 and then to bf16.               */
void orc_sparse_attention(int heads, int dim, int layout, const uint16_t* q_bf16,
                          const uint8_t* codes, const uint8_t* scales, int64_t n_ent,
                          int n_idx, const int32_t* idx, int n_swa,
                          const uint16_t* swa_bf16, float scale, uint16_t* out_bf16,
                          double* out_f64, double* lse) {
  const int g = orc_group(layout);
  int n_cand = 0;
  for (int t = 0; t < n_idx; ++t)
    if (idx[t] >= 0 && idx[t] < n_ent) ++n_cand;
  n_cand += n_swa;
  double* kv = (double*)malloc(sizeof(double) * (size_t)(n_cand > 0 ? n_cand : 1) * dim);
  float* row = (float*)malloc(sizeof(float) * (size_t)dim);
  int j = 0;
  for (int t = 0; t < n_idx; ++t) {
    int64_t s = idx[t];
    if (s < 0 || s >= n_ent) continue;
    orc_dequantise(1, dim, layout, codes + s * (dim / 2), scales + s * (dim / g), row);
    for (int c = 0; c < dim; ++c) kv[(int64_t)j * dim + c] = (double)row[c];
    ++j;
  }
  for (int r = 0; r < n_swa; ++r, ++j)
    for (int c = 0; c < dim; ++c)
      kv[(int64_t)j * dim + c] = (double)bf16f(swa_bf16[(int64_t)r * dim + c]);
  free(row);

#pragma omp parallel for schedule(static)
  for (int h = 0; h < heads; ++h) {
    double* l = (double*)malloc(sizeof(double) * (size_t)(n_cand > 0 ? n_cand : 1));
    double mx = -INFINITY;
    for (int a = 0; a < n_cand; ++a) {
      double dot = 0.0;
      for (int c = 0; c < dim; ++c)
        dot += (double)bf16f(q_bf16[(int64_t)h * dim + c]) * kv[(int64_t)a * dim + c];
      l[a] = (double)scale * dot;
      if (l[a] > mx) mx = l[a];
    }
    double sum = 0.0;
    for (int a = 0; a < n_cand; ++a) { l[a] = exp(l[a] - mx); sum += l[a]; }
    for (int c = 0; c < dim; ++c) {
      double o = 0.0;
      for (int a = 0; a < n_cand; ++a) o += l[a] * kv[(int64_t)a * dim + c];
      o = n_cand > 0 ? o / sum : 0.0;
      if (out_f64) out_f64[(int64_t)h * dim + c] = o;
      if (out_bf16) out_bf16[(int64_t)h * dim + c] = f32_bf16_rne((float)o);
    }
    if (lse) lse[h] = n_cand > 0 ? mx + log(sum) : -INFINITY;
    free(l);
  }
  free(kv);
}
