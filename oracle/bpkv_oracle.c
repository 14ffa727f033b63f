/*
 * Plain CPU oracle for query-dependent prefix reads of a bit-plane K cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the bench's CPU-baseline /
 * reference arm use it.  It shares no code, header or constant generator with
 * the CUDA library.
 *
 * Every function works on one unit = one (sequence, KV head) of one layer and
 * follows "Fathom: per-query read depth for sparse decoding over an offloaded
 * KV cache" (the Fathom page):
 *   - section 3.2 (bit-plane K cache): 4-bit uniform symmetric per-channel code,
 *     one fp16 scale per 64-token block, s = blockmax/8,
 *     c = clip(floor(k/s), -8, 7) + 8, bit p of the 64 codes of a block packed
 *     into one 64-bit plane word, p = 0 the most significant bit (the sign);
 *   - section 1, observation 2: the first t planes of a channel are its t-bit
 *     mid-rise quantiser with the same block scale;
 *   - section 1, observation 1: depth allocation by marginal value
 *     g_j * 4^-t_j (reverse water-filling), g_j the channel's contribution to the
 *     score variance;
 *   - section 2 ("Top-k decoding"): first 4 and last 32 tokens always kept, the
 *     other k-36 are each query head's top scores, exact attention
 *     softmax(q K^T / sqrt(D)) V over the selected set;
 *   - section 2 ("SparQ"): fixed channel sets by summed |q| over the group;
 *   - section 2 ("Double Sparsity"): channel sets chosen offline from
 *     calibration statistics (mean |q| times mean |k| per channel);
 *   - contributions, basis rule: KLT planes (an orthogonal basis) for models
 *     without QK norm, applied to keys and queries alike.
 * The value-side functions (or_v_*, or_attend_vdepth) follow the second read
 * stage of "ReadKV" (the ReadKV page, sections 5.3 and 5.4): per-token value
 * depths from the squared attention probabilities.
 * Readings where the page is silent (bit order inside a word, zero and
 * overflowing scales, tie rules, stop rule of the allocator) are stated at each
 * function.
 *
 * Planted mistakes: building with -DOR_MUTANT=n (n >= 1) swaps in one plausible
 * error per n, so that a test can check that the pins catch it.  The default
 * build (OR_MUTANT undefined, i.e. 0) contains none of them.
 *
 * Floating point: scores and attention in double.  Where a float decides an
 * integer (the code floor, the allocator's comparisons) the oracle takes that
 * decision in the same precision as the CUDA kernels: float32 IEEE division for
 * k/s and float32 products/sums for g_j.  Build with -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef OR_MUTANT
#define OR_MUTANT 0
#endif

/* ---------------------------------------------------------------- scalars */

static double or_bf16_value(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16 value of a bit pattern (finite patterns only). */
double or_fp16_value(uint16_t h) {
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v = (e == 0) ? ldexp((double)m, -24) : ldexp((double)(1024 + m), e - 25);
  return (h & 0x8000) ? -v : v;
}

/* Round x >= 0 to the nearest binary16 value, ties to even.  Reading: values at
 * or above the largest finite half (65504) saturate to it instead of becoming
 * infinity, so a block scale is always finite. */
uint16_t or_fp16_bits(double x) {
  if (!(x > 0.0)) return 0;
  if (x >= 65504.0) return 0x7BFF;
  int e2;
  frexp(x, &e2);            /* x = m 2^e2, m in [0.5, 1) */
  int E = e2 - 1;           /* x in [2^E, 2^(E+1)) */
  if (E < -14) {            /* subnormal range: spacing 2^-24 */
    double r = nearbyint(ldexp(x, 24));
    return (uint16_t)r;     /* r == 1024 is the smallest normal, encoded alike */
  }
  double r = nearbyint(ldexp(x, 10 - E)); /* in [1024, 2048] */
  return (uint16_t)(((E + 15) << 10) + ((int)r - 1024));
}

/* ---------------------------------------------------------------- encode */

/*
 * Encode the first n rows of one unit's keys.
 *   k      : bf16 bit patterns, row-major [n][D] (row i = token i)
 *   scales : out, fp16 bit patterns [D][nb_cap]  (channel-major)
 *   planes : out, [D][4][nb_cap] 64-bit words; word (j, p, b) bit i holds bit
 *            (3 - p) of the code of token 64 b + i (reading: token i of a block
 *            is bit i, least significant first); bits of absent tokens are 0.
 * Blocks >= ceil(n/64) are left untouched.
 * Readings: s16 = fp16(a/8) with a/8 exact in double; if s16 == 0 (an all-zero
 * block, or a block whose max underflows fp16) every code is 8, which
 * dequantises to 0 at every depth.
 */
void or_encode(int64_t n, int32_t D, const uint16_t *k, int64_t nb_cap,
               uint16_t *scales, uint64_t *planes) {
  int64_t nb = (n + 63) / 64;
  for (int32_t j = 0; j < D; ++j) {
    for (int64_t b = 0; b < nb; ++b) {
      int64_t i0 = b * 64, i1 = i0 + 64 < n ? i0 + 64 : n;
      double a = 0.0;
      for (int64_t i = i0; i < i1; ++i) {
        double x = fabs(or_bf16_value(k[i * D + j]));
        if (x > a) a = x;
      }
      uint16_t s16 = or_fp16_bits(a / 8.0);
      float s = (float)or_fp16_value(s16);
      uint64_t w[4] = {0, 0, 0, 0};
      for (int64_t i = i0; i < i1; ++i) {
        int c;
        if (s16 == 0) {
          c = 8;
        } else {
          float kv = (float)or_bf16_value(k[i * D + j]);
          float qt = kv / s; /* IEEE float32 division, round to nearest */
          double f = (OR_MUTANT == 7) ? nearbyint((double)qt) : floor((double)qt);
          if (f < -8.0) f = -8.0;
          if (f > 7.0) f = 7.0;
          c = (int)f + 8;
        }
        for (int p = 0; p < 4; ++p) {
          int src_bit = (OR_MUTANT == 2) ? p : 3 - p;
          int dst_bit = (OR_MUTANT == 1) ? 63 - (int)(i - i0) : (int)(i - i0);
          if ((c >> src_bit) & 1) w[p] |= (uint64_t)1 << dst_bit;
        }
      }
      scales[(int64_t)j * nb_cap + b] = s16;
      for (int p = 0; p < 4; ++p) planes[((int64_t)j * 4 + p) * nb_cap + b] = w[p];
    }
  }
}

/* Code c (t-bit prefix, t in 0..4) of token i, channel j, read from the planes. */
static int or_prefix_code(const uint64_t *planes, int64_t nb_cap, int32_t j, int t, int64_t i) {
  int64_t b = i / 64;
  int bit = (int)(i % 64);
  int c = 0;
  for (int p = 0; p < t; ++p)
    c = (c << 1) | (int)((planes[((int64_t)j * 4 + p) * nb_cap + b] >> bit) & 1);
  return c;
}

/* Dequantised key from a t-plane prefix: the t-bit mid-rise quantiser with the
 * block scale s, cell width s 2^(4-t), reconstruction at the cell midpoint
 * (reading of "mid-rise"): khat = s ((c_t + 1/2) 2^(4-t) - 8); t = 0 gives 0. */
double or_dequant(double s, int c_t, int t) {
  if (t == 0) return 0.0;
  double half = (OR_MUTANT == 3) ? 0.0 : 0.5;
  return s * (((double)c_t + half) * ldexp(1.0, 4 - t) - 8.0);
}

/* ---------------------------------------------------------------- depths */

/* g_j = sum over the G query heads of q_hj^2 sigma_j^2, in float32, heads in
 * order 0..G-1, each product and sum rounded separately (no fused multiply-add). */
static void or_importance(int32_t D, int32_t G, const float *q, const float *sigma2, float *g) {
  for (int32_t j = 0; j < D; ++j) {
    float acc = 0.0f;
    for (int32_t h = 0; h < G; ++h) {
      float qq = (OR_MUTANT == 6) ? fabsf(q[h * D + j]) : q[h * D + j] * q[h * D + j];
      float term = qq * sigma2[j];
      acc = acc + term;
    }
    g[j] = acc;
  }
}

/*
 * Greedy reverse water-filling.  Items are (channel j, next bit t_j) with value
 * v = g_j * 4^-t_j (float32, one product by the exact constant 4^-t).  The bit
 * costs 4 quarter-bits per token, plus 1 for the channel's fp16 scale when it is
 * the channel's first bit (16 bits per 64 tokens).  At each step the item with
 * the largest v is taken, ties to the lower channel index; allocation stops when
 * that item's v <= 0, when it does not fit the remaining budget (reading: stop,
 * not skip, which makes the result a single water level), or when every
 * channel has 4 bits.  budget_q is in quarter-bits per token (4 x bits).
 * Returns the quarter-bits used.
 */
int32_t or_alloc_depths(int32_t D, int32_t G, const float *q, const float *sigma2,
                        int32_t budget_q, uint8_t *depth) {
  static const float quarter_pow[4] = {1.0f, 0.25f, 0.0625f, 0.015625f};
  float *g = (float *)malloc(sizeof(float) * (size_t)D);
  or_importance(D, G, q, sigma2, g);
  for (int32_t j = 0; j < D; ++j) depth[j] = 0;
  int32_t left = budget_q;
  for (;;) {
    int32_t best = -1;
    float bv = 0.0f;
    for (int32_t j = 0; j < D; ++j) {
      if (depth[j] >= 4) continue;
      float v = g[j] * quarter_pow[depth[j]];
      if (best < 0 || v > bv) { best = j; bv = v; }
    }
    if (best < 0 || !(bv > 0.0f)) break;
    int32_t cost = (depth[best] == 0 && OR_MUTANT != 4) ? 5 : 4;
    if (cost > left) {
      if (OR_MUTANT == 10) { /* skip the item and keep going */
        int32_t any = 0;
        for (int32_t j = 0; j < D; ++j)
          if (depth[j] > 0 && depth[j] < 4 && g[j] * quarter_pow[depth[j]] > 0.0f && left >= 4) any = 1;
        if (any) {
          int32_t b2 = -1;
          float v2 = 0.0f;
          for (int32_t j = 0; j < D; ++j) {
            if (depth[j] == 0 || depth[j] >= 4) continue;
            float v = g[j] * quarter_pow[depth[j]];
            if (b2 < 0 || v > v2) { b2 = j; v2 = v; }
          }
          left -= 4;
          depth[b2] += 1;
          continue;
        }
      }
      break;
    }
    left -= cost;
    depth[best] += 1;
  }
  free(g);
  return budget_q - left;
}

/* Fixed-depth channel sets (section 2, "SparQ"): the r channels with the
 * largest sum over the group of |q_hj| (float32, heads in order; ties to the
 * lower index) are read at depth t, the rest not at all.  r >= D reads every
 * channel at depth t (the 2-bit thumbnail when t = 2). */
void or_fixed_depths(int32_t D, int32_t G, const float *q, int32_t r, int32_t t, uint8_t *depth) {
  float *a = (float *)malloc(sizeof(float) * (size_t)D);
  for (int32_t j = 0; j < D; ++j) {
    float acc = 0.0f;
    for (int32_t h = 0; h < G; ++h) acc = acc + fabsf(q[h * D + j]);
    a[j] = acc;
    depth[j] = 0;
  }
  for (int32_t j = 0; j < D; ++j) {
    int32_t rank = 0; /* channels ordered before j */
    for (int32_t i = 0; i < D; ++i)
      if (a[i] > a[j] || (a[i] == a[j] && i < j)) ++rank;
    if (rank < r) depth[j] = (uint8_t)t;
  }
  free(a);
}

/* Offline-calibrated channel sets (section 2, "Double Sparsity"): a channel's
 * calibration statistic is the mean of |q_j| over the m_q calibration queries
 * and the G query heads of the unit, times the mean of |k_j| over the m_k
 * calibration keys.  The c channels with the largest statistic (ties to the
 * lower index) are read at depth t, the others not at all.  Reading: the page
 * fixes the statistic and c = 32 for a 136-bit read; the precision is ours.
 * Each sum runs in double in storage order (queries, then heads within a
 * query; keys in order), each mean divides its sum once and the product is one
 * double multiplication.  q_cal float [m_q][G][D], k_cal bf16 [m_k][D]. */
void or_calibrate_channels(int32_t D, int32_t G, int64_t m_q, const float *q_cal, int64_t m_k,
                           const uint16_t *k_cal, int32_t c, int32_t t, uint8_t *depth) {
  double *st = (double *)malloc(sizeof(double) * (size_t)D);
  for (int32_t j = 0; j < D; ++j) {
    double a = 0.0, b = 0.0;
    for (int64_t m = 0; m < m_q; ++m)
      for (int32_t h = 0; h < G; ++h) {
        double v = (double)q_cal[(m * G + h) * D + j];
        a = a + ((OR_MUTANT == 12) ? v * v : fabs(v));
      }
    for (int64_t m = 0; m < m_k; ++m) b = b + fabs(or_bf16_value(k_cal[m * D + j]));
    const double qa = a / (double)(m_q * G), kb = b / (double)m_k;
    st[j] = (OR_MUTANT == 11) ? qa : qa * kb;
    depth[j] = 0;
  }
  for (int32_t j = 0; j < D; ++j) {
    int32_t rank = 0; /* channels ordered before j */
    for (int32_t i = 0; i < D; ++i)
      if (st[i] > st[j] || (st[i] == st[j] && i < j)) ++rank;
    if (rank < c) depth[j] = (uint8_t)t;
  }
  free(st);
}

/* ---------------------------------------------------------------- basis */

/* A fixed orthogonal basis for the scanned key codes (Fathom page, section 1,
 * contributions: KLT planes of the keys for models without QK norm; ReadKV
 * page, section 5.1: the same Hadamard-sign transform on keys and queries keeps
 * their inner products).  Reading: y_l = sum_j x_j R[j][l] with R [D][D], as a
 * chain of float32 fused multiply-adds in order j = 0 .. D-1 starting from 0,
 * one chain per output. */
void or_rotate(int32_t D, int64_t rows, const float *x, const float *R, float *y) {
  for (int64_t r = 0; r < rows; ++r)
    for (int32_t l = 0; l < D; ++l) {
      float acc = 0.0f;
      for (int32_t j = 0; j < D; ++j) {
        const float rv = (OR_MUTANT == 13) ? R[l * D + j] : R[j * D + l];
        acc = fmaf(x[r * D + j], rv, acc);
      }
      y[r * D + l] = acc;
    }
}

/* float32 to bf16 bit pattern, round to nearest even (finite values). */
static uint16_t or_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Keys in the basis, rounded to bf16: the encoder codes these (the stored
 * rows for exact attention stay in the original channels). */
void or_rotate_keys(int32_t D, int64_t n, const uint16_t *k_bits, const float *R, uint16_t *out_bits) {
  float *x = (float *)malloc(sizeof(float) * (size_t)D);
  float *y = (float *)malloc(sizeof(float) * (size_t)D);
  for (int64_t i = 0; i < n; ++i) {
    for (int32_t j = 0; j < D; ++j) x[j] = (float)or_bf16_value(k_bits[i * D + j]);
    or_rotate(D, 1, x, R, y);
    for (int32_t l = 0; l < D; ++l) out_bits[i * D + l] = or_bf16_bits(y[l]);
  }
  free(x);
  free(y);
}

/* ---------------------------------------------------------------- scores */

/* score[h][i] = sum_j q_hj khat_ij(t_j) for every token i < n and query head h,
 * in double, channels in index order; no 1/sqrt(D) factor (it does not change
 * the ranking).  Reads only planes p < t_j and the scales of channels t_j > 0.
 * A code has four planes, so a depth value above 4 is read as 4 (reading:
 * the Fathom page's depth ranges over 0..4 bits; larger values read the
 * whole code, never past it). */
void or_scores(int64_t n, int32_t D, int32_t G, const uint16_t *scales, const uint64_t *planes,
               int64_t nb_cap, const uint8_t *depth, const float *q, double *score) {
  for (int64_t i = 0; i < n; ++i) {
    for (int32_t h = 0; h < G; ++h) score[(int64_t)h * n + i] = 0.0;
    for (int32_t j = 0; j < D; ++j) {
      int t = depth[j] > 4 ? 4 : depth[j];
      if (t == 0) continue;
      double s = or_fp16_value(scales[(int64_t)j * nb_cap + i / 64]);
      double kh = or_dequant(s, or_prefix_code(planes, nb_cap, j, t, i), t);
      for (int32_t h = 0; h < G; ++h) score[(int64_t)h * n + i] += (double)q[h * D + j] * kh;
    }
  }
}

/* ---------------------------------------------------------------- top-k */

typedef struct { double s; int64_t i; } or_cand;

static int or_cand_cmp(const void *x, const void *y) {
  const or_cand *a = (const or_cand *)x, *b = (const or_cand *)y;
  if (a->s > b->s) return -1;
  if (a->s < b->s) return 1;
  if (OR_MUTANT == 5) return (a->i > b->i) ? -1 : (a->i < b->i);
  return (a->i < b->i) ? -1 : (a->i > b->i);
}

/*
 * Selection of one query head: tokens [0, n_sink) and [n - n_recent, n) always,
 * plus the k - n_sink - n_recent highest-scoring tokens among the rest, ties to
 * the lower token index (reading).  k counts the fixed tokens (reading of
 * "the other k-36 keys").  Writes the selected token indices in ascending order
 * to idx[0..count) and -1 to idx[count..k); returns count.
 */
int32_t or_topk(int64_t n, const double *score, int32_t k, int32_t n_sink, int32_t n_recent,
                int32_t *idx) {
  uint8_t *sel = (uint8_t *)calloc((size_t)(n > 0 ? n : 1), 1);
  int64_t lo = n_sink < n ? n_sink : n;
  int64_t hi = n - n_recent > lo ? n - n_recent : lo;
  for (int64_t i = 0; i < lo; ++i) sel[i] = 1;
  for (int64_t i = hi; i < n; ++i) sel[i] = 1;
  int64_t n_top = (int64_t)k - n_sink - n_recent;
  if (n_top < 0) n_top = 0;
  int64_t nc = hi - lo;
  if (nc > 0 && n_top > 0) {
    or_cand *c = (or_cand *)malloc(sizeof(or_cand) * (size_t)nc);
    for (int64_t i = lo; i < hi; ++i) { c[i - lo].s = score[i]; c[i - lo].i = i; }
    qsort(c, (size_t)nc, sizeof(or_cand), or_cand_cmp);
    for (int64_t r = 0; r < nc && r < n_top; ++r) sel[c[r].i] = 1;
    free(c);
  }
  int32_t cnt = 0;
  for (int64_t i = 0; i < n; ++i)
    if (sel[i]) idx[cnt++] = (int32_t)i;
  for (int32_t r = cnt; r < k; ++r) idx[r] = -1;
  free(sel);
  return cnt;
}

/* ---------------------------------------------------------------- union */

typedef struct { int32_t i; int32_t h; } or_pair;

static int or_pair_cmp(const void *x, const void *y) {
  const or_pair *a = (const or_pair *)x, *b = (const or_pair *)y;
  if (a->i != b->i) return (a->i < b->i) ? -1 : 1;
  return (a->h < b->h) ? -1 : (a->h > b->h);
}

/* Union of the G selections of one KV head (the rows fetched once for all its
 * query heads): distinct token indices in ascending order, and for each a mask
 * whose bit h is set when query head h selected it.  idx is [G][k], -1 padded.
 * Returns the union size. */
int32_t or_union(int32_t G, int32_t k, const int32_t *idx, int32_t *uidx, uint8_t *umask) {
  or_pair *p = (or_pair *)malloc(sizeof(or_pair) * (size_t)(G * k > 0 ? G * k : 1));
  int32_t m = 0;
  for (int32_t h = 0; h < G; ++h)
    for (int32_t r = 0; r < k; ++r)
      if (idx[h * k + r] >= 0) { p[m].i = idx[h * k + r]; p[m].h = h; ++m; }
  qsort(p, (size_t)m, sizeof(or_pair), or_pair_cmp);
  int32_t u = 0;
  for (int32_t r = 0; r < m; ++r) {
    if (u > 0 && uidx[u - 1] == p[r].i) {
      if (OR_MUTANT != 9) umask[u - 1] |= (uint8_t)(1u << p[r].h);
    } else {
      uidx[u] = p[r].i;
      umask[u] = (uint8_t)(1u << p[r].h);
      ++u;
    }
  }
  free(p);
  return u;
}

/* ---------------------------------------------------------------- attention */

/* Exact attention of each query head over its own selected rows:
 * o_h = sum_i softmax_i(q_h . k_i / sqrt(D)) v_i, with the stored bf16 K and V
 * rows (row-major [*][D]) taken exactly, everything in double.  idx is [G][k],
 * -1 padded; out is [G][D]. */
void or_attend(int32_t D, int32_t G, const float *q, const uint16_t *k_rows, const uint16_t *v_rows,
               const int32_t *idx, int32_t k, double *out) {
  double *logit = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  double scale = (OR_MUTANT == 8) ? 1.0 : 1.0 / sqrt((double)D);
  for (int32_t h = 0; h < G; ++h) {
    double m = -INFINITY;
    int32_t cnt = 0;
    for (int32_t r = 0; r < k; ++r) {
      int32_t i = idx[h * k + r];
      if (i < 0) continue;
      double acc = 0.0;
      for (int32_t d = 0; d < D; ++d) acc += (double)q[h * D + d] * or_bf16_value(k_rows[(int64_t)i * D + d]);
      logit[r] = acc * scale;
      if (logit[r] > m) m = logit[r];
      ++cnt;
    }
    for (int32_t d = 0; d < D; ++d) out[h * D + d] = 0.0;
    if (cnt == 0) continue;
    double z = 0.0;
    for (int32_t r = 0; r < k; ++r) {
      int32_t i = idx[h * k + r];
      if (i < 0) continue;
      double w = exp(logit[r] - m);
      z += w;
      for (int32_t d = 0; d < D; ++d) out[h * D + d] += w * or_bf16_value(v_rows[(int64_t)i * D + d]);
    }
    for (int32_t d = 0; d < D; ++d) out[h * D + d] /= z;
  }
  free(logit);
}

/* Dense attention over the first n rows (the dense bf16 baseline). */
void or_dense_attend(int64_t n, int32_t D, int32_t G, const float *q, const uint16_t *k_rows,
                     const uint16_t *v_rows, double *out) {
  double scale = 1.0 / sqrt((double)D);
  double *logit = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int32_t h = 0; h < G; ++h) {
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
      double acc = 0.0;
      for (int32_t d = 0; d < D; ++d) acc += (double)q[h * D + d] * or_bf16_value(k_rows[i * D + d]);
      logit[i] = acc * scale;
      if (logit[i] > m) m = logit[i];
    }
    for (int32_t d = 0; d < D; ++d) out[h * D + d] = 0.0;
    if (n == 0) continue;
    double z = 0.0;
    for (int64_t i = 0; i < n; ++i) {
      double w = exp(logit[i] - m);
      z += w;
      for (int32_t d = 0; d < D; ++d) out[h * D + d] += w * or_bf16_value(v_rows[i * D + d]);
    }
    for (int32_t d = 0; d < D; ++d) out[h * D + d] /= z;
  }
  free(logit);
}

/* ------------------------------------------------- value-side depth (stage 2) */

/*
 * Second read stage of "ReadKV" (the ReadKV page, sections 5.3 and 5.4): after
 * the keys decide the attention, each value row is read to a per-token depth,
 * all channels of a token sharing it, and the depths go to the rows whose
 * attention weight matters most.
 *
 * Value bit planes (readings: the page's value codes are progressive per
 * token; the code is the same 4-bit mid-rise code as the keys, with the scale
 * taken over the row instead of a block of a channel, since a row is what
 * one depth covers): token i has one fp16 scale s_i = fp16(max_j |v_ij| / 8),
 * codes c_ij = clip(floor(v_ij / s_i), -8, 7) + 8 (float32 division, as for the
 * keys; a zero scale gives code 8), and plane p of token i is D / 64 words, bit
 * b of word w = bit (3 - p) of the code of channel 64 w + b.  Layout: vscales
 * [n], vplanes [n][4][D / 64].  D is a multiple of 64.
 */
void or_v_encode(int64_t n, int32_t D, const uint16_t *v, uint16_t *vscales, uint64_t *vplanes) {
  const int32_t W = D / 64;
  for (int64_t i = 0; i < n; ++i) {
    double a = 0.0;
    for (int32_t j = 0; j < D; ++j) {
      double x = fabs(or_bf16_value(v[i * D + j]));
      if (x > a) a = x;
    }
    uint16_t s16 = or_fp16_bits(a / 8.0);
    float s = (float)or_fp16_value(s16);
    vscales[i] = s16;
    for (int64_t e = 0; e < 4 * (int64_t)W; ++e) vplanes[i * 4 * W + e] = 0;
    for (int32_t j = 0; j < D; ++j) {
      int c = 8;
      if (s16 != 0) {
        float qt = (float)or_bf16_value(v[i * D + j]) / s;
        double f = floor((double)qt);
        if (f < -8.0) f = -8.0;
        if (f > 7.0) f = 7.0;
        c = (int)f + 8;
      }
      int w = j / 64, b = (OR_MUTANT == 16) ? 63 - j % 64 : j % 64;
      for (int p = 0; p < 4; ++p)
        if ((c >> (3 - p)) & 1) vplanes[(i * 4 + p) * W + w] |= (uint64_t)1 << b;
    }
  }
}

/* Value row i read to depth t (0..4): vhat_j = s_i ((c_t + 1/2) 2^(4-t) - 8),
 * the same mid-rise reconstruction as the keys; t = 0 reads nothing and gives
 * the zero row. */
void or_v_row(int32_t D, const uint16_t *vscales, const uint64_t *vplanes, int64_t i, int t, double *out) {
  const int32_t W = D / 64;
  double s = or_fp16_value(vscales[i]);
  for (int32_t j = 0; j < D; ++j) {
    int c = 0;
    for (int p = 0; p < t; ++p) c = (c << 1) | (int)((vplanes[(i * 4 + p) * W + j / 64] >> (j % 64)) & 1);
    out[j] = or_dequant(s, c, t);
  }
}

/*
 * Per-token value depths (the ReadKV page, section 5.4): greedy on the
 * predicted error drop.  Items are (row r, next plane t_r) with value
 * a_r 4^-t_r, the error of a mid-rise code in standardised units shrinking by
 * 4 per plane; each item costs one plane (D bits per token, section 5.4), the
 * budget is budget planes; the largest value goes first, ties to the lower
 * row; allocation stops when the value is <= 0, the budget is spent or every
 * row has 4 planes.  Row scales are read for rows with t_r > 0 and are not
 * charged to the budget (the page counts value bits in planes).  Returns the
 * planes used.
 */
int32_t or_v_alloc(int32_t n_rows, const double *a, int32_t budget, uint8_t *depth) {
  for (int32_t r = 0; r < n_rows; ++r) depth[r] = 0;
  int32_t left = budget;
  while (left > 0) {
    int32_t best = -1;
    double bv = 0.0;
    for (int32_t r = 0; r < n_rows; ++r) {
      if (depth[r] >= 4) continue;
      double v = a[r] * ldexp(1.0, -2 * depth[r]);
      if (best < 0 || v > bv || (OR_MUTANT == 15 && v == bv)) { best = r; bv = v; }
    }
    if (best < 0 || !(bv > 0.0)) break;
    depth[best] += 1;
    left -= 1;
  }
  return budget - left;
}

/*
 * Stage 2 over one KV head's union (rows uidx[0..n_u), ascending, with head
 * masks umask: bit h set when query head h selected the row).  Head h attends
 * over its own rows with exact bf16 keys: p_h(r) = softmax_r(q_h . k / sqrt(D)).
 * The weight of a row is a_r = sum_h p_h(r)^2 (ReadKV page, section 5.3: squared
 * attention probabilities summed over the query heads sharing the KV head, head
 * scale coefficient 1), depths come from or_v_alloc (or are taken from
 * depth_in when it is not NULL, to evaluate another allocation), and
 * o_h = sum_r p_h(r) vhat_r(t_r).  Everything in double.  Outputs: depth[n_u],
 * weight[n_u] (a_r), out[G][D].
 */
void or_attend_vdepth(int32_t D, int32_t G, const float *q, const uint16_t *k_rows, const uint16_t *vscales,
                      const uint64_t *vplanes, const int32_t *uidx, const uint8_t *umask, int32_t n_u,
                      int32_t budget_v, const uint8_t *depth_in, uint8_t *depth, double *weight, double *out) {
  const double scale = 1.0 / sqrt((double)D);
  double *p = (double *)malloc(sizeof(double) * (size_t)(n_u > 0 ? n_u : 1) * (size_t)G);
  double *row = (double *)malloc(sizeof(double) * (size_t)D);
  for (int32_t h = 0; h < G; ++h) {
    double m = -INFINITY;
    for (int32_t r = 0; r < n_u; ++r) {
      if (!((umask[r] >> h) & 1)) { p[h * n_u + r] = -INFINITY; continue; }
      double acc = 0.0;
      for (int32_t d = 0; d < D; ++d) acc += (double)q[h * D + d] * or_bf16_value(k_rows[(int64_t)uidx[r] * D + d]);
      p[h * n_u + r] = acc * scale;
      if (p[h * n_u + r] > m) m = p[h * n_u + r];
    }
    double z = 0.0;
    for (int32_t r = 0; r < n_u; ++r) {
      double e = ((umask[r] >> h) & 1) ? exp(p[h * n_u + r] - m) : 0.0;
      p[h * n_u + r] = e;
      z += e;
    }
    for (int32_t r = 0; r < n_u; ++r) p[h * n_u + r] = z > 0.0 ? p[h * n_u + r] / z : 0.0;
  }
  for (int32_t r = 0; r < n_u; ++r) {
    double acc = 0.0;
    for (int32_t h = 0; h < G; ++h) acc += (OR_MUTANT == 14) ? p[h * n_u + r] : p[h * n_u + r] * p[h * n_u + r];
    weight[r] = acc;
  }
  if (depth_in) {
    for (int32_t r = 0; r < n_u; ++r) depth[r] = depth_in[r] > 4 ? 4 : depth_in[r];
  } else {
    or_v_alloc(n_u, weight, budget_v, depth);
  }
  for (int64_t e = 0; e < (int64_t)G * D; ++e) out[e] = 0.0;
  for (int32_t r = 0; r < n_u; ++r) {
    or_v_row(D, vscales, vplanes, uidx[r], depth[r], row);
    for (int32_t h = 0; h < G; ++h) {
      double w = p[h * n_u + r];
      if (w == 0.0) continue;
      for (int32_t d = 0; d < D; ++d) out[h * D + d] += w * row[d];
    }
  }
  free(row);
  free(p);
}
