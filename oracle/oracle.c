/*
 * Float64 CPU oracle for the indexer-selected sparse attention step.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
 * benchmark's CPU-baseline leg call it; the product path never does.  It is
 * plain and slow on purpose: one loop nest per definition, no blocking, no
 * fusion, every value decoded from its storage format and combined in IEEE
 * double.  The only parallelism is an OpenMP loop over independent query
 * tokens.
 *
 * Sources (page title, section):
 *  - "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Indexer.forward: the
 *    index score einsum, its ReLU and the weighted sum over index heads; the
 *    visibility rule for compressed positions; the top-k kept per query,
 *    re-sorted into position order, with -1 for unreachable picks.
 *  - same page, get_window_topk_idxs and Attention._window_kv: the raw
 *    sliding window (a ring of window_size slots, the query's own token
 *    included) and Attention.forward: one sparse attention over the window
 *    rows concatenated with the selected compressed rows.
 *  - "DeepSeek-V3.2-Exp inference/model.py", Indexer.forward: fp8-e4m3 index
 *    keys with one fp32 scale per position (head_dim 128 = one block), and
 *    fp8 queries with a per-(token, head) scale folded into the weights;
 *    rotate_activation and act_quant, the producer of those codes and scales.
 *  - "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", select_candidate_blocks
 *    (level one of the two-level top-k) and its use in Indexer.forward;
 *    Compressor.forward with RMSNorm.forward (gated pooling of r tokens).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - scales are dequantisation multipliers: q_hat = q * q_scale[t,h],
 *    k_hat = k * k_scale[b,s]; w is used as given (callers fold softmax and
 *    head-count scaling into it, as both pages do);
 *  - ties in the top-k go to the lower position;
 *  - the optional attention sink adds exp(sink_h - m) to the softmax
 *    denominator only (parity unpinned: the formula is not on the pages);
 *  - window rows and compressed rows are concatenated, never de-duplicated;
 *  - the Hadamard rotation of the producer is the exact value rounded once to
 *    bf16; the producer's act_quant (scale and codes) is taken in fp32, the
 *    precision of the page's quantiser.
 *
 * Compile-time ORC_MUTANT=n builds deliberately wrong variants; the pin tests
 * build them to show that each plausible mistake fails at least one pin.  The
 * default build (ORC_MUTANT undefined) is the oracle.
 */
#define _DEFAULT_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle.h"

#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif

/* ---- storage formats ---------------------------------------------------- */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits. */
double orc_bf16_value(uint16_t bits) {
  int sign = bits >> 15;
  int e = (bits >> 7) & 0xFF;
  int m = bits & 0x7F;
  double v;
  if (e == 0xFF)
    v = m ? NAN : INFINITY;
  else if (e == 0)
    v = ldexp((double)m, -126 - 7); /* subnormal: 0.m * 2^-126 */
  else
    v = ldexp(128.0 + m, e - 127 - 7); /* 1.m * 2^(e-127) */
  return sign ? -v : v;
}

/* float8 e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, exponent 0 holds the subnormals. */
double orc_e4m3_value(uint8_t bits) {
  int sign = bits >> 7;
  int e = (bits >> 3) & 0xF;
  int m = bits & 0x7;
  double v;
  if (e == 0xF && m == 0x7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -6 - 3); /* subnormal: 0.m * 2^-6 */
  else
    v = ldexp(8.0 + m, e - 7 - 3); /* 1.m * 2^(e-7) */
  return sign ? -v : v;
}

static double elem(const void *base, int32_t dtype, int64_t i) {
  if (dtype == ORC_BF16) return orc_bf16_value(((const uint16_t *)base)[i]);
  return orc_e4m3_value(((const uint8_t *)base)[i]);
}

/* ---- visibility and window ---------------------------------------------- */

/* Compressed entry j stands for tokens [j*r, (j+1)*r) and becomes visible once
 * the query has passed its last token: the query at absolute position p sees
 * the entries j < floor((p + 1) / r).  (Prefill: compress_lens =
 * arange(1, seqlen + 1) // ratio; decode: end_pos // ratio with
 * end_pos = p + 1.) */
int32_t orc_n_vis(int32_t pos, int32_t r) {
#if ORC_MUTANT == 4
  return pos / r;
#else
  return (pos + 1) / r;
#endif
}

/* The raw window of the query at position p: positions max(0, p-W+1) .. p,
 * its own token included (decode writes the token into its ring slot before
 * attending).  Each lives in ring slot position mod R.  Oldest first. */
int32_t orc_window_slots(int32_t pos, int32_t W, int32_t R, int32_t *slots) {
  int32_t n = 0;
#if ORC_MUTANT == 6
  for (int32_t p = pos - W; p <= pos - 1; ++p)
#else
  for (int32_t p = pos - W + 1; p <= pos; ++p)
#endif
  {
    if (p < 0) continue;
    slots[n++] = p % R;
  }
  return n;
}

static int valid_token(const orc_problem *P, int32_t t) {
  if (t < 0 || t >= P->T) return 0;
  int32_t b = P->q_seq[t];
  if (b < 0 || b >= P->B) return 0;
  if (P->q_pos[t] < 0) return 0;
  if (orc_n_vis(P->q_pos[t], P->r) > P->N_c) return 0;
  return 1;
}

/* ---- index scores -------------------------------------------------------- */

/* S[t,s] = sum_h w[t,h] * ReLU( sum_d q_hat[t,h,d] * k_hat[b,s,d] ) for the
 * visible positions s < n_vis(t); -inf elsewhere.  A[t,s] is the condition
 * magnitude sum_h |w[t,h]| * sum_d |q_hat[t,h,d] * k_hat[b,s,d]| that bounds
 * any rounding error of a finite-precision evaluation. */
static void score_token(const orc_problem *P, int32_t t, double *S, double *A) {
  const int64_t N_c = P->N_c, H_I = P->H_I, D_I = P->D_I;
  const int32_t b = P->q_seq[t];
  const int32_t nv = orc_n_vis(P->q_pos[t], P->r);
  for (int64_t s = 0; s < N_c; ++s) {
    double sum = 0.0, mag = 0.0;
    if (s >= nv) {
      S[s] = -INFINITY;
      if (A) A[s] = 0.0;
      continue;
    }
#if ORC_MUTANT == 3
    const int64_t krow = (int64_t)0 * N_c + s;
#else
    const int64_t krow = (int64_t)b * N_c + s;
#endif
#if ORC_MUTANT == 2
    const double ks = 1.0;
#else
    const double ks = P->k_scale ? (double)P->k_scale[krow] : 1.0;
#endif
    for (int64_t h = 0; h < H_I; ++h) {
#if ORC_MUTANT == 11
      const double qs = 1.0;
#else
      const double qs = P->q_scale ? (double)P->q_scale[t * H_I + h] : 1.0;
#endif
      double dot = 0.0, adot = 0.0;
#if ORC_MUTANT == 7
      for (int64_t d = 0; d < D_I - 1; ++d) {
#else
      for (int64_t d = 0; d < D_I; ++d) {
#endif
        const double qv = elem(P->q_I, P->q_dtype, (t * H_I + h) * D_I + d) * qs;
        const double kv = elem(P->k_I, P->k_dtype, krow * D_I + d) * ks;
        dot += qv * kv;
        adot += fabs(qv * kv);
      }
      const double wh = (double)P->w[t * H_I + h];
#if ORC_MUTANT == 1
      sum += wh * dot;
#elif ORC_MUTANT == 10
      sum += (dot > 0.0 ? dot : 0.0);
#else
      sum += wh * (dot > 0.0 ? dot : 0.0);
#endif
      mag += fabs(wh) * adot;
    }
    S[s] = sum;
    if (A) A[s] = mag;
  }
}

int32_t orc_index_scores(const orc_problem *P, const int32_t *rows, int32_t n_rows,
                         double *S, double *A) {
  for (int32_t i = 0; i < n_rows; ++i)
    if (!valid_token(P, rows[i])) return -1;
  const int64_t N_c = P->N_c;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t i = 0; i < n_rows; ++i)
    score_token(P, rows[i], S + i * N_c, A ? A + i * N_c : NULL);
  return 0;
}

/* ---- top-k --------------------------------------------------------------- */

typedef struct {
  double score;
  int32_t pos;
} scored_pos;

/* Higher score first; among equal scores the lower position first. */
static int by_score_then_pos(const void *a, const void *b) {
  const scored_pos *x = (const scored_pos *)a, *y = (const scored_pos *)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
#if ORC_MUTANT == 5
  return (x->pos > y->pos) ? -1 : (x->pos < y->pos);
#else
  return (x->pos < y->pos) ? -1 : (x->pos > y->pos);
#endif
}

static int ascending_int(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x < y) ? -1 : (x > y);
}

/* Keeps K_eff = min(K, n_vis) of the visible positions 0 .. n_vis-1, the
 * highest scores first with ties to the lower position, and writes them in
 * ascending position order followed by K - K_eff entries of -1.  Returns
 * K_eff. */
int32_t orc_topk_row(const double *S, int32_t n_vis, int32_t K, int32_t *idx) {
  if (n_vis < 0 || K < 0) return -1;
  int32_t k_eff = K < n_vis ? K : n_vis;
  scored_pos *all = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)(n_vis > 0 ? n_vis : 1));
  for (int32_t s = 0; s < n_vis; ++s) {
    all[s].score = S[s];
    all[s].pos = s;
  }
  qsort(all, (size_t)n_vis, sizeof(scored_pos), by_score_then_pos);
  for (int32_t i = 0; i < k_eff; ++i) idx[i] = all[i].pos;
  qsort(idx, (size_t)k_eff, sizeof(int32_t), ascending_int);
  for (int32_t i = k_eff; i < K; ++i) idx[i] = -1;
  free(all);
  return k_eff;
}

/* ---- two-level top-k, level one ------------------------------------------ */

/* "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", select_candidate_blocks (and
 * Indexer.forward, which calls it in the candidate source layer): positions
 * [0, N_c) of a score row are cut into blocks of bs, the last one short; a
 * block's score is the best score of its positions, where positions at or
 * past n_vis count as -inf (not reachable yet); the block holding the newest
 * visible position, (n_vis - 1) / bs, is pinned to +inf; the min(topk_blocks,
 * number of blocks) highest-scoring blocks are taken (ties: the lower block)
 * and those whose score is -inf are dropped.  keep[b] = 1 for a kept block.
 * Returns the number of blocks kept, or -1 on bad arguments. */
int32_t orc_candidate_blocks(const double *S, int32_t n_vis, int32_t N_c, int32_t bs, int32_t topk_blocks,
                             uint8_t *keep) {
  if (n_vis < 0 || N_c < 0 || n_vis > N_c || bs < 1 || topk_blocks < 0) return -1;
  const int32_t nb = (N_c + bs - 1) / bs;
  scored_pos *blk = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)(nb > 0 ? nb : 1));
  for (int32_t b = 0; b < nb; ++b) {
    double m = -INFINITY;
    for (int32_t s = b * bs; s < (b + 1) * bs && s < N_c; ++s)
      if (s < n_vis && S[s] > m) m = S[s];
    blk[b].score = m;
    blk[b].pos = b;
    keep[b] = 0;
  }
  if (n_vis >= 1) blk[(n_vis - 1) / bs].score = INFINITY;
  qsort(blk, (size_t)nb, sizeof(scored_pos), by_score_then_pos);
  const int32_t n = topk_blocks < nb ? topk_blocks : nb;
  int32_t kept = 0;
  for (int32_t i = 0; i < n; ++i)
    if (blk[i].score > -INFINITY) {
      keep[blk[i].pos] = 1;
      ++kept;
    }
  free(blk);
  return kept;
}

/* ---- V3.2 index producer: Hadamard rotation and fp8 quantisation -------- */

/* Nearest bfloat16 (ties to even) of a finite float, as bits. */
static uint16_t bf16_nearest(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof(u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* bfloat16 bits of sign * c * 2^q (c < 512 a count of quanta 2^q, already
 * rounded): renormalises a carry into the next binade and saturates to inf. */
static uint16_t bf16_encode(int sign, uint64_t c, int q) {
  if (c == 0) return sign ? 0x8000u : 0u;
  while (c >= 256) { /* only an exact power of two after a carry */
    c >>= 1;
    q += 1;
  }
  uint16_t bits;
  if (c < 128) {
    bits = (uint16_t)c; /* subnormal: q == -133 */
  } else {
    const int bexp = q + 7 + 127;
    bits = bexp >= 255 ? 0x7F80u : (uint16_t)((bexp << 7) | (int)(c - 128));
  }
  return sign ? (uint16_t)(bits | 0x8000u) : bits;
}

static int bitlen_u128(unsigned __int128 a) {
  int n = 0;
  while (a) {
    a >>= 1;
    ++n;
  }
  return n;
}

/* floor(sqrt(a)) of a 128-bit integer, bit by bit. */
static unsigned __int128 isqrt_u128(unsigned __int128 a) {
  unsigned __int128 r = 0;
  for (int b = 63; b >= 0; --b) {
    const unsigned __int128 t = r | ((unsigned __int128)1 << b);
    if (t * t <= a) r = t;
  }
  return r;
}

/* The bfloat16 nearest (ties to even) to v = A * 2^E, times sqrt(2) when
 * `root2` is set, decided exactly in integer arithmetic.  A < 2^62.  A product
 * with sqrt(2) is irrational, so it never ties. */
static uint16_t bf16_round_exact(int sign, uint64_t A, int E, int root2) {
  if (A == 0) return 0; /* an exact zero is +0 */
  const unsigned __int128 A2 = (unsigned __int128)A * A;
  const int L = bitlen_u128(A);
  int f = L - 1 + E; /* floor(log2 v) */
  if (root2 && A2 >= ((unsigned __int128)1 << (2 * L - 1))) f += 1;
  int q = f - 7; /* 8 significant bits */
  if (q < -133) q = -133;
  const int s = E - q; /* v / 2^q = A * 2^s (* sqrt 2) */
  uint64_t c;
  if (!root2) {
    if (s >= 0) return bf16_encode(sign, A << s, q);
    if (-s >= 64) return bf16_encode(sign, 0, q); /* far below half a quantum */
    const uint64_t fl = A >> -s, rem = A & ((1ull << -s) - 1), half = 1ull << (-s - 1);
    c = fl + ((rem > half || (rem == half && (fl & 1))) ? 1 : 0);
    return bf16_encode(sign, c, q);
  }
  /* c0 = floor(A sqrt2 2^s) = isqrt(floor(2 A^2 2^(2s))); round up iff
   * A sqrt2 2^s > c0 + 1/2, i.e. 8 A^2 2^(2s) > (2 c0 + 1)^2 */
  unsigned __int128 z;
  if (s >= 0)
    z = (2 * A2) << (2 * s);
  else
    z = (-2 * s >= 127) ? 0 : (2 * A2) >> (-2 * s);
  const uint64_t c0 = (uint64_t)isqrt_u128(z);
  const unsigned __int128 odd2 = (unsigned __int128)(2 * c0 + 1) * (2 * c0 + 1);
  int up;
  if (s >= 0)
    up = (8 * A2) << (2 * s) > odd2;
  else
    up = (-2 * s >= 120) ? 0 : (8 * A2 > (odd2 << (-2 * s)));
  c = c0 + (up ? 1 : 0);
  return bf16_encode(sign, c, q);
}

/* "DeepSeek-V3.2-Exp inference/model.py", rotate_activation: a bf16 row x of n
 * values (n a power of two) maps to y = H x * n^-1/2, H the Sylvester-Hadamard
 * matrix of order n (H[i][j] = (-1)^popcount(i & j)), returned in bf16.
 * Reading: y is the exact value rounded once to the nearest bfloat16 (ties to
 * even); the page calls a library whose internal precision and order it does
 * not show.  Each sum is formed exactly in integers (every bf16 value is an
 * integer multiple of the row's smallest quantum), then scaled by
 * n^-1/2 = 2^(-k/2) for n = 2^k (times sqrt 2 when k is odd) and rounded by an
 * exact comparison.  Returns -1 for a bad n, -2 when the row's exact sums do
 * not fit in 62 bits (a dynamic range beyond about 2^46 within one row). */
int32_t orc_hadamard_bf16(const uint16_t *x, int32_t n, uint16_t *y) {
  if (n < 1 || (n & (n - 1))) return -1;
  int k = 0;
  while ((1 << k) < n) ++k;
  /* x_j = m_j * 2^e_j with m_j an integer of at most 8 bits */
  int64_t *m = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
  int *e = (int *)malloc(sizeof(int) * (size_t)n);
  int emin = 1 << 30, emax = -(1 << 30);
  for (int32_t j = 0; j < n; ++j) {
    const int ex = (x[j] >> 7) & 0xFF, man = x[j] & 0x7F;
    m[j] = ex ? 128 + man : man;
    e[j] = ex ? ex - 127 - 7 : -133;
    if (x[j] & 0x8000) m[j] = -m[j];
    if (m[j] != 0) {
      if (e[j] < emin) emin = e[j];
      if (e[j] > emax) emax = e[j];
    }
  }
  int32_t rc = 0;
  if (emax >= emin && emax - emin + 8 + k > 61) rc = -2;
  for (int32_t i = 0; i < n && rc == 0; ++i) {
    int64_t N = 0;
    for (int32_t j = 0; j < n; ++j) {
      if (m[j] == 0) continue;
#if ORC_MUTANT == 12
      const int neg = __builtin_popcount((unsigned)(i ^ j)) & 1; /* wrong sign rule */
#else
      const int neg = __builtin_popcount((unsigned)(i & j)) & 1;
#endif
      const int64_t term = m[j] * ((int64_t)1 << (e[j] - emin));
      N += neg ? -term : term;
    }
    const int sign = N < 0;
    const uint64_t A = (uint64_t)(N < 0 ? -N : N);
    /* n^-1/2 = 2^(-k/2) for even k, 2^(-(k+1)/2) sqrt 2 for odd k */
    y[i] = bf16_round_exact(sign, A, emin - (k + 1) / 2, k & 1);
  }
  free(e);
  free(m);
  return rc;
}

/* The same rotation without the final rounding, in double (each exact sum
 * times n^-1/2, one rounding to double): what the bf16 result rounds. */
int32_t orc_hadamard_f64(const uint16_t *x, int32_t n, double *y) {
  if (n < 1 || (n & (n - 1))) return -1;
  for (int32_t i = 0; i < n; ++i) {
    long double acc = 0.0L; /* the row's sums are exact in 64 bits for the rows tests use */
    for (int32_t j = 0; j < n; ++j) {
      const double v = orc_bf16_value(x[j]);
      acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -(long double)v : (long double)v;
    }
    y[i] = (double)(acc / sqrtl((long double)n));
  }
  return 0;
}

/* The float8 e4m3fn code nearest to v (ties to the even code), saturating at
 * +-448, the largest finite value: from the format's definition (subnormals
 * are multiples of 2^-9 below 2^-6; a normal 1.m * 2^E has 3 mantissa bits). */
uint8_t orc_e4m3_encode(float v) {
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs((double)v);
  if (!(a < 448.0)) return sign | 0x7E;
#if ORC_MUTANT == 13
#define ORC_RINT round /* ties away from zero */
#else
#define ORC_RINT rint
#endif
  if (a < 0x1p-6) return sign | (uint8_t)ORC_RINT(a * 512.0); /* 8 is the smallest normal's code */
  int e;
  const double fr = frexp(a, &e); /* a = fr * 2^e, fr in [0.5, 1) */
  int E = e - 1;
  double m = ORC_RINT((2.0 * fr - 1.0) * 8.0);
  if (m == 8.0) {
    m = 0.0;
    E += 1;
  }
  int code = ((E + 7) << 3) | (int)m;
  if (code > 0x7E) code = 0x7E;
  return sign | (uint8_t)code;
}

/* act_quant over one block of n values (V3.2 Indexer.forward quantises each
 * head_dim = 128 row as one block; reading: the scale is amax / 448 in fp32,
 * the codes are e4m3(y / scale) with an fp32 division, and an all-zero block
 * gets scale 1).  y: bf16 bits. */
int32_t orc_act_quant_row(const uint16_t *y, int32_t n, uint8_t *codes, float *scale) {
  if (n < 1) return -1;
  float amax = 0.f;
  for (int32_t i = 0; i < n; ++i) {
    const float a = (float)fabs(orc_bf16_value(y[i]));
    if (a > amax) amax = a;
  }
#if ORC_MUTANT == 14
  const float s = amax > 0.f ? amax / 240.0f : 1.0f;
#else
  const float s = amax > 0.f ? amax / 448.0f : 1.0f;
#endif
  for (int32_t i = 0; i < n; ++i) codes[i] = orc_e4m3_encode((float)orc_bf16_value(y[i]) / s);
  *scale = s;
  return 0;
}

/* ---- V4.1 compressor: gated pooling of r tokens, then RMSNorm ------------- */

/* "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", RMSNorm.forward: c times
 * (mean over the D channels of c^2 + eps)^-1/2, times weight. */
static void rms_norm(double *c, int32_t D, const float *weight, double eps) {
  double ss = 0.0;
  for (int32_t d = 0; d < D; ++d) ss += c[d] * c[d];
#if ORC_MUTANT == 16
  const double inv = 1.0 / sqrt(ss + eps); /* sum instead of mean */
#else
  const double inv = 1.0 / sqrt(ss / (double)D + eps);
#endif
  for (int32_t d = 0; d < D; ++d) c[d] = c[d] * inv * (double)weight[d];
}

/* One group (same page, Compressor.forward): for every channel d, the r
 * tokens' kv values weighted by the softmax over the r tokens of their gate
 * scores, summed; rounded to bf16 (the cast to the activation dtype); then
 * rms_norm.  kv, score: [r, D] with row stride ld. */
static void pool_group(const float *kv, const float *score, int64_t ld, int32_t D, int32_t r, const float *weight,
                       double eps, double *out) {
#if ORC_MUTANT == 15
  /* softmax over the channels of each token instead of over the tokens */
  for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
  for (int32_t j = 0; j < r; ++j) {
    double m = -INFINITY, z = 0.0;
    for (int32_t d = 0; d < D; ++d) m = fmax(m, (double)score[j * ld + d]);
    for (int32_t d = 0; d < D; ++d) z += exp((double)score[j * ld + d] - m);
    for (int32_t d = 0; d < D; ++d) out[d] += (double)kv[j * ld + d] * exp((double)score[j * ld + d] - m) / z;
  }
#else
  for (int32_t d = 0; d < D; ++d) {
    double m = -INFINITY, z = 0.0, acc = 0.0;
    for (int32_t j = 0; j < r; ++j) m = fmax(m, (double)score[j * ld + d]);
    for (int32_t j = 0; j < r; ++j) {
      const double e = exp((double)score[j * ld + d] - m);
      z += e;
      acc += e * (double)kv[j * ld + d];
    }
    out[d] = acc / z;
  }
#endif
  /* the pooled row is cast to the activation dtype (bf16) before the norm:
   * Compressor.forward returns norm(kv.to(dtype)) */
  for (int32_t d = 0; d < D; ++d) out[d] = orc_bf16_value(bf16_nearest((float)out[d]));
  rms_norm(out, D, weight, eps);
}

/* Prefill of one sequence from position 0 (Compressor.forward, start_pos == 0):
 * kv and score [S, D] (the fp32 projections wkv(x), wgate(x)); ratio r >= 2.
 * Writes the S / r complete groups to out [S / r, D] (before the cast to the
 * activation dtype) and the trailing S % r tokens to slots 0 .. S % r - 1 of
 * the state [r, D] (kv_state, score_state; may be NULL).  Returns S / r. */
int32_t orc_compress_prefill(const float *kv, const float *score, int32_t S, int32_t D, int32_t r,
                             const float *weight, double eps, double *out, float *kv_state, float *score_state) {
  if (S < 0 || D < 1 || r < 2) return -1;
  const int32_t G = S / r;
  for (int32_t g = 0; g < G; ++g)
    pool_group(kv + (int64_t)g * r * D, score + (int64_t)g * r * D, D, D, r, weight, eps, out + (int64_t)g * D);
  if (kv_state && score_state)
    for (int32_t j = 0; j < S - G * r; ++j)
      for (int32_t d = 0; d < D; ++d) {
        kv_state[(int64_t)j * D + d] = kv[((int64_t)G * r + j) * D + d];
        score_state[(int64_t)j * D + d] = score[((int64_t)G * r + j) * D + d];
      }
  return G;
}

/* One decode step at absolute position pos (start_pos > 0): the token goes to
 * slot pos % r of the state; when the group just completed ((pos + 1) % r ==
 * 0) the state's r slots are pooled into out [D] and 1 is returned, else 0. */
int32_t orc_compress_decode(const float *kv_tok, const float *score_tok, int32_t pos, int32_t D, int32_t r,
                            float *kv_state, float *score_state, const float *weight, double eps, double *out) {
  if (pos < 0 || D < 1 || r < 2) return -1;
#if ORC_MUTANT == 17
  const int32_t slot = (pos + 1) % r;
#else
  const int32_t slot = pos % r;
#endif
  for (int32_t d = 0; d < D; ++d) {
    kv_state[(int64_t)slot * D + d] = kv_tok[d];
    score_state[(int64_t)slot * D + d] = score_tok[d];
  }
  if ((pos + 1) % r != 0) return 0;
  pool_group(kv_state, score_state, D, D, r, weight, eps, out);
  return 1;
}

/* ---- V4.1 rotary embedding (YaRN) ------------------------------------------ */

/* "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", precompute_freqs_cis: the
 * angle of pair i (i < dim / 2) at position pos.  The base frequency is
 * base^(-2i / dim); with original_seq_len > 0 (YaRN) the pairs below the
 * corrected dimension of beta_fast keep it, those above that of beta_slow are
 * divided by factor, and a linear ramp fades between them (low, high: floor
 * and ceil of the corrected dimensions, clamped to [0, dim - 1]; the ramp's
 * span is at least 1e-3).  The page computes the frequencies in fp32; the
 * oracle takes them in double.  angle = pos * freq. */
double orc_rope_angle(int32_t dim, int32_t i, int64_t pos, double base, double factor, int32_t original_seq_len,
                      double beta_fast, double beta_slow) {
  double freq = 1.0 / pow(base, (double)(2 * i) / (double)dim);
  if (original_seq_len > 0) {
    const double lo_d = dim * log(original_seq_len / (beta_fast * 2.0 * M_PI)) / (2.0 * log(base));
    const double hi_d = dim * log(original_seq_len / (beta_slow * 2.0 * M_PI)) / (2.0 * log(base));
    const double low = fmax(floor(lo_d), 0.0);
    const double high = fmin(ceil(hi_d), (double)(dim - 1));
    double ramp = ((double)i - low) / fmax(high - low, 1e-3);
    ramp = fmin(fmax(ramp, 0.0), 1.0);
    const double smooth = 1.0 - ramp;
#if ORC_MUTANT == 18
    freq = freq / factor * smooth + freq * (1.0 - smooth); /* ramp reversed */
#else
    freq = freq / factor * (1.0 - smooth) + freq * smooth;
#endif
  }
  return (double)pos * freq;
}

/* Same page, apply_rotary_emb: adjacent pairs (x[2i], x[2i+1]) of a row of
 * dim values taken as complex numbers and multiplied by e^(i angle_i) (its
 * conjugate when inverse is set), in place, in double. */
void orc_apply_rope(double *x, int32_t dim, int64_t pos, double base, double factor, int32_t original_seq_len,
                    double beta_fast, double beta_slow, int32_t inverse) {
  for (int32_t i = 0; i < dim / 2; ++i) {
    const double a = orc_rope_angle(dim, i, pos, base, factor, original_seq_len, beta_fast, beta_slow);
    const double c = cos(a), s = inverse ? -sin(a) : sin(a);
    const double re = x[2 * i], im = x[2 * i + 1];
    x[2 * i] = re * c - im * s;
    x[2 * i + 1] = re * s + im * c;
  }
}

/* ---- V4.1 index keys of a compressing layer ------------------------------- */

/* The bfloat16 nearest (ties to even) to a finite double, rounded once. */
static uint16_t bf16_nearest_d(double v) {
  const uint16_t sign = signbit(v) ? 0x8000u : 0u;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e); /* a = f 2^e, f in [0.5, 1): the leading bit has weight 2^(e-1) */
  int q = e - 1 - 7;  /* quantum of 8 significant bits */
  if (q < -133) q = -133; /* subnormal range */
  double c = rint(ldexp(a, -q)); /* exact scaling, one rounding (ties to even) */
  if (c >= 256.0) { /* carried into the next binade */
    c = 128.0;
    q += 1;
  }
  uint16_t bits;
  if (c < 128.0) {
    bits = (uint16_t)c; /* subnormal */
  } else {
    const int bexp = q + 7 + 127;
    bits = bexp >= 255 ? 0x7F80u : (uint16_t)((bexp << 7) | (int)(c - 128.0));
  }
  return sign | bits;
}

/* "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Indexer.forward in a layer
 * that owns the index keys: k = k_norm(wk(latent)), then apply_rotary_emb on
 * the last rope_dim values at the position of the group's first token, then
 * the key's quantisation, then the write to the key cache at row
 * start_pos // ratio.  Here x is one row of wk(latent) (bf16, D values):
 *   RMSNorm.forward: y = weight * x / sqrt(mean(x^2) + eps), cast to bf16;
 *   the rotation of pairs (y[D - rope_dim + 2i], y[D - rope_dim + 2i + 1]) by
 *   the angle of pair i at `pos` (orc_rope_angle), cast back to bf16;
 *   the page's fp4 block quantisation read as the V3.2 act_quant of one
 *   128-value block: scale = amax / 448 and e4m3 codes (orc_act_quant_row).
 * Arithmetic in double between the two bf16 roundings, each a single
 * rounding of the exact value; the quantiser in fp32.  k_bf16 (optional)
 * receives the bf16 key before quantisation. */
int32_t orc_index_key(const uint16_t *x, int32_t D, const float *weight, double eps, int64_t pos, int32_t rope_dim,
                      double base, double factor, int32_t original_seq_len, double beta_fast, double beta_slow,
                      uint8_t *codes, float *scale, uint16_t *k_bf16) {
  if (D < 1 || rope_dim < 0 || rope_dim > D || (rope_dim & 1) || pos < 0) return -1;
  double *v = (double *)malloc(sizeof(double) * (size_t)D);
  uint16_t *k = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)D);
  double ss = 0.0;
  for (int32_t d = 0; d < D; ++d) {
    v[d] = orc_bf16_value(x[d]);
    ss += v[d] * v[d];
  }
#if ORC_MUTANT == 23
  const double inv = 1.0 / sqrt(ss / (double)D); /* eps left out */
#else
  const double inv = 1.0 / sqrt(ss / (double)D + eps);
#endif
  for (int32_t d = 0; d < D; ++d) k[d] = bf16_nearest_d((double)weight[d] * (v[d] * inv));
#if ORC_MUTANT == 22
  const int32_t r0 = 0; /* the rotation applied to the first rope_dim values */
#else
  const int32_t r0 = D - rope_dim;
#endif
  for (int32_t d = 0; d < rope_dim; ++d) v[d] = orc_bf16_value(k[r0 + d]);
  orc_apply_rope(v, rope_dim, pos, base, factor, original_seq_len, beta_fast, beta_slow, 0);
  for (int32_t d = 0; d < rope_dim; ++d) k[r0 + d] = bf16_nearest_d(v[d]);
  if (k_bf16) memcpy(k_bf16, k, sizeof(uint16_t) * (size_t)D);
  orc_act_quant_row(k, D, codes, scale);
  free(k);
  free(v);
  return 0;
}

/* ---- sparse attention ---------------------------------------------------- */

/* For query token t (sequence b, position p) the key set J is the window rows
 * (ring slots of Kw/Vw) followed by the compressed rows idx[t, :] that are not
 * -1.  For each head h: l_j = scale * Q[t,h] . K_j, a_j = exp(l_j - m) / Z with
 * m = max_j l_j and Z = sum_j exp(l_j - m) (+ exp(sink_h - m) when a sink is
 * given), and O[t,h] = sum_j a_j V_j. */
static void attn_token(const orc_problem *P, int32_t t, const int32_t *idx_row, int32_t K,
                       double *O) {
  const int64_t H = P->H, D = P->D, R = P->R, N_c = P->N_c;
  const int32_t b = P->q_seq[t];
  int32_t *slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)(P->W > 0 ? P->W : 1));
  const int32_t nw = orc_window_slots(P->q_pos[t], P->W, P->R, slots);
  const int32_t nj = nw + K;
  const uint16_t **krows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nj > 0 ? nj : 1));
  const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(nj > 0 ? nj : 1));
  double *logit = (double *)malloc(sizeof(double) * (size_t)(nj > 0 ? nj : 1));
  int32_t n = 0;
  for (int32_t j = 0; j < nw; ++j) {
    krows[n] = P->Kw + ((int64_t)b * R + slots[j]) * D;
    vrows[n] = P->Vw + ((int64_t)b * R + slots[j]) * D;
    ++n;
  }
  for (int32_t k = 0; k < K; ++k) {
    const int32_t c = idx_row[k];
    if (c < 0) continue;
    krows[n] = P->Kc + ((int64_t)b * N_c + c) * D;
    vrows[n] = P->Vc + ((int64_t)b * N_c + c) * D;
    ++n;
  }
  for (int64_t h = 0; h < H; ++h) {
    const uint16_t *q = P->Q + ((int64_t)t * H + h) * D;
    double m = -INFINITY;
    for (int32_t j = 0; j < n; ++j) {
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d) dot += orc_bf16_value(q[d]) * orc_bf16_value(krows[j][d]);
#if ORC_MUTANT == 9
      logit[j] = -(double)P->scale * dot;
#else
      logit[j] = (double)P->scale * dot;
#endif
      if (logit[j] > m) m = logit[j];
    }
#if ORC_MUTANT == 21
    const double sink = P->sink ? (double)P->scale * (double)P->sink[h] : 0.0; /* sink taken as a dot product */
#else
    const double sink = P->sink ? (double)P->sink[h] : 0.0;
#endif
    if (P->sink && sink > m) m = sink;
    double Z = 0.0;
    for (int32_t j = 0; j < n; ++j) Z += exp(logit[j] - m);
#if ORC_MUTANT != 20 /* mutant 20: the sink left out of the denominator */
    if (P->sink) Z += exp(sink - m);
#endif
    double *o = O + h * D;
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
#if ORC_MUTANT == 19
    /* the sink taken as a key whose value row is all ones (it joins the numerator too) */
    if (P->sink)
      for (int64_t d = 0; d < D; ++d) o[d] += exp(sink - m) / Z;
#endif
    for (int32_t j = 0; j < n; ++j) {
      const double a = exp(logit[j] - m) / Z;
#if ORC_MUTANT == 8
      const uint16_t *v = krows[j];
#else
      const uint16_t *v = vrows[j];
#endif
      for (int64_t d = 0; d < D; ++d) o[d] += a * orc_bf16_value(v[d]);
    }
  }
  free(logit);
  free(vrows);
  free(krows);
  free(slots);
}

static int valid_idx_row(const orc_problem *P, int32_t t, const int32_t *idx_row, int32_t K) {
  const int32_t nv = orc_n_vis(P->q_pos[t], P->r);
  for (int32_t k = 0; k < K; ++k)
    if (idx_row[k] < -1 || idx_row[k] >= nv) return 0;
  return 1;
}

int32_t orc_sparse_attn(const orc_problem *P, const int32_t *idx, int32_t K,
                        const int32_t *rows, int32_t n_rows, double *O) {
  for (int32_t i = 0; i < n_rows; ++i)
    if (!valid_token(P, rows[i]) || !valid_idx_row(P, rows[i], idx + (int64_t)rows[i] * K, K))
      return -1;
  const int64_t HD = (int64_t)P->H * P->D;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t i = 0; i < n_rows; ++i)
    attn_token(P, rows[i], idx + (int64_t)rows[i] * K, K, O + i * HD);
  return 0;
}

/* ---- the whole step --------------------------------------------------------
 * Scores, top-k and attention for the tokens rows[0..n_rows), one token at a
 * time.  idx and O are written compactly (row i for token rows[i]). */
int32_t orc_fused(const orc_problem *P, int32_t K, const int32_t *rows, int32_t n_rows,
                  int32_t *idx, double *O) {
  for (int32_t i = 0; i < n_rows; ++i)
    if (!valid_token(P, rows[i])) return -1;
  const int64_t HD = (int64_t)P->H * P->D;
#pragma omp parallel for schedule(dynamic, 1)
  for (int32_t i = 0; i < n_rows; ++i) {
    const int32_t t = rows[i];
    double *S = (double *)malloc(sizeof(double) * (size_t)(P->N_c > 0 ? P->N_c : 1));
    score_token(P, t, S, NULL);
    orc_topk_row(S, orc_n_vis(P->q_pos[t], P->r), K, idx + (int64_t)i * K);
    attn_token(P, t, idx + (int64_t)i * K, K, O + i * HD);
    free(S);
  }
  return 0;
}

void orc_set_threads(int32_t n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int32_t orc_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
