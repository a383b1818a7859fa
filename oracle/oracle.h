/*
 * Float64 CPU oracle for the indexer-selected sparse attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the tests, the package smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or table with the
 * CUDA library.
 *
 * Every input is passed as raw storage bits (bf16 as uint16, fp8-e4m3fn as
 * uint8) plus fp32 scale/weight arrays, exactly as the GPU library receives
 * them; the oracle decodes each element from its format definition and does
 * all arithmetic in IEEE double.
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_FP8_E4M3 = 1 };

/* One problem: the indexer inputs and the attention inputs of T query tokens
 * drawn from B sequences.  All arrays are dense row-major on the host. */
typedef struct {
  int32_t B, T;
  int32_t r;          /* compression ratio: compressed entry j covers tokens [j*r, (j+1)*r) */
  int32_t N_c;        /* compressed rows stored per sequence */
  const int32_t *q_seq; /* [T] sequence of each query token */
  const int32_t *q_pos; /* [T] absolute position of each query token */
  /* indexer */
  int32_t H_I, D_I;
  const void *q_I; int32_t q_dtype; const float *q_scale; /* [T,H_I,D_I]; q_scale [T,H_I] or NULL */
  const float *w;                                         /* [T,H_I] head weights */
  const void *k_I; int32_t k_dtype; const float *k_scale; /* [B,N_c,D_I]; k_scale [B,N_c] or NULL */
  /* attention (one shared KV head) */
  int32_t H, D, W, R; /* query heads, head dim, window length, raw ring slots */
  const uint16_t *Q;  /* [T,H,D] bf16 bits */
  const uint16_t *Kw, *Vw; /* [B,R,D] bf16 bits: raw ring, slot = position mod R */
  const uint16_t *Kc, *Vc; /* [B,N_c,D] bf16 bits: compressed rows */
  const float *sink;  /* [H] or NULL */
  float scale;        /* softmax scale */
} orc_problem;

double orc_bf16_value(uint16_t bits);
double orc_e4m3_value(uint8_t bits);
int32_t orc_n_vis(int32_t pos, int32_t r);
int32_t orc_window_slots(int32_t pos, int32_t W, int32_t R, int32_t *slots);

/* Each "rows" function evaluates the query tokens rows[0..n_rows) and writes
 * output i for token rows[i].  Return 0 on success, -1 on invalid input. */
int32_t orc_index_scores(const orc_problem *P, const int32_t *rows, int32_t n_rows,
                         double *S /*[n_rows,N_c]*/, double *A /*[n_rows,N_c] or NULL*/);
int32_t orc_topk_row(const double *S, int32_t n_vis, int32_t K, int32_t *idx /*[K]*/);
int32_t orc_candidate_blocks(const double *S, int32_t n_vis, int32_t N_c, int32_t bs, int32_t topk_blocks,
                             uint8_t *keep /*[ceil(N_c / bs)]*/);
int32_t orc_hadamard_bf16(const uint16_t *x, int32_t n, uint16_t *y);
int32_t orc_hadamard_f64(const uint16_t *x, int32_t n, double *y);
uint8_t orc_e4m3_encode(float v);
int32_t orc_act_quant_row(const uint16_t *y, int32_t n, uint8_t *codes, float *scale);
int32_t orc_compress_prefill(const float *kv, const float *score, int32_t S, int32_t D, int32_t r,
                             const float *weight, double eps, double *out, float *kv_state, float *score_state);
double orc_rope_angle(int32_t dim, int32_t i, int64_t pos, double base, double factor, int32_t original_seq_len,
                      double beta_fast, double beta_slow);
void orc_apply_rope(double *x, int32_t dim, int64_t pos, double base, double factor, int32_t original_seq_len,
                    double beta_fast, double beta_slow, int32_t inverse);
int32_t orc_index_key(const uint16_t *x, int32_t D, const float *weight, double eps, int64_t pos, int32_t rope_dim,
                      double base, double factor, int32_t original_seq_len, double beta_fast, double beta_slow,
                      uint8_t *codes, float *scale, uint16_t *k_bf16);
int32_t orc_compress_decode(const float *kv_tok, const float *score_tok, int32_t pos, int32_t D, int32_t r,
                            float *kv_state, float *score_state, const float *weight, double eps, double *out);
int32_t orc_sparse_attn(const orc_problem *P, const int32_t *idx /*[T,K]*/, int32_t K,
                        const int32_t *rows, int32_t n_rows, double *O /*[n_rows,H,D]*/);
int32_t orc_fused(const orc_problem *P, int32_t K, const int32_t *rows, int32_t n_rows,
                  int32_t *idx /*[n_rows,K]*/, double *O /*[n_rows,H,D]*/);
void orc_set_threads(int32_t n);
int32_t orc_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
