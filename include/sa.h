/*
 * sa.h -- C ABI of the GB300 (sm_103a) sparse attention step:
 *
 *   index scores  ->  per-query top-k  ->  windowed + sparse MQA  (+ split-KV combine)
 *
 * The step is the one of "DeepSeek-V4.1-Flash-NVFP4 inference/model.py"
 * (Indexer.forward, get_window_topk_idxs, Attention._window_kv,
 * Attention.forward) with the fp8 index keys and per-position key scales of
 * "DeepSeek-V3.2-Exp inference/model.py" (Indexer.forward, fp8_index).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Notation: B sequences, T query tokens, token t belongs to sequence
 * q_seq[t] and sits at absolute position q_pos[t].  Compressed entry j of a
 * sequence stands for its tokens [j*r, (j+1)*r); token t can see the entries
 * j < n_vis(t) = floor((q_pos[t] + 1) / r) (Indexer.forward, "compress_lens").
 * Its raw window is the positions max(0, p-W+1) .. p, its own token included
 * (Attention._window_kv writes the token before attending), stored in a ring
 * of R slots per sequence at slot = position mod R.
 *
 * Memory: every pointer argument except the argument structs themselves is a
 * DEVICE pointer owned by the caller, 16-byte aligned, holding a dense
 * row-major array of the stated shape.  The library never allocates or frees
 * device memory: scratch comes from a caller workspace of
 * sa_workspace_size() bytes, which must be zero-filled once before its first
 * use (sa_workspace_init).  All work is enqueued on the caller's stream; no
 * call synchronises except sa_check_device_status.  Calls that share a
 * workspace must not run concurrently.
 *
 * Errors: arguments are checked on the host before anything is enqueued; a
 * bad argument returns an error and enqueues nothing.  sa_last_error_detail()
 * gives a one-line reason for the last error of the calling thread.  Values
 * that only the device sees (q_seq out of range, a position whose n_vis
 * exceeds N_c, an index >= n_vis) are never dereferenced: the kernels skip
 * them and set a sticky flag in the workspace, which sa_check_device_status
 * reports (SA_ERR_DEVICE_DATA) and clears.  No kernel traps or spins without
 * a bound.
 */
#ifndef SA_H
#define SA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SA_API __attribute__((visibility("default")))
#else
#define SA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st *sa_stream_t;

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1, /* null, negative, misaligned, or inconsistent argument */
  SA_ERR_UNSUPPORTED = 2, /* a shape or dtype combination outside the compiled kernels */
  SA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than sa_workspace_size() */
  SA_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
  SA_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (reported by sa_check_device_status) */
  SA_ERR_DEVICE_DATA = 6  /* device-resident data was out of range and skipped */
} sa_status;

typedef enum { SA_BF16 = 0, SA_FP8_E4M3 = 1 } sa_dtype;

/* Indexer inputs ("DeepSeek-V3.2-Exp inference/model.py", Indexer.forward:
 * fp8 q with a per-(token, head) scale, fp8 k_cache with a per-position
 * fp32 k_scale_cache; "DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
 * Indexer.forward: bf16-valued q and k). */
typedef struct {
  int32_t B, T;        /* sequences, query tokens (T >= 0, B >= 1) */
  int32_t H_I, D_I;    /* index heads (1..128), index head dim (64 or 128) */
  int32_t N_c;         /* compressed rows stored per sequence (>= 1) */
  int32_t r;           /* compression ratio (>= 1) */
  const int32_t *q_seq; /* [T] sequence id of each token, in [0, B) */
  const int32_t *q_pos; /* [T] absolute position of each token, >= 0 */
  const void *q_I;     /* [T, H_I, D_I] index queries, bf16 or fp8-e4m3fn */
  int32_t q_dtype;     /* sa_dtype of q_I */
  const float *q_scale; /* [T, H_I] dequantisation scale of q_I (> 0), or NULL for 1 */
  const float *w;      /* [T, H_I] head weights, used as given (callers fold
                          softmax_scale * H_I^-0.5 and any q scale into them
                          or pass q_scale) */
  const void *k_I;     /* [B, N_c, D_I] index keys, bf16 or fp8-e4m3fn (rows of sequence b
                          start k_seq_stride elements after those of b - 1) */
  int32_t k_dtype;     /* sa_dtype of k_I */
  const float *k_scale; /* [B, N_c] dequantisation scale of each key row (> 0), or NULL for 1;
                           sequence stride k_seq_stride / D_I */
  int64_t k_seq_stride; /* elements of k_I between consecutive sequences: 0 for dense
                           (N_c * D_I), else a multiple of D_I of at least N_c * D_I -- e.g. a
                           cache allocated for max_seq_len / r rows of which N_c are in use
                           ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Indexer.__init__
                           k_cache and Indexer.forward index_k[:bsz, :end_pos // ratio]) */
} sa_index_args;

/* Attention inputs: one shared KV head across H query heads
 * ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Attention.forward:
 * sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale) over the window KV
 * concatenated with the compressed KV). */
typedef struct {
  int32_t H, D;        /* query heads and head dim: D 128 with H 16/32/64/128, or D 512
                          (the released V4.1 shape) with H 16/32/64 */
  int32_t W;           /* window length (>= 1) */
  int32_t R;           /* raw ring slots per sequence (>= W; a prefill chunk of n
                          tokens needs R >= n + W - 1) */
  const void *Q;       /* [T, H, D] bf16 queries */
  const void *Kw;      /* [B, R, D] bf16 raw window keys, slot = position mod R */
  const void *Vw;      /* [B, R, D] bf16 raw window values (may equal Kw) */
  const void *Kc;      /* [B, N_c, D] bf16 compressed keys */
  const void *Vc;      /* [B, N_c, D] bf16 compressed values (may equal Kc; when Vw == Kw
                          and Vc == Kc -- V4.1's single kv -- each row is read once) */
  const float *sink;   /* [H] per-head attention sink logit, or NULL for none */
  float scale;         /* softmax scale applied to Q.K (e.g. D^-0.5) */
  int64_t w_seq_stride; /* elements of Kw / Vw between consecutive sequences: 0 for dense
                           (R * D), else a multiple of D of at least R * D */
  int64_t c_seq_stride; /* elements of Kc / Vc between consecutive sequences: 0 for dense
                           (N_c * D), else a multiple of D of at least N_c * D ("DeepSeek-V4.1-
                           Flash-NVFP4 inference/model.py", Attention.__init__ compress_kv_cache
                           of max_seq_len / ratio rows) */
} sa_attn_args;

/* Bytes of workspace the calls below need for these shapes and this K
 * (attn may be NULL for sa_indexer_scores / sa_topk alone).  Returns 0 when
 * the arguments are invalid. */
SA_API size_t sa_workspace_size(const sa_index_args *ia, const sa_attn_args *aa, int32_t K);

/* Zero-fills the workspace header (the sticky device status word).  Call it
 * once on a new workspace.  Enqueued on `stream`. */
SA_API sa_status sa_workspace_init(void *ws, size_t ws_bytes, sa_stream_t stream);

/* Index scores ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
 * Indexer.forward: einsum over the head dim, ReLU, times weights, sum over
 * index heads; "DeepSeek-V3.2-Exp inference/model.py", fp8_index):
 *
 *   scores[t, s] = sum_h w[t,h] * ReLU( sum_d q[t,h,d] q_scale[t,h] * k[b,s,d] k_scale[b,s] )
 *
 * for s < n_vis(t) (b = q_seq[t]) and -inf for n_vis(t) <= s < N_c.
 * scores: [T, ld] fp32, device; columns 0 .. N_c - 1 of every row are written,
 * the rest untouched.  ld >= N_c (a multiple of 4 keeps rows 16-byte aligned,
 * which the top-k entry points read fastest).  Arithmetic: the products are
 * exact in fp32 and accumulated in fp32. */
SA_API sa_status sa_indexer_scores(const sa_index_args *ia, float *scores, int64_t ld, void *ws,
                                   size_t ws_bytes, sa_stream_t stream);

/* Per-query top-k ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
 * Indexer.forward: topk = min(index_topk, n_vis); the picks re-sorted into
 * position order; unreachable picks are -1).  For each token t keeps
 * K_eff = min(K, n_vis(t)) positions s < n_vis(t) with the highest
 * scores[t, s] (ties: the lower position wins) and writes them in ascending
 * order to idx[t, 0 .. K_eff), then -1 to idx[t, K_eff .. K).
 * scores: [T, ld] fp32, ld >= N_c (only s < n_vis(t) is read); idx: [T, K]
 * int32.  K may be 0.  The selection is exact on the fp32 values (no
 * tolerance). */
SA_API sa_status sa_topk(const float *scores, int64_t ld, const sa_index_args *ia, int32_t K, int32_t *idx,
                         void *ws, size_t ws_bytes, sa_stream_t stream);

/* Two-level top-k, level one ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
 * select_candidate_blocks, called by Indexer.forward in the layer that is the
 * candidate source).  Positions [0, N_c) are cut into
 * nb = ceil(N_c / block_size) blocks, the last one short.  For token t, block
 * b scores max{ scores[t, s] : s in block b, s < n_vis(t) }, or -inf when it
 * holds no visible position; the block holding the newest visible position,
 * (n_vis(t) - 1) / block_size, scores +inf instead.  The min(topk_blocks, nb)
 * highest-scoring blocks are taken (ties: the lower block wins) and those
 * scoring -inf are dropped.  A kept block b sets bit b % 32 of cand[t, b / 32];
 * every other bit of the row, those past nb included, is 0.
 * scores: [T, ld] fp32, ld >= N_c (only s < n_vis(t) is read; NaN scores give
 * unspecified picks); cand: [T, sa_candidate_words(N_c, block_size)] uint32,
 * written in full.  block_size >= 1, topk_blocks >= 0; nb > 32768 or
 * N_c > 2^30 returns SA_ERR_UNSUPPORTED.  The selection is exact on the fp32 values.  The
 * workspace needs only its 256-byte header (the status word). */
SA_API sa_status sa_candidate_blocks(const float *scores, int64_t ld, const sa_index_args *ia, int32_t block_size,
                                     int32_t topk_blocks, uint32_t *cand, void *ws, size_t ws_bytes,
                                     sa_stream_t stream);

/* uint32 words per token row of a candidate block mask:
 * ceil(ceil(N_c / block_size) / 32); 0 when N_c < 1 or block_size < 1. */
SA_API int32_t sa_candidate_words(int32_t N_c, int32_t block_size);

/* Two-level top-k, level two (Indexer.forward in a layer that uses the
 * candidates: its own scores masked to -inf outside the candidate blocks, then
 * the top-k of sa_topk).  Equals sa_topk on scores with scores[t, s] replaced
 * by -inf wherever bit (s / block_size) of cand[t] is clear: the K_eff =
 * min(K, n_vis(t)) picks are the positions of kept blocks by score and, when
 * fewer than K_eff visible positions lie in kept blocks, then the lowest
 * visible positions outside them (-inf ties go to the lower position).
 * cand: [T, sa_candidate_words(N_c, block_size)] uint32, e.g. from
 * sa_candidate_blocks (of this or another layer's scores).  N_c > 2^30
 * returns SA_ERR_UNSUPPORTED.  Other arguments and the output as for
 * sa_topk. */
SA_API sa_status sa_topk_candidates(const float *scores, int64_t ld, const sa_index_args *ia, int32_t K,
                                    const uint32_t *cand, int32_t block_size, int32_t *idx, void *ws,
                                    size_t ws_bytes, sa_stream_t stream);

/* Index producer of the uncompressed indexer ("DeepSeek-V3.2-Exp
 * inference/model.py", Indexer.forward: rotate_activation, act_quant of q and
 * k, the k_cache / k_scale_cache write).  For each row r of x ([rows, dim]
 * bf16, dim 128): y = bf16(H x_r * 128^-1/2), H the Sylvester-Hadamard matrix
 * (H[i][j] = (-1)^popcount(i & j)), computed in fp32 by the butterfly stages
 * h = 1, 2, ..., 64 in that order; then scale = amax|y| / 448 (fp32; 1 for an
 * all-zero row) and codes = float8 e4m3fn of y / scale (nearest, ties to
 * even, saturating at +-448).  The codes and the scale go to row d of codes
 * ([*, 128] uint8) and scales ([*] fp32), with d = r when dst is NULL and
 * d = dst[r] otherwise (e.g. b * N_c + position for the index key cache of r =
 * 1); a d outside [0, dst_rows) is skipped and flagged (sa_check_device_status
 * reports SA_ERR_DEVICE_DATA).  x 16-byte aligned; codes, scales and dst 4-byte
 * aligned; dim other than 128 returns SA_ERR_UNSUPPORTED.  The workspace needs
 * only its 256-byte header.  Feeding the codes and scales to sa_indexer_scores
 * (fp8 queries with q_scale, fp8 keys with k_scale) gives the V3.2 index score. */
SA_API sa_status sa_rotate_quant(const void *x, int32_t rows, int32_t dim, const int32_t *dst, int64_t dst_rows,
                                 uint8_t *codes, float *scales, void *ws, size_t ws_bytes, sa_stream_t stream);

/* Compressor from position 0 ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
 * Compressor.forward with start_pos 0, and RMSNorm.forward).  kv and score:
 * [B, S, D] fp32 (the projections wkv(x) and wgate(x)); for sequence b and
 * group g < S / r (tokens g*r .. g*r + r - 1):
 *   c[d] = bf16( sum_j softmax_j(score[b, g*r + j, d]) kv[b, g*r + j, d] )
 *   out[b, g, d] = bf16( weight[d] * c[d] / sqrt(mean_d c[d]^2 + eps) )
 * in fp32.  out: [B, S / r, D] bf16.  The trailing S % r tokens are the
 * partial group that decode steps complete: with kv_state and score_state
 * ([B, r, D] fp32, both or neither) they are copied to slots 0 .. S % r - 1,
 * as the page splits them into kv_state / score_state.
 * r >= 2; D a multiple of 32 in [32, 1024]; B <= 65535; eps >= 0. */
SA_API sa_status sa_compress_prefill(const float *kv, const float *score, int32_t B, int32_t S, int32_t D, int32_t r,
                                     const float *weight, float eps, void *out, float *kv_state, float *score_state,
                                     sa_stream_t stream);

/* One compressor decode step ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
 * Compressor.forward with start_pos > 0): for every sequence b, the token at
 * absolute position pos[b] (its projections kv[b], score[b]: [B, D] fp32)
 * fills slot pos[b] % r of the state (kv_state, score_state: [B, r, D] fp32,
 * caller-owned and kept across steps; a sequence that starts without a
 * prefill begins with kv_state 0 and score_state -inf, as the page's buffers
 * do).  When the group has just completed, (pos[b] + 1) % r == 0, its r slots
 * are pooled and normalised exactly as in sa_compress_prefill and written to
 * out[b] ([B, D] bf16); the other rows of out are left untouched.  A negative
 * pos[b] is skipped and flagged in the workspace status word
 * (sa_check_device_status reports SA_ERR_DEVICE_DATA); the workspace needs
 * only its 256-byte header.  Same limits on r, D, B and eps as
 * sa_compress_prefill. */
SA_API sa_status sa_compress_decode(const float *kv, const float *score, const int32_t *pos, int32_t B, int32_t D,
                                    int32_t r, float *kv_state, float *score_state, const float *weight, float eps,
                                    void *out, void *ws, size_t ws_bytes, sa_stream_t stream);

/* Rotary embedding parameters ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
 * precompute_freqs_cis and apply_rotary_emb): pair i < dim / 2 of the rotated
 * values turns by pos * f_i with f_i = base^(-2i / dim), and, when
 * original_seq_len > 0, YaRN's correction: pairs below the corrected dimension
 * of beta_fast keep f_i, those above that of beta_slow take f_i / factor, and
 * a linear ramp fades between (the page's low / high bounds, span at least
 * 1e-3).  Pairs are adjacent values (x[2i], x[2i + 1]) taken as complex
 * numbers. */
typedef struct {
  int32_t dim;              /* rotated values at the end of the row (rope_head_dim) */
  double base;              /* rope theta (compress_rope_theta for compressed rows) */
  double factor;            /* YaRN factor */
  int32_t original_seq_len; /* > 0 applies YaRN */
  double beta_fast, beta_slow;
} sa_rope_args;

/* Index keys of the layer that owns them ("DeepSeek-V4.1-Flash-NVFP4
 * inference/model.py", Indexer.forward: k = k_norm(wk(latent)),
 * apply_rotary_emb on its last rope_head_dim values at the position of the
 * group's first token, the key quantisation, k_cache[:, start_pos // ratio]).
 * kproj: [n, D_I] bf16, row i = wk(latent) of compressed row grp[i] of
 * sequence seq[i] (the projection stays with the caller).  For each row:
 *   k = bf16( weight * x / sqrt(mean(x^2) + eps) )        (RMSNorm.forward)
 *   k[D_I - dim ..] rotated at position grp[i] * r, rounded to bf16
 *   scale = amax|k| / 448 (1 for a zero row), codes = e4m3(k / scale)
 * written to k_I at element seq[i] * k_seq_stride + grp[i] * D_I (128 codes)
 * and to k_scale at seq[i] * (k_seq_stride / D_I) + grp[i].  The page
 * quantises these keys to fp4; here they take the e4m3 codes with one fp32
 * scale per position that sa_indexer_scores reads.  Norm and rotation are
 * evaluated in double and each bf16 result is one rounding of it; the
 * quotients are correctly rounded fp32.  D_I = 128, dim a multiple of 4 in
 * [0, 128]; k_seq_stride 0 (dense: N_rows * D_I) or a multiple of D_I of at
 * least N_rows * D_I; seq[i] outside [0, B) or grp[i] outside [0, N_rows) is
 * skipped and flagged (SA_ERR_DEVICE_DATA).  The workspace needs only its
 * 256-byte header. */
SA_API sa_status sa_index_key_publish(const void *kproj, int32_t n, int32_t D_I, const int32_t *seq,
                                      const int32_t *grp, int32_t r, const float *weight, float eps,
                                      const sa_rope_args *rope, uint8_t *k_I, float *k_scale, int32_t B,
                                      int32_t N_rows, int64_t k_seq_stride, void *ws, size_t ws_bytes,
                                      sa_stream_t stream);

/* Sparse MQA over the window and the selected compressed rows
 * ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Attention.forward and
 * sparse_attn): for token t and head h the keys are the window rows then the
 * compressed rows idx[t, k] != -1 (concatenated, not de-duplicated);
 * l_j = scale * Q[t,h] . K_j; out[t,h] = sum_j softmax(l)_j V_j, where the
 * softmax denominator also holds exp(sink[h]) when sink is given.
 * idx: [T, K] int32, each entry -1 or in [0, n_vis(t)); out: [T, H, D] bf16
 * (round to nearest even).  Only ia->B, T, N_c, r, q_seq and q_pos are read
 * from ia. */
SA_API sa_status sa_sparse_attn(const sa_index_args *ia, const sa_attn_args *aa, const int32_t *idx,
                         int32_t K, void *out, void *ws, size_t ws_bytes, sa_stream_t stream);

/* The whole step in one call, no host synchronisation: index scores into the
 * workspace, top-k, sparse MQA with the split-KV combine.  idx_out: [T, K]
 * int32 or NULL (then the indices stay in the workspace); out: [T, H, D]
 * bf16.  Serves decode (one token per sequence) and prefill chunks alike. */
SA_API sa_status sa_fused_decode(const sa_index_args *ia, const sa_attn_args *aa, int32_t K,
                          int32_t *idx_out, void *out, void *ws, size_t ws_bytes,
                          sa_stream_t stream);

/* sa_fused_decode with timing marks: the same launches on the same stream,
 * with the caller's CUDA events (cudaEvent_t handles) recorded on `stream`
 * before the index-score kernel, before the top-k kernel, before the
 * attention kernel(s) and after the last kernel: stage_events[0..3].  For
 * measuring each stage's device time inside a timed loop. */
SA_API sa_status sa_fused_decode_staged(const sa_index_args *ia, const sa_attn_args *aa, int32_t K,
                                        int32_t *idx_out, void *out, void *ws, size_t ws_bytes,
                                        sa_stream_t stream, void *const *stage_events);

/* Number of kernel launches one sa_fused_decode call makes for these shapes
 * (0 when the arguments are invalid). */
SA_API int32_t sa_fused_decode_launch_count(const sa_index_args *ia, const sa_attn_args *aa,
                                            int32_t K);

/* Bytes of the fixed device scratch array behind sa_fused_decode_noalloc. */
#define SA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/* SA_NOALLOC_SCRATCH_BYTES as compiled into the library (for bindings that
 * cannot read this header). */
SA_API size_t sa_noalloc_scratch_bytes(void);

/* sa_fused_decode for callers that cannot allocate device memory.  (The model
 * pages have no counterpart: this is a deployment variant of the fused step.)
 *
 * Who needs it: code that has no device allocator at hand or must not
 * allocate on its execution path -- a plugin host that hands its kernels no
 * workspace, or a serving loop that fixes its memory budget at start-up and
 * treats any allocation while serving a request as a failure.  Such a caller
 * cannot obtain the workspace the other entry points ask for.
 *
 * Same inputs, outputs and results as sa_fused_decode (idx_out may be NULL;
 * out is [T, H, D] bf16), but the scratch lives in one library-owned device
 * array of SA_NOALLOC_SCRATCH_BYTES bytes: every GPU that loads the library
 * holds that array until the process exits.  Nothing is allocated or freed:
 * no cudaMalloc, cudaFree or allocating library routine is called.
 *
 * - Size limit: a problem whose scratch (sa_workspace_size for the same
 *   arguments) exceeds SA_NOALLOC_SCRATCH_BYTES is rejected with
 *   SA_ERR_UNSUPPORTED and enqueues nothing.
 * - Set-up: the first call in each CUDA context (a device's primary context,
 *   with that device current, in the usual case) looks up the array's device
 *   address once (cudaGetSymbolAddress); make that first call before any
 *   stream capture.  After cudaDeviceReset, or in another context, the array
 *   may sit elsewhere; the address is looked up again there.
 * - Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents (no part of it needs to start at zero).  Calls whose work
 *   overlaps on the GPU -- on different streams, or from different host
 *   threads -- race on it and give undefined results; serialise them.
 * - device_status: optional 4-byte device word that the kernels OR their
 *   out-of-range-data flags into (see sa_check_device_status for their
 *   meaning); NULL to skip reporting.  The caller zeroes and reads it. */
SA_API sa_status sa_fused_decode_noalloc(const sa_index_args *ia, const sa_attn_args *aa,
                                         int32_t K, int32_t *idx_out, void *out,
                                         uint32_t *device_status, sa_stream_t stream);

/* Synchronises `stream`, then reads and clears the workspace's sticky device
 * status: SA_OK, SA_ERR_DEVICE_DATA (out-of-range device data was skipped)
 * or SA_ERR_TIMEOUT. */
SA_API sa_status sa_check_device_status(void *ws, sa_stream_t stream);

/* Bound on each pipeline wait of the tensor-core attention kernels (heads of
 * dim 128 and of dim 512, as sa_sparse_attn, sa_fused_decode and
 * sa_fused_decode_noalloc launch them), in SM clock cycles; 0 restores the
 * default of 2e9 cycles (about a second).  A wait between the kernel's own
 * stages (copies, products, softmax, the hand-off between the two CTAs of a
 * split token) that runs out makes the kernel set the timeout flag of the
 * status word (sa_check_device_status then returns SA_ERR_TIMEOUT), wait for
 * the copies and products it already started (those waits keep the default
 * bound), and return; its outputs are then undefined and the CUDA context
 * stays usable.  Meant for testing that path and for callers that prefer an
 * early error to a long stall.  Process-wide; applies to launches made after
 * it returns.  Returns SA_ERR_INVALID_ARG for a negative value. */
SA_API sa_status sa_set_wait_budget(int64_t cycles);

/* Text for a status code (static storage). */
SA_API const char *sa_status_string(sa_status s);

/* One-line reason for the calling thread's most recent non-OK return. */
SA_API const char *sa_last_error_detail(void);

#ifdef __cplusplus
}
#endif
#endif /* SA_H */
