// The C ABI declared in include/sa.h: argument checks on the host, workspace
// carve-up, and the launch sequence of each entry point.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace {

thread_local std::string g_detail;

sa_status fail(sa_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
sa_status fail(sa_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return s;
}

sa_status cuda_fail(cudaError_t e, const char *what) {
  return fail(SA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t round_up(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

sa_status check_k_stride(const sa_index_args *ia) {
  if (ia->k_seq_stride != 0 &&
      (ia->k_seq_stride % ia->D_I != 0 || ia->k_seq_stride < static_cast<int64_t>(ia->N_c) * ia->D_I))
    return fail(SA_ERR_INVALID_ARG, "k_seq_stride %lld: need 0 or a multiple of D_I = %d of at least N_c * D_I",
                static_cast<long long>(ia->k_seq_stride), ia->D_I);
  if (static_cast<int64_t>(ia->B - 1) * sa::k_rows_per_seq(*ia) + ia->N_c >= (int64_t{1} << 31) - 256)
    return fail(SA_ERR_UNSUPPORTED, "index key cache rows must fit in 31 bits");
  return SA_OK;
}

sa_status check_index(const sa_index_args *ia, bool need_index_inputs) {
  if (!ia) return fail(SA_ERR_INVALID_ARG, "index args pointer is NULL");
  if (ia->B < 1 || ia->T < 0 || ia->N_c < 1 || ia->r < 1)
    return fail(SA_ERR_INVALID_ARG, "need B >= 1, T >= 0, N_c >= 1, r >= 1 (got B=%d T=%d N_c=%d r=%d)",
                ia->B, ia->T, ia->N_c, ia->r);
  if (ia->T > 0 && (!ia->q_seq || !ia->q_pos))
    return fail(SA_ERR_INVALID_ARG, "q_seq and q_pos must be device pointers");
  if (!aligned4(ia->q_seq) || !aligned4(ia->q_pos))
    return fail(SA_ERR_INVALID_ARG, "q_seq / q_pos must be 4-byte aligned");
  if (!need_index_inputs) return SA_OK;
  if (ia->q_dtype != SA_BF16 && ia->q_dtype != SA_FP8_E4M3)
    return fail(SA_ERR_INVALID_ARG, "q_dtype %d is not a sa_dtype", ia->q_dtype);
  if (ia->k_dtype != SA_BF16 && ia->k_dtype != SA_FP8_E4M3)
    return fail(SA_ERR_INVALID_ARG, "k_dtype %d is not a sa_dtype", ia->k_dtype);
  if (!sa::index_shape_supported(ia->H_I, ia->D_I))
    return fail(SA_ERR_UNSUPPORTED, "index heads %d x dim %d: need 1..128 heads of dim 64 or 128",
                ia->H_I, ia->D_I);
  if (ia->T > 0 && (!ia->q_I || !ia->w || !ia->k_I))
    return fail(SA_ERR_INVALID_ARG, "q_I, w and k_I must be device pointers");
  if (!aligned16(ia->q_I) || !aligned16(ia->k_I))
    return fail(SA_ERR_INVALID_ARG, "q_I and k_I must be 16-byte aligned");
  if (!aligned4(ia->w) || !aligned4(ia->q_scale) || !aligned4(ia->k_scale))
    return fail(SA_ERR_INVALID_ARG, "w, q_scale and k_scale must be 4-byte aligned");
  return check_k_stride(ia);
}

sa_status check_ld(int64_t ld, const sa_index_args *ia) {
  if (ld < ia->N_c)
    return fail(SA_ERR_INVALID_ARG, "score row stride ld = %lld is below N_c = %d", static_cast<long long>(ld),
                ia->N_c);
  return SA_OK;
}

sa_status check_attn(const sa_attn_args *aa, int T) {
  if (!aa) return fail(SA_ERR_INVALID_ARG, "attention args pointer is NULL");
  if (!sa::attn_shape_supported(aa->H, aa->D))
    return fail(SA_ERR_UNSUPPORTED,
                "attention %d heads x dim %d: need dim 128 with 16/32/64/128 heads or dim 512 with 16/32/64",
                aa->H, aa->D);
  if (aa->W < 1 || aa->R < aa->W)
    return fail(SA_ERR_INVALID_ARG, "need W >= 1 and R >= W (got W=%d R=%d)", aa->W, aa->R);
  if (!std::isfinite(aa->scale)) return fail(SA_ERR_INVALID_ARG, "softmax scale is not finite");
  if (T > 0 && (!aa->Q || !aa->Kw || !aa->Vw || !aa->Kc || !aa->Vc))
    return fail(SA_ERR_INVALID_ARG, "Q, Kw, Vw, Kc, Vc must be device pointers");
  if (!aligned16(aa->Q) || !aligned16(aa->Kw) || !aligned16(aa->Vw) || !aligned16(aa->Kc) ||
      !aligned16(aa->Vc))
    return fail(SA_ERR_INVALID_ARG, "Q, Kw, Vw, Kc, Vc must be 16-byte aligned");
  if (!aligned4(aa->sink)) return fail(SA_ERR_INVALID_ARG, "sink must be 4-byte aligned");
  if (aa->w_seq_stride != 0 &&
      (aa->w_seq_stride % aa->D != 0 || aa->w_seq_stride < static_cast<int64_t>(aa->R) * aa->D))
    return fail(SA_ERR_INVALID_ARG, "w_seq_stride %lld: need 0 or a multiple of D = %d of at least R * D",
                static_cast<long long>(aa->w_seq_stride), aa->D);
  return SA_OK;
}

sa_status check_c_stride(const sa_attn_args *aa, const sa_index_args *ia) {
  if (aa->c_seq_stride != 0 &&
      (aa->c_seq_stride % aa->D != 0 || aa->c_seq_stride < static_cast<int64_t>(ia->N_c) * aa->D))
    return fail(SA_ERR_INVALID_ARG, "c_seq_stride %lld: need 0 or a multiple of D = %d of at least N_c * D",
                static_cast<long long>(aa->c_seq_stride), aa->D);
  // row indices of the caches are 32-bit
  const int64_t last = static_cast<int64_t>(ia->B - 1) *
                       std::max(sa::w_rows_per_seq(*aa), sa::c_rows_per_seq(*ia, *aa)) +
                       std::max<int64_t>(aa->R, ia->N_c);
  if (last >= (int64_t{1} << 31) - 256)
    return fail(SA_ERR_UNSUPPORTED, "caches of %lld rows: row indices must fit in 31 bits", static_cast<long long>(last));
  return SA_OK;
}

sa_status check_ws(void *ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(SA_ERR_WORKSPACE, "workspace pointer is NULL");
  if (!aligned16(ws)) return fail(SA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (ws_bytes < need)
    return fail(SA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return SA_OK;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

}  // namespace

namespace sa {

WsLayout ws_layout(const sa_index_args &ia, const sa_attn_args *aa, int K) {
  WsLayout L{};
  size_t off = 0;
  L.status = off;
  off += 256;
  L.scores = off;
  off += round_up(sizeof(float) * static_cast<size_t>(ia.T) * ia.N_c);
  L.idx = off;
  off += round_up(sizeof(int32_t) * static_cast<size_t>(ia.T) * (K > 0 ? K : 0));
  L.score_scratch = off;
  off += round_up(idx_score_scratch(ia));
  L.attn_scratch = L.part_m = L.part_l = L.part_o = off;
  if (aa && attn_umma_supported(*aa)) {
    off += round_up(attn_umma_scratch(ia, aa ? *aa : sa_attn_args{}, K));
  } else if (aa && attn_umma512_supported(*aa)) {
    // the head-dim-512 tensor-core attention keeps nothing in global memory
  } else if (aa) {
    const SplitPlan plan = plan_splits(ia.T, aa->W, K);
    const size_t th = static_cast<size_t>(ia.T) * aa->H * plan.splits;
    L.part_m = off;
    off += round_up(sizeof(float) * th);
    L.part_l = off;
    off += round_up(sizeof(float) * th);
    L.part_o = off;
    off += round_up(sizeof(float) * th * aa->D);
  }
  L.total = off;
  return L;
}

}  // namespace sa

namespace sa {

std::atomic<long long> g_wait_budget{0};
long long attn_wait_budget() { return g_wait_budget.load(); }

sa_status set_error(sa_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return s;
}

sa_status fused_with_scratch(const sa_index_args *ia, const sa_attn_args *aa, int K,
                             int32_t *idx_out, void *out, void *scratch, size_t scratch_bytes,
                             uint32_t *status, cudaStream_t st) {
  if (sa_status s = check_index(ia, true)) return s;
  if (sa_status s = check_attn(aa, ia->T)) return s;
  if (sa_status s = check_c_stride(aa, ia)) return s;
  if (K < 0) return fail(SA_ERR_INVALID_ARG, "K must be >= 0 (got %d)", K);
  if (ia->T > 0 && !out) return fail(SA_ERR_INVALID_ARG, "out must be a device pointer");
  if (!aligned4(idx_out) || !aligned16(out))
    return fail(SA_ERR_INVALID_ARG, "idx_out must be 4-byte and out 16-byte aligned");
  const WsLayout L = ws_layout(*ia, aa, K);
  if (sa_status s = check_ws(scratch, scratch_bytes, L.total)) return s;
  float *scores = at<float>(scratch, L.scores);
  int32_t *idx = idx_out ? idx_out : at<int32_t>(scratch, L.idx);
  cudaError_t e =
      launch_idx_score(*ia, scores, ia->N_c, false, at<void>(scratch, L.score_scratch), status, st);
  if (e != cudaSuccess) return cuda_fail(e, "index score launch");
  e = launch_topk(scores, ia->N_c, *ia, K, idx, status, st, nullptr, 0, 1, true);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  const SplitPlan plan = plan_splits(ia->T, aa->W, K);
  // the chain began with an ordinary launch made after every input was written
  e = launch_sparse_mqa(*ia, *aa, idx, K, out, at<float>(scratch, L.part_m),
                        at<float>(scratch, L.part_l), at<float>(scratch, L.part_o),
                        at<void>(scratch, L.attn_scratch), plan, true, status, st);
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "sparse attention launch");
}

}  // namespace sa

extern "C" {

size_t sa_workspace_size(const sa_index_args *ia, const sa_attn_args *aa, int32_t K) {
  if (check_index(ia, false) != SA_OK || K < 0) return 0;
  if (sa::index_shape_supported(ia->H_I, ia->D_I) && check_k_stride(ia) != SA_OK) return 0;
  if (aa && (check_attn(aa, 0) != SA_OK || check_c_stride(aa, ia) != SA_OK)) return 0;
  return sa::ws_layout(*ia, aa, K).total;
}

sa_status sa_workspace_init(void *ws, size_t ws_bytes, sa_stream_t stream) {
  if (sa_status s = check_ws(ws, ws_bytes, 256)) return s;
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "cudaMemsetAsync");
}

sa_status sa_indexer_scores(const sa_index_args *ia, float *scores, int64_t ld, void *ws, size_t ws_bytes,
                            sa_stream_t stream) {
  if (sa_status s = check_index(ia, true)) return s;
  if (sa_status s = check_ld(ld, ia)) return s;
  if (ia->T > 0 && !scores) return fail(SA_ERR_INVALID_ARG, "scores must be a device pointer");
  if (!aligned4(scores)) return fail(SA_ERR_INVALID_ARG, "scores must be 4-byte aligned");
  const sa::WsLayout L = sa::ws_layout(*ia, nullptr, 0);
  if (sa_status s = check_ws(ws, ws_bytes, L.total)) return s;
  cudaError_t e = sa::launch_idx_score(*ia, scores, ld, true, at<void>(ws, L.score_scratch),
                                       at<uint32_t>(ws, 0), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "index score launch");
}

sa_status sa_topk(const float *scores, int64_t ld, const sa_index_args *ia, int32_t K, int32_t *idx, void *ws,
                  size_t ws_bytes, sa_stream_t stream) {
  if (sa_status s = check_index(ia, false)) return s;
  if (sa_status s = check_ld(ld, ia)) return s;
  if (K < 0) return fail(SA_ERR_INVALID_ARG, "K must be >= 0 (got %d)", K);
  if (ia->T > 0 && K > 0 && (!scores || !idx))
    return fail(SA_ERR_INVALID_ARG, "scores and idx must be device pointers");
  if (!aligned4(scores) || !aligned4(idx))
    return fail(SA_ERR_INVALID_ARG, "scores and idx must be 4-byte aligned");
  if (sa_status s = check_ws(ws, ws_bytes, 256)) return s;
  cudaError_t e = sa::launch_topk(scores, ld, *ia, K, idx, at<uint32_t>(ws, 0),
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "top-k launch");
}

static sa_status check_compressor(int32_t B, int32_t D, int32_t r, float eps) {
  if (B < 0 || B > 65535) return fail(SA_ERR_INVALID_ARG, "need 0 <= B <= 65535 (got %d)", B);
  if (r < 2) return fail(SA_ERR_INVALID_ARG, "compression ratio must be >= 2 (got %d)", r);
  if (D < 32 || D > 1024 || D % 32) return fail(SA_ERR_UNSUPPORTED, "head dim %d: need a multiple of 32 in [32, 1024]", D);
  if (!std::isfinite(eps) || eps < 0.f) return fail(SA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  return SA_OK;
}

sa_status sa_compress_prefill(const float *kv, const float *score, int32_t B, int32_t S, int32_t D, int32_t r,
                              const float *weight, float eps, void *out, float *kv_state, float *score_state,
                              sa_stream_t stream) {
  if (sa_status s = check_compressor(B, D, r, eps)) return s;
  if (S < 0) return fail(SA_ERR_INVALID_ARG, "need S >= 0 (got %d)", S);
  if (B > 0 && S >= r && (!kv || !score || !weight || !out))
    return fail(SA_ERR_INVALID_ARG, "kv, score, weight and out must be device pointers");
  if ((kv_state == nullptr) != (score_state == nullptr))
    return fail(SA_ERR_INVALID_ARG, "kv_state and score_state go together");
  if (B > 0 && S % r && kv_state && (!kv || !score))
    return fail(SA_ERR_INVALID_ARG, "kv and score must be device pointers");
  if (!aligned4(kv) || !aligned4(score) || !aligned4(weight) || !aligned4(out) || !aligned4(kv_state) ||
      !aligned4(score_state))
    return fail(SA_ERR_INVALID_ARG, "kv, score, weight, out and the states must be 4-byte aligned");
  cudaError_t e = sa::launch_compress_prefill(kv, score, B, S, D, r, weight, eps, out, kv_state, score_state,
                                              reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "compressor launch");
}

sa_status sa_compress_decode(const float *kv, const float *score, const int32_t *pos, int32_t B, int32_t D,
                             int32_t r, float *kv_state, float *score_state, const float *weight, float eps,
                             void *out, void *ws, size_t ws_bytes, sa_stream_t stream) {
  if (sa_status s = check_compressor(B, D, r, eps)) return s;
  if (B > 0 && (!kv || !score || !pos || !kv_state || !score_state || !weight || !out))
    return fail(SA_ERR_INVALID_ARG, "kv, score, pos, the states, weight and out must be device pointers");
  if (!aligned4(kv) || !aligned4(score) || !aligned4(pos) || !aligned4(kv_state) || !aligned4(score_state) ||
      !aligned4(weight) || !aligned4(out))
    return fail(SA_ERR_INVALID_ARG, "every pointer must be 4-byte aligned");
  if (sa_status s = check_ws(ws, ws_bytes, 256)) return s;
  cudaError_t e = sa::launch_compress_decode(kv, score, pos, B, D, r, kv_state, score_state, weight, eps, out,
                                             at<uint32_t>(ws, 0), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "compressor decode launch");
}

sa_status sa_index_key_publish(const void *kproj, int32_t n, int32_t D_I, const int32_t *seq, const int32_t *grp,
                               int32_t r, const float *weight, float eps, const sa_rope_args *rope, uint8_t *k_I,
                               float *k_scale, int32_t B, int32_t N_rows, int64_t k_seq_stride, void *ws,
                               size_t ws_bytes, sa_stream_t stream) {
  if (n < 0 || B < 1 || N_rows < 1 || r < 1)
    return fail(SA_ERR_INVALID_ARG, "need n >= 0, B >= 1, N_rows >= 1, r >= 1");
  if (D_I != 128) return fail(SA_ERR_UNSUPPORTED, "index head dim %d: the key producer takes 128", D_I);
  if (!rope) return fail(SA_ERR_INVALID_ARG, "rope args pointer is NULL");
  if (rope->dim < 0 || rope->dim > D_I || rope->dim % 4)
    return fail(SA_ERR_INVALID_ARG, "rope dim %d: need a multiple of 4 in [0, %d]", rope->dim, D_I);
  if (rope->dim > 0 && (!std::isfinite(rope->base) || rope->base <= 1.0 || !std::isfinite(rope->factor) ||
                        rope->factor <= 0.0 ||
                        (rope->original_seq_len > 0 && !(rope->beta_fast > 0.0 && rope->beta_slow > 0.0))))
    return fail(SA_ERR_INVALID_ARG, "rope base > 1, factor > 0 and, with YaRN, beta_fast and beta_slow > 0");
  if (!std::isfinite(eps) || eps < 0.f) return fail(SA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (k_seq_stride != 0 && (k_seq_stride % D_I || k_seq_stride < static_cast<int64_t>(N_rows) * D_I))
    return fail(SA_ERR_INVALID_ARG, "k_seq_stride %lld: need 0 or a multiple of D_I of at least N_rows * D_I",
                static_cast<long long>(k_seq_stride));
  if (n > 0 && (!kproj || !seq || !grp || !weight || !k_I || !k_scale))
    return fail(SA_ERR_INVALID_ARG, "kproj, seq, grp, weight, k_I and k_scale must be device pointers");
  if (!aligned16(kproj) || !aligned4(k_I) || !aligned4(seq) || !aligned4(grp) || !aligned4(weight) ||
      !aligned4(k_scale))
    return fail(SA_ERR_INVALID_ARG, "kproj must be 16-byte aligned; k_I and the other arrays 4-byte aligned");
  if (sa_status s = check_ws(ws, ws_bytes, 256)) return s;
  cudaError_t e = sa::launch_index_key_publish(kproj, n, seq, grp, r, weight, eps, *rope, k_I, k_scale, B, N_rows,
                                               k_seq_stride, at<uint32_t>(ws, 0),
                                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "index key launch");
}

sa_status sa_rotate_quant(const void *x, int32_t rows, int32_t dim, const int32_t *dst, int64_t dst_rows,
                          uint8_t *codes, float *scales, void *ws, size_t ws_bytes, sa_stream_t stream) {
  if (rows < 0) return fail(SA_ERR_INVALID_ARG, "rows must be >= 0 (got %d)", rows);
  if (dim != 128) return fail(SA_ERR_UNSUPPORTED, "row length %d: the producer takes rows of 128", dim);
  if (dst && dst_rows < 0) return fail(SA_ERR_INVALID_ARG, "dst_rows must be >= 0");
  if (rows > 0 && (!x || !codes || !scales))
    return fail(SA_ERR_INVALID_ARG, "x, codes and scales must be device pointers");
  if (!aligned16(x) || !aligned4(codes) || !aligned4(scales) || !aligned4(dst))
    return fail(SA_ERR_INVALID_ARG, "x must be 16-byte aligned; codes, scales and dst 4-byte aligned");
  if (sa_status s = check_ws(ws, ws_bytes, 256)) return s;
  cudaError_t e = sa::launch_rotate_quant(x, rows, dst, dst_rows, codes, scales, at<uint32_t>(ws, 0),
                                          reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "rotate-quant launch");
}

int32_t sa_candidate_words(int32_t N_c, int32_t block_size) {
  if (N_c < 1 || block_size < 1) return 0;
  return sa::candidate_words(N_c, block_size);
}

sa_status sa_candidate_blocks(const float *scores, int64_t ld, const sa_index_args *ia, int32_t block_size,
                              int32_t topk_blocks, uint32_t *cand, void *ws, size_t ws_bytes, sa_stream_t stream) {
  if (sa_status s = check_index(ia, false)) return s;
  if (sa_status s = check_ld(ld, ia)) return s;
  if (block_size < 1 || topk_blocks < 0)
    return fail(SA_ERR_INVALID_ARG, "need block_size >= 1 and topk_blocks >= 0 (got %d, %d)", block_size,
                topk_blocks);
  if (ia->N_c > (1 << 30)) return fail(SA_ERR_UNSUPPORTED, "N_c %d above 2^30", ia->N_c);
  const int64_t nb = (static_cast<int64_t>(ia->N_c) + block_size - 1) / block_size;
  if (nb > sa::kMaxCandidateBlocks)
    return fail(SA_ERR_UNSUPPORTED, "%lld candidate blocks per row (at most %d)", static_cast<long long>(nb),
                sa::kMaxCandidateBlocks);
  if (ia->T > 0 && (!scores || !cand))
    return fail(SA_ERR_INVALID_ARG, "scores and cand must be device pointers");
  if (!aligned4(scores) || !aligned4(cand))
    return fail(SA_ERR_INVALID_ARG, "scores and cand must be 4-byte aligned");
  if (sa_status s = check_ws(ws, ws_bytes, 256)) return s;
  cudaError_t e = sa::launch_candidate_blocks(scores, ld, *ia, block_size, topk_blocks, cand,
                                              at<uint32_t>(ws, 0), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "candidate block launch");
}

sa_status sa_topk_candidates(const float *scores, int64_t ld, const sa_index_args *ia, int32_t K,
                             const uint32_t *cand, int32_t block_size, int32_t *idx, void *ws, size_t ws_bytes,
                             sa_stream_t stream) {
  if (sa_status s = check_index(ia, false)) return s;
  if (sa_status s = check_ld(ld, ia)) return s;
  if (K < 0) return fail(SA_ERR_INVALID_ARG, "K must be >= 0 (got %d)", K);
  if (block_size < 1) return fail(SA_ERR_INVALID_ARG, "block_size must be >= 1 (got %d)", block_size);
  if (ia->N_c > (1 << 30)) return fail(SA_ERR_UNSUPPORTED, "N_c %d above 2^30", ia->N_c);
  if (ia->T > 0 && K > 0 && (!scores || !idx || !cand))
    return fail(SA_ERR_INVALID_ARG, "scores, cand and idx must be device pointers");
  if (!aligned4(scores) || !aligned4(idx) || !aligned4(cand))
    return fail(SA_ERR_INVALID_ARG, "scores, cand and idx must be 4-byte aligned");
  if (sa_status s = check_ws(ws, ws_bytes, 256)) return s;
  cudaError_t e = sa::launch_topk(scores, ld, *ia, K, idx, at<uint32_t>(ws, 0),
                                  reinterpret_cast<cudaStream_t>(stream), cand,
                                  sa::candidate_words(ia->N_c, block_size), block_size);
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "top-k launch");
}

sa_status sa_sparse_attn(const sa_index_args *ia, const sa_attn_args *aa, const int32_t *idx,
                         int32_t K, void *out, void *ws, size_t ws_bytes, sa_stream_t stream) {
  if (sa_status s = check_index(ia, false)) return s;
  if (sa_status s = check_attn(aa, ia->T)) return s;
  if (sa_status s = check_c_stride(aa, ia)) return s;
  if (K < 0) return fail(SA_ERR_INVALID_ARG, "K must be >= 0 (got %d)", K);
  if (ia->T > 0 && (!out || (K > 0 && !idx)))
    return fail(SA_ERR_INVALID_ARG, "out and idx must be device pointers");
  if (!aligned4(idx) || !aligned16(out))
    return fail(SA_ERR_INVALID_ARG, "idx must be 4-byte and out 16-byte aligned");
  const sa::WsLayout L = sa::ws_layout(*ia, aa, K);
  if (sa_status s = check_ws(ws, ws_bytes, L.total)) return s;
  const sa::SplitPlan plan = sa::plan_splits(ia->T, aa->W, K);
  cudaError_t e = sa::launch_sparse_mqa(*ia, *aa, idx, K, out, at<float>(ws, L.part_m),
                                        at<float>(ws, L.part_l), at<float>(ws, L.part_o), at<void>(ws, L.attn_scratch), plan,
                                        false, at<uint32_t>(ws, 0), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "sparse attention launch");
}

static sa_status fused_impl(const sa_index_args *ia, const sa_attn_args *aa, int32_t K,
                            int32_t *idx_out, void *out, void *ws, size_t ws_bytes,
                            sa_stream_t stream, void *const *ev) {
  if (sa_status s = check_index(ia, true)) return s;
  if (sa_status s = check_attn(aa, ia->T)) return s;
  if (sa_status s = check_c_stride(aa, ia)) return s;
  if (K < 0) return fail(SA_ERR_INVALID_ARG, "K must be >= 0 (got %d)", K);
  if (ia->T > 0 && !out) return fail(SA_ERR_INVALID_ARG, "out must be a device pointer");
  if (!aligned4(idx_out) || !aligned16(out))
    return fail(SA_ERR_INVALID_ARG, "idx_out must be 4-byte and out 16-byte aligned");
  const sa::WsLayout L = sa::ws_layout(*ia, aa, K);
  if (sa_status s = check_ws(ws, ws_bytes, L.total)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto mark = [&](int i) -> cudaError_t {
    // external record nodes: the events are really recorded when the call is
    // captured into a CUDA graph and replayed
    return ev ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev[i]), st, cudaEventRecordExternal)
              : cudaSuccess;
  };
  uint32_t *status = at<uint32_t>(ws, 0);
  float *scores = at<float>(ws, L.scores);
  int32_t *idx = idx_out ? idx_out : at<int32_t>(ws, L.idx);
  cudaError_t e = mark(0);
  if (e == cudaSuccess)
    e = sa::launch_idx_score(*ia, scores, ia->N_c, false, at<void>(ws, L.score_scratch), status, st);
  if (e != cudaSuccess) return cuda_fail(e, "index score launch");
  e = mark(1);
  if (e == cudaSuccess) e = sa::launch_topk(scores, ia->N_c, *ia, K, idx, status, st, nullptr, 0, 1, !ev);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  const sa::SplitPlan plan = sa::plan_splits(ia->T, aa->W, K);
  e = mark(2);
  if (e == cudaSuccess)
    e = sa::launch_sparse_mqa(*ia, *aa, idx, K, out, at<float>(ws, L.part_m), at<float>(ws, L.part_l),
                              at<float>(ws, L.part_o), at<void>(ws, L.attn_scratch), plan, true, status, st);
  if (e == cudaSuccess) e = mark(3);
  return e == cudaSuccess ? SA_OK : cuda_fail(e, "sparse attention launch");
}

sa_status sa_fused_decode(const sa_index_args *ia, const sa_attn_args *aa, int32_t K,
                          int32_t *idx_out, void *out, void *ws, size_t ws_bytes,
                          sa_stream_t stream) {
  return fused_impl(ia, aa, K, idx_out, out, ws, ws_bytes, stream, nullptr);
}

sa_status sa_fused_decode_staged(const sa_index_args *ia, const sa_attn_args *aa, int32_t K,
                                 int32_t *idx_out, void *out, void *ws, size_t ws_bytes,
                                 sa_stream_t stream, void *const *stage_events) {
  if (!stage_events) return fail(SA_ERR_INVALID_ARG, "stage_events is NULL");
  for (int i = 0; i < 4; ++i)
    if (!stage_events[i]) return fail(SA_ERR_INVALID_ARG, "stage event %d is NULL", i);
  return fused_impl(ia, aa, K, idx_out, out, ws, ws_bytes, stream, stage_events);
}

int32_t sa_fused_decode_launch_count(const sa_index_args *ia, const sa_attn_args *aa, int32_t K) {
  if (check_index(ia, true) != SA_OK || check_attn(aa, 0) != SA_OK || check_c_stride(aa, ia) != SA_OK || K < 0)
    return 0;
  if (ia->T == 0) return 0;
  const sa::SplitPlan plan = sa::plan_splits(ia->T, aa->W, K);
  return sa::fused_launch_count(*ia, *aa, K, plan);
}

sa_status sa_set_wait_budget(int64_t cycles) {
  if (cycles < 0) return fail(SA_ERR_INVALID_ARG, "wait budget must be >= 0 (got %lld)", static_cast<long long>(cycles));
  sa::g_wait_budget.store(static_cast<long long>(cycles));
  return SA_OK;
}

sa_status sa_check_device_status(void *ws, sa_stream_t stream) {
  if (!ws) return fail(SA_ERR_WORKSPACE, "workspace pointer is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t flags = 0;
  e = cudaMemcpy(&flags, ws, sizeof(flags), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy (status word)");
  if (flags == 0) return SA_OK;
  e = cudaMemset(ws, 0, sizeof(flags));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset (status word)");
  if (flags & sa::kFlagTimeout) return fail(SA_ERR_TIMEOUT, "a bounded device wait gave up (flags 0x%x)", flags);
  return fail(SA_ERR_DEVICE_DATA, "device data out of range was skipped (flags 0x%x:%s%s%s)", flags,
              (flags & sa::kFlagBadSeq) ? " q_seq" : "", (flags & sa::kFlagBadPos) ? " q_pos" : "",
              (flags & sa::kFlagBadIndex) ? " idx" : "");
}

const char *sa_status_string(sa_status s) {
  switch (s) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument";
    case SA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case SA_ERR_WORKSPACE: return "workspace missing or too small";
    case SA_ERR_CUDA: return "CUDA error";
    case SA_ERR_TIMEOUT: return "bounded device wait timed out";
    case SA_ERR_DEVICE_DATA: return "out-of-range device data skipped";
  }
  return "unknown status";
}

const char *sa_last_error_detail(void) { return g_detail.c_str(); }

}  // extern "C"
