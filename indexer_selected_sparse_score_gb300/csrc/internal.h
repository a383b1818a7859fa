// Host-side launchers behind the C ABI (one per kernel family).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sa.h"

namespace sa {

// Attention split-KV plan: each token's key list (window rows then its K
// index slots) is cut into `splits` chunks of `split_keys` keys.
struct SplitPlan {
  int splits;
  int split_keys;
};
SplitPlan plan_splits(int T, int W, int K);

// Workspace carve-up (byte offsets, 256-byte aligned).
struct WsLayout {
  size_t status, scores, idx, score_scratch, attn_scratch, part_m, part_l, part_o, total;
};

// Driver entry point cuTensorMapEncodeTiled (NULL if unavailable) and the
// current device's SM count.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
int sm_count();
// Sets a kernel's dynamic shared-memory limit once per device (flag array of
// 64 devices owned by the caller).
cudaError_t set_smem_once(const void *func, size_t bytes, bool *done_per_device);
WsLayout ws_layout(const sa_index_args &ia, const sa_attn_args *aa, int K);

// Index scores.  `scratch` (idx_score_scratch(ia) bytes, 256-byte aligned)
// holds the tensor-core kernel's packed queries and folded head weights.
cudaError_t launch_idx_score(const sa_index_args &ia, float *scores, int64_t ld,
                             bool write_masked, void *scratch, uint32_t *status,
                             cudaStream_t stream);
size_t idx_score_scratch(const sa_index_args &ia);

// Tensor-core (tcgen05) variant: fp8 keys of dim 128, 32/64/128 index heads.
bool idx_score_umma_supported(const sa_index_args &ia);
size_t idx_score_umma_scratch(const sa_index_args &ia);
cudaError_t launch_idx_score_umma(const sa_index_args &ia, float *scores, int64_t ld,
                                  bool write_masked, void *scratch, uint32_t *status,
                                  cudaStream_t stream);

// Per-query top-k.  With `cand` ([T, cand_words] block mask, blocks of
// block_size positions) the positions outside kept blocks count as -inf.
// `programmatic`: the previous kernel on the stream is one this library
// launched that writes no token array (the kernel reads those before it waits
// for the previous kernel), so the launch may overlap its end.
cudaError_t launch_topk(const float *scores, int64_t ld, const sa_index_args &ia, int K,
                        int32_t *idx, uint32_t *status, cudaStream_t stream,
                        const uint32_t *cand = nullptr, int cand_words = 0, int block_size = 1,
                        bool programmatic = false);

// Level one of the two-level top-k: per token, the block mask of the kept
// candidate blocks ([T, candidate_words(N_c, block_size)] uint32).
int candidate_words(int N_c, int block_size);
constexpr int kMaxCandidateBlocks = 32768;
// Index producer of the uncompressed indexer: Hadamard rotation and e4m3
// block quantisation of rows of 128 bf16 values, optionally scattered to
// rows dst[r] of the destination.
cudaError_t launch_rotate_quant(const void *x, int rows, const int32_t *dst, int64_t dst_rows, uint8_t *codes,
                                float *scales, uint32_t *status, cudaStream_t stream);
// V4.1 compressor from position 0: S / r pooled, normalised bf16 rows per sequence.
cudaError_t launch_compress_prefill(const float *kv, const float *score, int B, int S, int D, int r,
                                    const float *weight, float eps, void *out, float *kv_state, float *score_state,
                                    cudaStream_t stream);
cudaError_t launch_compress_decode(const float *kv, const float *score, const int32_t *pos, int B, int D, int r,
                                   float *kv_state, float *score_state, const float *weight, float eps, void *out,
                                   uint32_t *status, cudaStream_t stream);
// V4.1 index keys of a compressing layer: k_norm, rotary embedding of the last
// rope.dim values at position grp * r, e4m3 block quantisation, cache write.
cudaError_t launch_index_key_publish(const void *kproj, int n, const int32_t *seq, const int32_t *grp, int r,
                                     const float *weight, float eps, const sa_rope_args &rope, uint8_t *k_I,
                                     float *k_scale, int B, int N_rows, int64_t k_seq_stride, uint32_t *status,
                                     cudaStream_t stream);
cudaError_t launch_candidate_blocks(const float *scores, int64_t ld, const sa_index_args &ia, int block_size,
                                   int topk_blocks, uint32_t *cand, uint32_t *status, cudaStream_t stream);

// Attention + combine.  The tensor-core kernel (64 heads of dim 128) uses
// `attn_scratch` (attn_umma_scratch bytes); the CUDA-core kernel uses the
// split partials part_m/part_l/part_o laid out by `plan`.  `inputs_ready`:
// the chain of programmatic launches this one ends began with an ordinary
// launch made after every input but idx was written (each kernel of the chain
// starts only after every CTA of its predecessor has started), so the
// tensor-core kernels may read those inputs before waiting for the previous
// kernel.
cudaError_t launch_sparse_mqa(const sa_index_args &ia, const sa_attn_args &aa, const int32_t *idx,
                              int K, void *out, float *part_m, float *part_l, float *part_o,
                              void *attn_scratch, const SplitPlan &plan, bool inputs_ready, uint32_t *status,
                              cudaStream_t stream);
bool attn_umma_supported(const sa_attn_args &aa);
// Tensor-core (tcgen05) attention at the released V4.1 shape: 64 heads of dim
// 512 over one kv tensor (Kw == Vw, Kc == Vc); no scratch.
bool attn_umma512_supported(const sa_attn_args &aa);
// The wait bound set by sa_set_wait_budget (SM cycles; 0 = the default).
long long attn_wait_budget();

cudaError_t launch_sparse_mqa_umma512(const sa_index_args &ia, const sa_attn_args &aa, const int32_t *idx, int K,
                                      void *out, bool inputs_ready, uint32_t *status, cudaStream_t stream);
size_t attn_umma_scratch(const sa_index_args &ia, const sa_attn_args &aa, int K);
cudaError_t launch_sparse_mqa_umma(const sa_index_args &ia, const sa_attn_args &aa, const int32_t *idx, int K,
                                   void *out, void *scratch, bool inputs_ready, uint32_t *status, cudaStream_t stream);

// Kernel launches of one fused call (index score, top-k, attention, combine).
int fused_launch_count(const sa_index_args &ia, const sa_attn_args &aa, int K,
                       const SplitPlan &plan);

// Launches `kernel`; with `pdl` it may start while the previous kernel of
// `stream` runs (programmatic stream serialization) and must pdl_wait() before
// it reads what that kernel wrote.  `cluster` > 1 adds a cluster dimension.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      int cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Records a one-line error detail for sa_last_error_detail() and returns s.
sa_status set_error(sa_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));

// The fused launch sequence on a caller-chosen scratch region (laid out by
// ws_layout) with a caller-chosen status word (may be NULL).
sa_status fused_with_scratch(const sa_index_args *ia, const sa_attn_args *aa, int K,
                             int32_t *idx_out, void *out, void *scratch, size_t scratch_bytes,
                             uint32_t *status, cudaStream_t stream);

bool attn_shape_supported(int H, int D);

// Rows between consecutive sequences of each cache (the strides of the
// argument structs, 0 meaning dense).
inline int64_t k_rows_per_seq(const sa_index_args &ia) {
  return ia.k_seq_stride ? ia.k_seq_stride / ia.D_I : ia.N_c;
}
inline int64_t w_rows_per_seq(const sa_attn_args &aa) { return aa.w_seq_stride ? aa.w_seq_stride / aa.D : aa.R; }
inline int64_t c_rows_per_seq(const sa_index_args &ia, const sa_attn_args &aa) {
  return aa.c_seq_stride ? aa.c_seq_stride / aa.D : ia.N_c;
}
bool index_shape_supported(int H_I, int D_I);

}  // namespace sa
