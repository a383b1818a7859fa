// Compressor of the V4.1 indexer and attention caches ("DeepSeek-V4.1-Flash-
// NVFP4 inference/model.py", Compressor.forward from position 0, and
// RMSNorm.forward): every group of r consecutive tokens becomes one row.  For
// each channel d the group's kv values are weighted by the softmax, over the r
// tokens, of their gate scores and summed (fp32, as the page promotes the
// pooling to fp32); the pooled row is cast to bf16 (the activation dtype) and
// RMS-normalised in fp32: c * rsqrt(mean(c^2) + eps), times the norm weight,
// cast to bf16.
//
// One CTA per (sequence, group), one thread per channel: the r loads of a
// thread are D apart, so each of the r token rows is read coalesced; the mean
// of squares is a block reduction.  Decode steps use a state of r slots per
// sequence (kv_state, score_state: [B, r, D] fp32), pooled every r steps.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

__global__ void __launch_bounds__(1024)
compress_prefill_kernel(const float *__restrict__ kv, const float *__restrict__ score, int S, int D, int r, int G,
                        const float *__restrict__ weight, float eps, __nv_bfloat16 *__restrict__ out) {
  __shared__ float warp_sq[32];
  __shared__ float total_sq;
  const int g = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int lane = d & 31, warp = d >> 5;
  const int64_t base = (static_cast<int64_t>(b) * S + static_cast<int64_t>(g) * r) * D + d;
  float m = -INFINITY;
  for (int j = 0; j < r; ++j) m = fmaxf(m, score[base + static_cast<int64_t>(j) * D]);
  float z = 0.f, acc = 0.f;
  for (int j = 0; j < r; ++j) {
    const float e = expf(score[base + static_cast<int64_t>(j) * D] - m);
    z += e;
    acc = fmaf(e, kv[base + static_cast<int64_t>(j) * D], acc);
  }
  const float c = __bfloat162float(__float2bfloat16_rn(acc / z));  // the cast before the norm
  float sq = c * c;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (lane == 0) warp_sq[warp] = sq;
  __syncthreads();
  if (warp == 0) {
    float v = lane < (D >> 5) ? warp_sq[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) total_sq = v;
  }
  __syncthreads();
  const float inv = rsqrtf(total_sq / static_cast<float>(D) + eps);
  out[(static_cast<int64_t>(b) * G + g) * D + d] = __float2bfloat16_rn(weight[d] * (c * inv));
}

// The trailing S % r tokens of each sequence go to state slots 0 .. S % r - 1
// (Compressor.forward at start_pos 0 splits them off into kv_state and
// score_state), where decode steps complete the group.
__global__ void compress_state_kernel(const float *__restrict__ kv, const float *__restrict__ score, int S, int D,
                                      int r, int rem, float *__restrict__ kv_state, float *__restrict__ score_state) {
  const int b = blockIdx.y;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < rem * D; i += gridDim.x * blockDim.x) {
    const int64_t src = (static_cast<int64_t>(b) * S + (S - rem)) * D + i;
    const int64_t dst = static_cast<int64_t>(b) * r * D + i;
    kv_state[dst] = kv[src];
    score_state[dst] = score[src];
  }
}

// One decode step per sequence (Compressor.forward with start_pos > 0): the
// token at position pos[b] fills state slot pos[b] % r; when the group has
// just completed ((pos[b] + 1) % r == 0) the r slots are pooled like a prefill
// group and row b of `out` is written.  One CTA per sequence, one thread per
// channel: the slot a thread writes is the one it reads back, so no barrier
// separates them.
__global__ void __launch_bounds__(1024)
compress_decode_kernel(const float *__restrict__ kv, const float *__restrict__ score, const int32_t *__restrict__ pos,
                       int D, int r, float *__restrict__ kv_state, float *__restrict__ score_state,
                       const float *__restrict__ weight, float eps, __nv_bfloat16 *__restrict__ out,
                       uint32_t *status) {
  __shared__ float warp_sq[32];
  __shared__ float total_sq;
  const int b = blockIdx.x, d = threadIdx.x;
  const int lane = d & 31, warp = d >> 5;
  const int p = pos[b];
  if (p < 0) {
    if (d == 0) raise_flag(status, kFlagBadPos);
    return;
  }
  const int64_t st = static_cast<int64_t>(b) * r * D + d;
  kv_state[st + static_cast<int64_t>(p % r) * D] = kv[static_cast<int64_t>(b) * D + d];
  score_state[st + static_cast<int64_t>(p % r) * D] = score[static_cast<int64_t>(b) * D + d];
  if ((p + 1) % r != 0) return;  // the whole CTA leaves together (p is per sequence)
  float m = -INFINITY;
  for (int j = 0; j < r; ++j) m = fmaxf(m, score_state[st + static_cast<int64_t>(j) * D]);
  float z = 0.f, acc = 0.f;
  for (int j = 0; j < r; ++j) {
    const float e = expf(score_state[st + static_cast<int64_t>(j) * D] - m);
    z += e;
    acc = fmaf(e, kv_state[st + static_cast<int64_t>(j) * D], acc);
  }
  const float c = __bfloat162float(__float2bfloat16_rn(acc / z));  // the cast before the norm
  float sq = c * c;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (lane == 0) warp_sq[warp] = sq;
  __syncthreads();
  if (warp == 0) {
    float v = lane < (D >> 5) ? warp_sq[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) total_sq = v;
  }
  __syncthreads();
  const float inv = rsqrtf(total_sq / static_cast<float>(D) + eps);
  out[static_cast<int64_t>(b) * D + d] = __float2bfloat16_rn(weight[d] * (c * inv));
}

}  // namespace

cudaError_t launch_compress_prefill(const float *kv, const float *score, int B, int S, int D, int r,
                                    const float *weight, float eps, void *out, float *kv_state, float *score_state,
                                    cudaStream_t stream) {
  const int G = S / r;
  if (B == 0) return cudaSuccess;
  if (G > 0) {
    cudaError_t e = launch_ex(false, compress_prefill_kernel, dim3(G, B), dim3(D), 0, stream, 1, kv, score, S, D, r,
                              G, weight, eps, static_cast<__nv_bfloat16 *>(out));
    if (e != cudaSuccess) return e;
  }
  const int rem = S % r;
  if (kv_state && score_state && rem > 0)
    return launch_ex(false, compress_state_kernel, dim3((rem * D + 255) / 256, B), dim3(256), 0, stream, 1, kv,
                     score, S, D, r, rem, kv_state, score_state);
  return cudaSuccess;
}

cudaError_t launch_compress_decode(const float *kv, const float *score, const int32_t *pos, int B, int D, int r,
                                   float *kv_state, float *score_state, const float *weight, float eps, void *out,
                                   uint32_t *status, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  return launch_ex(false, compress_decode_kernel, dim3(B), dim3(D), 0, stream, 1, kv, score, pos, D, r, kv_state,
                   score_state, weight, eps, static_cast<__nv_bfloat16 *>(out), status);
}

}  // namespace sa
