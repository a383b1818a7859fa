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
// of squares is a block reduction.
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

}  // namespace

cudaError_t launch_compress_prefill(const float *kv, const float *score, int B, int S, int D, int r,
                                    const float *weight, float eps, void *out, cudaStream_t stream) {
  const int G = S / r;
  if (B == 0 || G == 0) return cudaSuccess;
  return launch_ex(false, compress_prefill_kernel, dim3(G, B), dim3(D), 0, stream, 1, kv, score, S, D, r, G, weight,
                   eps, static_cast<__nv_bfloat16 *>(out));
}

}  // namespace sa
