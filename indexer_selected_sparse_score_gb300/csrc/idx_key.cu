// Index keys of the V4.1 layer that owns them ("DeepSeek-V4.1-Flash-NVFP4
// inference/model.py", Indexer.forward: k = k_norm(wk(latent)), the rotary
// embedding of its last rope_head_dim values at the group's first position,
// quantisation, and the write into the index key cache at row
// start_pos // ratio; precompute_freqs_cis and apply_rotary_emb for the
// rotation).
//
// One warp per key row, lane l holding values 4l .. 4l + 3.  The norm and the
// rotation run in double, so that each of the two bf16 results (after the
// norm, after the rotation) is one rounding of a value whose error is far
// below a bf16 step; the block quantisation (scale = amax / 448, e4m3 codes of
// k / scale) takes correctly rounded fp32 quotients.  The rotation
// frequencies depend on the rotary parameters only and are tabled per launch
// on the host (as precompute_freqs_cis tables them once); each pair's angle
// and its sine and cosine are taken in double in the kernel.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int kKeyDim = 128;
constexpr int kKeyWarps = 4;
constexpr double kPi = 3.14159265358979323846;

constexpr int kMaxPairs = kKeyDim / 2;

// Rotation frequencies of the launch, one per pair (precompute_freqs_cis's
// table, computed once per launch on the host: they depend on the rotary
// parameters only).
struct RopeFreqs {
  double f[kMaxPairs];
};

__global__ void __launch_bounds__(32 * kKeyWarps)
index_key_kernel(const uint16_t *__restrict__ kproj, int n, const int32_t *__restrict__ seq,
                 const int32_t *__restrict__ grp, int r, const float *__restrict__ weight, float eps, int rope_dim,
                 const __grid_constant__ RopeFreqs freqs, uint8_t *__restrict__ k_I, float *__restrict__ k_scale,
                 int B, int N_rows, int64_t kseq_rows, uint32_t *status) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kKeyWarps + (threadIdx.x >> 5);
  if (row >= n) return;
  const int b = seq[row], j = grp[row];
  if (b < 0 || b >= B || j < 0 || j >= N_rows) {
    if (lane == 0) raise_flag(status, b < 0 || b >= B ? kFlagBadSeq : kFlagBadPos);
    return;
  }
  const uint2 raw = *reinterpret_cast<const uint2 *>(kproj + static_cast<int64_t>(row) * kKeyDim + 4 * lane);
  double x[4] = {static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xFFFFu))),
                 static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16))),
                 static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xFFFFu))),
                 static_cast<double>(bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16)))};
  // RMSNorm: the squares of bf16 values and their sum are exact in double
  double ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const double inv = 1.0 / sqrt(ss / kKeyDim + static_cast<double>(eps));
  float k[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    k[e] = __bfloat162float(__double2bfloat16(static_cast<double>(weight[4 * lane + e]) * (x[e] * inv)));
  // rotation of the last rope.dim values: pairs (first + 2i, first + 2i + 1)
  const int first = kKeyDim - rope_dim;
  if (4 * lane >= first) {
    const double pos = static_cast<double>(j) * r;  // a latent stands for its group's first token
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int i = (4 * lane + e - first) / 2;
      double sn, cs;
      sincos(pos * freqs.f[i], &sn, &cs);
      const double re = k[e], im = k[e + 1];
      k[e] = __bfloat162float(__double2bfloat16(re * cs - im * sn));
      k[e + 1] = __bfloat162float(__double2bfloat16(re * sn + im * cs));
    }
  }
  // block quantisation of the row
  float amax = fmaxf(fmaxf(fabsf(k[0]), fabsf(k[1])), fmaxf(fabsf(k[2]), fabsf(k[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(k[e], s), __NV_SATFINITE, __NV_E4M3);
    packed |= static_cast<uint32_t>(c) << (8 * e);
  }
  const int64_t krow = static_cast<int64_t>(b) * kseq_rows + j;
  *reinterpret_cast<uint32_t *>(k_I + krow * kKeyDim + 4 * lane) = packed;
  if (lane == 0) k_scale[krow] = s;
}

}  // namespace

cudaError_t launch_index_key_publish(const void *kproj, int n, const int32_t *seq, const int32_t *grp, int r,
                                     const float *weight, float eps, const sa_rope_args &rope, uint8_t *k_I,
                                     float *k_scale, int B, int N_rows, int64_t k_seq_stride, uint32_t *status,
                                     cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int64_t kseq_rows = k_seq_stride ? k_seq_stride / kKeyDim : N_rows;
  // f_i = base^(-2i / dim); with original_seq_len > 0 (YaRN) the pairs below
  // the corrected dimension of beta_fast keep it, those above that of
  // beta_slow are divided by factor, and a linear ramp fades between (the
  // corrected dimension: the one whose wavelength completes `turns` rotations
  // over the training context)
  RopeFreqs fr{};
  const int pairs = rope.dim / 2;
  double low = 0.0, high = 0.0;
  if (rope.original_seq_len > 0) {
    auto corrected = [&](double turns) {
      return rope.dim * std::log(rope.original_seq_len / (turns * 2.0 * kPi)) / (2.0 * std::log(rope.base));
    };
    low = std::max(std::floor(corrected(rope.beta_fast)), 0.0);
    high = std::min(std::ceil(corrected(rope.beta_slow)), static_cast<double>(rope.dim - 1));
  }
  for (int i = 0; i < pairs; ++i) {
    double f = 1.0 / std::pow(rope.base, static_cast<double>(2 * i) / rope.dim);
    if (rope.original_seq_len > 0) {
      const double ramp = std::min(std::max((i - low) / std::max(high - low, 1e-3), 0.0), 1.0);
      f = f / rope.factor * ramp + f * (1.0 - ramp);
    }
    fr.f[i] = f;
  }
  return launch_ex(false, index_key_kernel, dim3((n + kKeyWarps - 1) / kKeyWarps), dim3(32 * kKeyWarps), 0, stream, 1,
                   static_cast<const uint16_t *>(kproj), n, seq, grp, r, weight, eps, rope.dim, fr, k_I, k_scale, B,
                   N_rows, kseq_rows, status);
}

}  // namespace sa
