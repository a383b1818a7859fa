// Index producer of the uncompressed (r = 1) indexer ("DeepSeek-V3.2-Exp
// inference/model.py", Indexer.forward: rotate_activation, then act_quant of
// q and k, and the write of k into the index key cache).
//
// Each row of 128 bf16 values is multiplied by the Sylvester-Hadamard matrix
// and scaled by 128^-1/2: fp32 butterflies in the fixed stage order h = 1, 2,
// ..., 64, each taking the pair (i, i + h) from (a, b) to (a + b, a - b), then
// the product with the fp32 constant 128^-1/2 rounded to bf16.  The row is
// then quantised as one block: scale = amax / 448 and codes = e4m3(y / scale)
// (nearest, ties to even, saturating at 448), both divisions in fp32; an
// all-zero row gets scale 1.  Every rounding is an explicit _rn operation, so
// the codes are reproducible bit for bit.
//
// One warp per row: lane l holds elements 4l .. 4l+3, so stages 1 and 2 run in
// registers and stage h >= 4 pairs lane l with lane l ^ (h / 4).  A row may land
// at another row of the destination (dst[r]: e.g. row b * N_c + position of the
// k cache); a destination outside [0, dst_rows) is skipped and flagged.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int kProdDim = 128;
constexpr int kProdWarps = 8;

__global__ void __launch_bounds__(32 * kProdWarps)
rotate_quant_kernel(const uint16_t *__restrict__ x, int rows, float inv_sqrt_n, const int32_t *__restrict__ dst,
                    int64_t dst_rows, uint8_t *__restrict__ codes, float *__restrict__ scales, uint32_t *status) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kProdWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint2 raw = *reinterpret_cast<const uint2 *>(x + row * kProdDim + 4 * lane);
  float v[4] = {bf16_bits_to_float(static_cast<uint16_t>(raw.x & 0xFFFFu)),
                bf16_bits_to_float(static_cast<uint16_t>(raw.x >> 16)),
                bf16_bits_to_float(static_cast<uint16_t>(raw.y & 0xFFFFu)),
                bf16_bits_to_float(static_cast<uint16_t>(raw.y >> 16))};
  // stages h = 1 and 2 inside the lane
  {
    const float a = v[0], b = v[1], c = v[2], d = v[3];
    v[0] = __fadd_rn(a, b);
    v[1] = __fsub_rn(a, b);
    v[2] = __fadd_rn(c, d);
    v[3] = __fsub_rn(c, d);
  }
  {
    const float a = v[0], b = v[1], c = v[2], d = v[3];
    v[0] = __fadd_rn(a, c);
    v[2] = __fsub_rn(a, c);
    v[1] = __fadd_rn(b, d);
    v[3] = __fsub_rn(b, d);
  }
  // stages h = 4 .. 64 across lanes: the lower element of a pair keeps a + b,
  // the upper one a - b (a the lower element's value)
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float o = __shfl_xor_sync(0xffffffffu, v[k], m);
      v[k] = upper ? __fsub_rn(o, v[k]) : __fadd_rn(v[k], o);
    }
  }
  float y[4];
  uint32_t amax_bits = 0u;  // |y| as bits: non-negative floats order like their bits
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    y[k] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(v[k], inv_sqrt_n)));
    amax_bits = max(amax_bits, __float_as_uint(fabsf(y[k])));
  }
  const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, amax_bits));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint32_t packed = 0u;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(y[k], s), __NV_SATFINITE, __NV_E4M3);
    packed |= static_cast<uint32_t>(c) << (8 * k);
  }
  int64_t d = row;
  if (dst) {
    d = dst[row];
    if (d < 0 || d >= dst_rows) {
      if (lane == 0) raise_flag(status, kFlagBadIndex);
      return;
    }
  }
  *reinterpret_cast<uint32_t *>(codes + d * kProdDim + 4 * lane) = packed;
  if (lane == 0) scales[d] = s;
}

}  // namespace

cudaError_t launch_rotate_quant(const void *x, int rows, const int32_t *dst, int64_t dst_rows, uint8_t *codes,
                                float *scales, uint32_t *status, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const float inv_sqrt_n = static_cast<float>(1.0 / std::sqrt(static_cast<double>(kProdDim)));
  const int blocks = (rows + kProdWarps - 1) / kProdWarps;
  return launch_ex(false, rotate_quant_kernel, dim3(blocks), dim3(32 * kProdWarps), 0, stream, 1,
                   static_cast<const uint16_t *>(x), rows, inv_sqrt_n, dst, dst_rows, codes, scales, status);
}

}  // namespace sa
