// Index scores: S[t, s] = sum_h w[t,h] * ReLU(q[t,h] . k[b,s]) * scales
// ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Indexer.forward: the
// einsum over the head dim, relu_(), times weights, sum over heads;
// "DeepSeek-V3.2-Exp inference/model.py", fp8_index with fp8 keys and one
// fp32 scale per position).
//
// This file holds the CUDA-core kernel (index heads of dim 64, bf16 keys and
// any shape the tensor-core kernel in idx_score_umma.cu does not take): one
// thread per key row, the token's
// index queries dequantised once into shared memory (fp32) and broadcast to
// all threads.  The products of a bf16/fp8 query element and an fp8/bf16 key
// element are exact in fp32; each head's dot product accumulates in fp32 in
// the order d = 0..D_I-1, the positive part is weighted and summed over the
// heads in order, and the key's scale multiplies the sum (all scales are
// positive, so this equals scaling inside the ReLU).
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int kScoreThreads = 128;

template <int DI, bool QFP8, bool KFP8>
__global__ void __launch_bounds__(kScoreThreads)
idx_score_simt_kernel(int B, int H_I, int N_c, int64_t kseq, int r, const int32_t *__restrict__ q_seq,
                      const int32_t *__restrict__ q_pos, const void *__restrict__ q_I,
                      const float *__restrict__ q_scale, const float *__restrict__ w,
                      const void *__restrict__ k_I, const float *__restrict__ k_scale,
                      float *__restrict__ scores, int64_t ld, int write_masked,
                      uint32_t *status) {
  extern __shared__ float4 smem4[];
  float *qs = reinterpret_cast<float *>(smem4);  // [H_I][DI]
  float *wq = qs + H_I * DI;                     // [H_I]

  const int t = blockIdx.y;
  const int s0 = blockIdx.x * kScoreThreads;
  const int s = s0 + threadIdx.x;
  float *row = scores + static_cast<int64_t>(t) * ld;

  Token tk;
  const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk,
                             blockIdx.x == 0 && threadIdx.x == 0);
  const int nv = ok ? tk.nv : 0;
  if (s0 >= nv) {
    if (write_masked && s < N_c) row[s] = -INFINITY;
    return;
  }

  const int64_t qbase = static_cast<int64_t>(t) * H_I * DI;
  for (int i = threadIdx.x; i < H_I * DI; i += kScoreThreads) {
    if (QFP8)
      qs[i] = e4m3_bits_to_float(static_cast<const uint8_t *>(q_I)[qbase + i]);
    else
      qs[i] = bf16_bits_to_float(static_cast<const uint16_t *>(q_I)[qbase + i]);
  }
  for (int h = threadIdx.x; h < H_I; h += kScoreThreads) {
    const float qsc = q_scale ? q_scale[static_cast<int64_t>(t) * H_I + h] : 1.f;
    wq[h] = w[static_cast<int64_t>(t) * H_I + h] * qsc;
  }
  __syncthreads();

  if (s >= N_c) return;
  if (s >= nv) {
    if (write_masked) row[s] = -INFINITY;
    return;
  }

  const int64_t krow = static_cast<int64_t>(tk.b) * kseq + s;  // kseq: key rows per sequence
  float kf[DI];
  if (KFP8) {
    const uint4 *kp = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(k_I) + krow * DI);
#pragma unroll
    for (int i = 0; i < DI / 16; ++i) {
      const uint4 v = __ldg(kp + i);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          kf[16 * i + 4 * j + e] = e4m3_bits_to_float(static_cast<uint8_t>(wv[j] >> (8 * e)));
    }
  } else {
    const uint4 *kp =
        reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(k_I) + krow * DI);
#pragma unroll
    for (int i = 0; i < DI / 8; ++i) {
      const uint4 v = __ldg(kp + i);
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        kf[8 * i + 2 * j] = __uint_as_float(wv[j] << 16);
        kf[8 * i + 2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
      }
    }
  }

  float acc = 0.f;
  for (int h = 0; h < H_I; ++h) {
    const float4 *qh = reinterpret_cast<const float4 *>(qs + h * DI);
    float dot = 0.f;
#pragma unroll
    for (int d4 = 0; d4 < DI / 4; ++d4) {
      const float4 q4 = qh[d4];
      dot = fmaf(q4.x, kf[4 * d4 + 0], dot);
      dot = fmaf(q4.y, kf[4 * d4 + 1], dot);
      dot = fmaf(q4.z, kf[4 * d4 + 2], dot);
      dot = fmaf(q4.w, kf[4 * d4 + 3], dot);
    }
    acc = fmaf(wq[h], fmaxf(dot, 0.f), acc);
  }
  const float ks = k_scale ? k_scale[krow] : 1.f;
  row[s] = acc * ks;
}

template <int DI, bool QFP8, bool KFP8>
cudaError_t launch_simt(const sa_index_args &ia, float *scores, int64_t ld, bool write_masked,
                        uint32_t *status, cudaStream_t stream) {
  auto kern = idx_score_simt_kernel<DI, QFP8, KFP8>;
  const size_t smem = (static_cast<size_t>(ia.H_I) * DI + ia.H_I) * sizeof(float);
  if (smem > 48 * 1024) {
    static bool attr_done[64] = {};
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), 64 * 1024 + 1024, attr_done);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((ia.N_c + kScoreThreads - 1) / kScoreThreads, ia.T);
  kern<<<grid, kScoreThreads, smem, stream>>>(ia.B, ia.H_I, ia.N_c, k_rows_per_seq(ia), ia.r, ia.q_seq, ia.q_pos,
                                              ia.q_I, ia.q_scale, ia.w, ia.k_I, ia.k_scale,
                                              scores, ld, write_masked ? 1 : 0, status);
  return cudaGetLastError();
}

}  // namespace

bool index_shape_supported(int H_I, int D_I) {
  return H_I >= 1 && H_I <= 128 && (D_I == 64 || D_I == 128);
}

size_t idx_score_scratch(const sa_index_args &ia) {
  return idx_score_umma_supported(ia) ? idx_score_umma_scratch(ia) : 0;
}

cudaError_t launch_idx_score(const sa_index_args &ia, float *scores, int64_t ld,
                             bool write_masked, void *scratch, uint32_t *status,
                             cudaStream_t stream) {
  if (ia.T == 0) return cudaSuccess;
  if (idx_score_umma_supported(ia))
    return launch_idx_score_umma(ia, scores, ld, write_masked, scratch, status, stream);
  const bool qf8 = ia.q_dtype == SA_FP8_E4M3, kf8 = ia.k_dtype == SA_FP8_E4M3;
#define SA_SCORE_CASE(DI, QF, KF)                                              \
  if (ia.D_I == DI && qf8 == QF && kf8 == KF)                                  \
    return launch_simt<DI, QF, KF>(ia, scores, ld, write_masked, status, stream);
  SA_SCORE_CASE(64, false, false)
  SA_SCORE_CASE(64, false, true)
  SA_SCORE_CASE(64, true, false)
  SA_SCORE_CASE(64, true, true)
  SA_SCORE_CASE(128, false, false)
  SA_SCORE_CASE(128, false, true)
  SA_SCORE_CASE(128, true, false)
  SA_SCORE_CASE(128, true, true)
#undef SA_SCORE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace sa
