// Per-query top-k of the index scores ("DeepSeek-V4.1-Flash-NVFP4
// inference/model.py", Indexer.forward: topk = min(index_topk, n_vis), the
// picks re-sorted into position order, -1 for unreachable picks).
//
// One CTA per query token.  The k-th largest score is found exactly by a
// most-significant-digit-first radix select over order-preserving 32-bit keys
// (four 8-bit digits), then one ordered compaction pass writes every position
// whose key is above that threshold plus the lowest-positioned ones equal to
// it, so ties go to the lower position and the output comes out ascending.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_radix_kernel(const float *__restrict__ scores, int64_t ld, int B, int N_c, int r,
                  const int32_t *__restrict__ q_seq, const int32_t *__restrict__ q_pos, int K,
                  int32_t *__restrict__ idx, uint32_t *status) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_eq[kTopkWarps], warp_take[kTopkWarps];
  __shared__ uint32_t sh_digit, sh_above;

  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Token tk;
  const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk, tid == 0);
  const int nv = ok ? tk.nv : 0;
  int32_t *out = idx + static_cast<int64_t>(t) * K;

  if (nv <= K) {  // every visible position is kept
    for (int i = tid; i < K; i += kTopkThreads) out[i] = i < nv ? i : -1;
    return;
  }

  const float *row = scores + static_cast<int64_t>(t) * ld;
  uint32_t prefix = 0, mask = 0;
  int remaining = K;  // picks still to make among keys matching `prefix`
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int s = tid; s < nv; s += kTopkThreads) {
      const uint32_t u = ordered_key(row[s]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 8l .. 8l+7; find the bin where the count of keys at
      // or above it first reaches `remaining`, scanning from the top.
      uint32_t c[8], local = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[8 * lane + j];
        local += c[j];
      }
      uint32_t sfx = local;  // keys in lanes >= this one
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, sfx, o);
        if (lane + o < 32) sfx += v;
      }
      const uint32_t above = sfx - local;
      if (above < static_cast<uint32_t>(remaining) && static_cast<uint32_t>(remaining) <= sfx) {
        uint32_t acc = above;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
          if (acc + c[j] >= static_cast<uint32_t>(remaining)) {
            sh_digit = 8 * lane + j;
            sh_above = acc;
            break;
          }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    remaining -= static_cast<int>(sh_above);
    prefix |= sh_digit << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t thr = prefix;
  const uint32_t need_eq = static_cast<uint32_t>(remaining);

  uint32_t sel_base = 0, eq_base = 0;
  for (int base = 0; base < nv; base += kTopkThreads) {
    const int s = base + tid;
    const uint32_t u = s < nv ? ordered_key(row[s]) : 0u;
    const bool gt = s < nv && u > thr;
    const bool eq = s < nv && u == thr;
    const uint32_t bal_eq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) warp_eq[warp] = __popc(bal_eq);
    __syncthreads();
    uint32_t eq_before = eq_base, eq_total = 0;
    for (int i = 0; i < kTopkWarps; ++i) {
      const uint32_t v = warp_eq[i];
      if (i < warp) eq_before += v;
      eq_total += v;
    }
    eq_before += __popc(bal_eq & lanemask_lt());
    const bool take = gt || (eq && eq_before < need_eq);
    const uint32_t bal_take = __ballot_sync(0xffffffffu, take);
    if (lane == 0) warp_take[warp] = __popc(bal_take);
    __syncthreads();
    uint32_t take_before = sel_base, take_total = 0;
    for (int i = 0; i < kTopkWarps; ++i) {
      const uint32_t v = warp_take[i];
      if (i < warp) take_before += v;
      take_total += v;
    }
    take_before += __popc(bal_take & lanemask_lt());
    if (take && take_before < static_cast<uint32_t>(K)) out[take_before] = s;
    sel_base += take_total;
    eq_base += eq_total;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_topk(const float *scores, int64_t ld, const sa_index_args &ia, int K,
                        int32_t *idx, uint32_t *status, cudaStream_t stream) {
  if (ia.T == 0 || K == 0) return cudaSuccess;
  topk_radix_kernel<<<ia.T, kTopkThreads, 0, stream>>>(scores, ld, ia.B, ia.N_c, ia.r, ia.q_seq,
                                                       ia.q_pos, K, idx, status);
  return cudaGetLastError();
}

}  // namespace sa
