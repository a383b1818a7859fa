// Per-query top-k of the index scores ("DeepSeek-V4.1-Flash-NVFP4
// inference/model.py", Indexer.forward: topk = min(index_topk, n_vis), the
// picks re-sorted into position order, -1 for unreachable picks).
//
// One CTA per query token.  The k-th largest score is found exactly by a
// most-significant-digit-first radix select over order-preserving 32-bit keys,
// then an ordered compaction writes every position whose key is above that
// threshold plus the lowest-positioned ones equal to it, so ties go to the
// lower position and the output comes out ascending.  Rows of up to 32768
// scores are held in registers (topk_reg_kernel); longer rows stream from
// global memory in four 8-bit passes (topk_radix_kernel).
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

  pdl_trigger();
  pdl_wait();  // the scores come from the previous kernel
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

// ---------------------------------------------------------------------------
// Register-resident variant for rows of up to kRegMax scores: each thread
// holds a contiguous block of E = ceil(n / 1024) keys, the K-th largest key is
// found by three radix passes of 11, 11 and 10 bits (warp-aggregated
// shared-memory histograms, one block-wide scan each), and the output offsets
// come from a single block scan of packed (greater, equal) counts: the number
// of picks before a thread is greater_before + min(equal_before, needed).

constexpr int kRegMax = 32768;
constexpr int kRegE = kRegMax / kTopkThreads;  // 32 keys per thread at most

// Block-wide exclusive scan of one uint32 per thread; returns the prefix and
// writes the total to *total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_sums, uint32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_sums[lane];
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - w;        // exclusive prefix of the warp totals
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const uint32_t r = warp_sums[warp] + incl - v;
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

// One radix pass: histogram of digit (key >> shift) & (nbins-1) over the keys
// that match `prefix` under `mask`, then locate the bin holding the
// `remaining`-th largest.  Returns the digit; `remaining` becomes the rank
// within that bin.
template <int E>
__device__ __forceinline__ uint32_t radix_pass(const uint32_t (&key)[E], int cnt, uint32_t prefix, uint32_t mask,
                                               int shift, int nbins, uint32_t *hist, uint32_t *warp_sums,
                                               int &remaining) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int i = tid; i < nbins; i += kTopkThreads) hist[i] = 0;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const bool in = e < cnt && (key[e] & mask) == prefix;
    const uint32_t active = __ballot_sync(0xffffffffu, in);
    if (in) {
      const uint32_t bin = (key[e] >> shift) & static_cast<uint32_t>(nbins - 1);
      const uint32_t peers = __match_any_sync(active, bin);
      if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[bin], __popc(peers));
    }
  }
  __syncthreads();
  // bins in descending order: thread t owns ranks r = 2t, 2t+1 (bin = nbins-1-r)
  uint32_t c0 = 0, c1 = 0;
  const int r0 = 2 * tid;
  if (r0 < nbins) c0 = hist[nbins - 1 - r0];
  if (r0 + 1 < nbins) c1 = hist[nbins - 2 - r0];
  uint32_t total;
  const uint32_t before = block_excl_scan(c0 + c1, warp_sums, &total);
  __shared__ uint32_t sel_digit, sel_above;
  const uint32_t rem = static_cast<uint32_t>(remaining);
  if (before < rem && rem <= before + c0 + c1) {
    if (rem <= before + c0) {
      sel_digit = nbins - 1 - r0;
      sel_above = before;
    } else {
      sel_digit = nbins - 2 - r0;
      sel_above = before + c0;
    }
  }
  __syncthreads();
  remaining -= static_cast<int>(sel_above);
  const uint32_t d = sel_digit;
  __syncthreads();
  return d;
}

template <int E>
__global__ void __launch_bounds__(kTopkThreads)
topk_reg_kernel(const float *__restrict__ scores, int64_t ld, int B, int N_c, int r,
                const int32_t *__restrict__ q_seq, const int32_t *__restrict__ q_pos, int K,
                int32_t *__restrict__ idx, uint32_t *status) {
  __shared__ uint32_t hist[2048];
  __shared__ uint32_t warp_sums[33];
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x;
  Token tk;
  const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk, tid == 0);
  const int nv = ok ? tk.nv : 0;
  pdl_wait();  // the scores come from the previous kernel
  int32_t *out = idx + static_cast<int64_t>(t) * K;
  if (nv <= K) {  // every visible position is kept
    for (int i = tid; i < K; i += kTopkThreads) out[i] = i < nv ? i : -1;
    return;
  }
  const float *row = scores + static_cast<int64_t>(t) * ld;
  const int per = (nv + kTopkThreads - 1) / kTopkThreads;  // <= E
  const int lo = tid * per;
  const int cnt = max(0, min(per, nv - lo));
  uint32_t key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) key[e] = e < cnt ? ordered_key(row[lo + e]) : 0u;

  int remaining = K;
  const uint32_t d1 = radix_pass<E>(key, cnt, 0u, 0u, 21, 2048, hist, warp_sums, remaining);
  const uint32_t p1 = d1 << 21, m1 = 0xFFE00000u;
  const uint32_t d2 = radix_pass<E>(key, cnt, p1, m1, 10, 2048, hist, warp_sums, remaining);
  const uint32_t p2 = p1 | (d2 << 10), m2 = 0xFFFFFC00u;
  const uint32_t d3 = radix_pass<E>(key, cnt, p2, m2, 0, 1024, hist, warp_sums, remaining);
  const uint32_t thr = p2 | d3;
  const uint32_t need_eq = static_cast<uint32_t>(remaining);

  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (e < cnt) {
      gt += key[e] > thr;
      eq += key[e] == thr;
    }
  }
  uint32_t tot;
  const uint32_t pre = block_excl_scan((gt << 16) | eq, warp_sums, &tot);
  const uint32_t gt_before = pre >> 16, eq_before = pre & 0xFFFFu;
  uint32_t pos = gt_before + min(eq_before, need_eq);
  uint32_t eq_seen = eq_before;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (e < cnt) {
      bool take = key[e] > thr;
      if (key[e] == thr) {
        take = eq_seen < need_eq;
        ++eq_seen;
      }
      if (take && pos < static_cast<uint32_t>(K)) out[pos++] = lo + e;
    }
  }
}

}  // namespace

cudaError_t launch_topk(const float *scores, int64_t ld, const sa_index_args &ia, int K,
                        int32_t *idx, uint32_t *status, cudaStream_t stream) {
  if (ia.T == 0 || K == 0) return cudaSuccess;
  // a row holds at most N_c visible scores
  auto kern = ia.N_c <= kRegMax / 4   ? topk_reg_kernel<kRegE / 4>
              : ia.N_c <= kRegMax / 2 ? topk_reg_kernel<kRegE / 2>
              : ia.N_c <= kRegMax     ? topk_reg_kernel<kRegE>
                                      : topk_radix_kernel;
  return launch_ex(false, kern, dim3(ia.T), dim3(kTopkThreads), 0, stream, 1, scores, ld, ia.B, ia.N_c, ia.r, ia.q_seq,
                    ia.q_pos, K, idx, status);
}

}  // namespace sa
