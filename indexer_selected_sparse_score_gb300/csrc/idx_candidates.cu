// Level one of the two-level top-k ("DeepSeek-V4.1-Flash-NVFP4
// inference/model.py", select_candidate_blocks, called from Indexer.forward
// in the layer that is the candidate source).
//
// Positions [0, N_c) of a token's score row are cut into blocks of
// block_size positions, the last one short.  A block scores the best of its
// visible positions (positions at or past n_vis count as -inf); the block
// holding the newest visible position, (n_vis - 1) / block_size, is pinned to
// +inf; the min(topk_blocks, blocks) best blocks are taken, ties to the lower
// block, and those that score -inf are dropped.  The result is one bit per
// block (bit b % 32 of word b / 32).
//
// One CTA per token.  The block maxima are built in shared memory as
// order-preserving keys by shared atomicMax over the visible positions only
// (the row's loads go out in batches before any is used; a chunk of four
// positions inside one block folds to one atomic, and the atomic that finds a
// block at 0 counts it as reachable).  A block that is -inf or unreachable
// keeps key 0, which is never taken.  When more blocks are reachable than are
// taken, an exact radix select over the positive keys (11-bit digits from the
// top, then a direct ranking of a bin of at most 256 keys) finds the key of
// the last block taken; each warp then writes its run of 32-block words in
// order, taking the blocks equal to that key lowest-numbered first until the
// quota is met.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // ordered_key(-inf)
constexpr uint32_t kKeyPosInf = 0xFF800000u;  // ordered_key(+inf)
constexpr int kLoadBatch = 8;                 // float4 loads each thread has in flight
constexpr int kDigitBits = 11;                // radix digit over the finite keys' range
constexpr int kBins = 1 << kDigitBits;
constexpr int kFinish = 256;                  // a bin this small is ranked directly

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Block keys into shared memory: bkey[b] = the largest key of a visible
// position of block b above ordered_key(-inf), else 0.  Returns how many
// blocks this thread turned from 0 to a positive key (each reachable block
// is counted once, by the atomic that saw 0).
template <int NT>
__device__ __forceinline__ uint32_t block_maxima(const float *__restrict__ row, int nv, FastDiv dbs,
                                                 uint32_t *bkey) {
  const int tid = threadIdx.x;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const float ninf = __uint_as_float(0xFF800000u);
  uint32_t first = 0;
  for (int base = 0; base < nv; base += 4 * NT * kLoadBatch) {
    float4 f[kLoadBatch];
#pragma unroll
    for (int i = 0; i < kLoadBatch; ++i) {  // every load of the batch goes out before any is used
      const int p0 = base + 4 * (NT * i + tid);
      if (vec && p0 + 3 < nv) {
        f[i] = *reinterpret_cast<const float4 *>(row + p0);
      } else {
        f[i].x = p0 < nv ? row[p0] : ninf;
        f[i].y = p0 + 1 < nv ? row[p0 + 1] : ninf;
        f[i].z = p0 + 2 < nv ? row[p0 + 2] : ninf;
        f[i].w = p0 + 3 < nv ? row[p0 + 3] : ninf;
      }
    }
#pragma unroll
    for (int i = 0; i < kLoadBatch; ++i) {
      const int p0 = base + 4 * (NT * i + tid);
      if (p0 < nv) {
        const uint32_t k[4] = {ordered_key(f[i].x), ordered_key(f[i].y), ordered_key(f[i].z), ordered_key(f[i].w)};
        const uint32_t b0 = fast_div(p0, dbs);
        if (fast_div(p0 + 3, dbs) == b0) {  // the four positions share a block
          const uint32_t m = max(max(k[0], k[1]), max(k[2], k[3]));
          if (m > kKeyNegInf) first += atomicMax(&bkey[b0], m) == 0u;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (k[j] > kKeyNegInf) first += atomicMax(&bkey[fast_div(p0 + j, dbs)], k[j]) == 0u;
        }
      }
    }
  }
  return first;
}

// Block-wide exclusive scan of one value per thread (warp_sums: kWarps + 1
// words); returns the prefix and the total.
template <int NT>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *warp_sums, uint32_t &total) {
  constexpr int kWarps = NT / 32;
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
    const uint32_t w = lane < kWarps ? warp_sums[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) warp_sums[lane] = wi - w;
    if (lane == 31) warp_sums[kWarps] = wi;
  }
  __syncthreads();
  const uint32_t r = warp_sums[warp] + incl - v;
  total = warp_sums[kWarps];
  __syncthreads();
  return r;
}

struct SelectSmem {
  uint32_t hist[kBins];
  uint32_t warp_sums[33];
  uint32_t fin[kFinish];
  uint32_t nfin, digit, above, in_bin, fin_v, fin_gt, fin_eq;
};

// Sum over the warps of one value per warp held in part[0, kWarps): each warp
// reads all of them with one lane-parallel load (count = the first `count`).
template <int NT>
__device__ __forceinline__ uint32_t sum_parts(const uint32_t *part, int count) {
  const int lane = threadIdx.x & 31;
  return __reduce_add_sync(0xffffffffu, lane < count ? part[lane] : 0u);
}

// The n-th largest positive key among bkey[0, nb) -- ties to the lower block
// -- as (thr, need_eq): a block is taken if its key is above thr, or equal to
// it and among the first need_eq such blocks.  Needs n >= 1 and more than n
// positive keys.  Radix select from the top, 11 bits at a time; once the
// chosen bin holds at most kFinish keys they are ranked directly.
template <int NT>
__device__ void select_threshold(const uint32_t *bkey, int nb, uint32_t n, SelectSmem &sm, uint32_t &thr,
                                 uint32_t &need_eq) {
  const int tid = threadIdx.x;
  uint32_t remaining = n, prefix = 0u, eq_total = 0u;
  for (int hi = 32; hi > 0;) {
    const int nbits = hi < kDigitBits ? hi : kDigitBits, shift = hi - nbits;
    const uint32_t nbins = 1u << nbits;
    const uint32_t fixed = hi >= 32 ? 0u : ~((1u << hi) - 1u);  // bits already chosen
    for (int i = tid; i < kBins; i += NT) sm.hist[i] = 0u;
    __syncthreads();
    for (int b = tid; b < nb; b += NT) {
      const uint32_t u = bkey[b];
      if (u != 0u && (u & fixed) == prefix) atomicAdd(&sm.hist[(u >> shift) & (nbins - 1u)], 1u);
    }
    __syncthreads();
    // bins in descending order: thread t owns ranks R t .. R t + R - 1 (bin nbins - 1 - rank)
    constexpr int R = (kBins + NT - 1) / NT;
    uint32_t c[R], sum = 0;
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int rk = R * tid + k;
      c[k] = rk < static_cast<int>(nbins) ? sm.hist[nbins - 1 - rk] : 0u;
      sum += c[k];
    }
    uint32_t total;
    const uint32_t before = block_scan<NT>(sum, sm.warp_sums, total);
    if (before < remaining && remaining <= before + sum) {
      uint32_t run = before;
#pragma unroll
      for (int k = 0; k < R; ++k) {
        if (run < remaining && remaining <= run + c[k]) {
          sm.digit = nbins - 1 - (R * tid + k);
          sm.above = run;
          sm.in_bin = c[k];
        }
        run += c[k];
      }
    }
    __syncthreads();
    remaining -= sm.above;
    prefix |= sm.digit << shift;
    eq_total = sm.in_bin;
    hi = shift;
    __syncthreads();
    if (hi > 0 && eq_total <= static_cast<uint32_t>(kFinish)) {
      // rank the bin's keys directly: the value v with #(> v) < remaining <= #(>= v)
      if (tid == 0) sm.nfin = 0;
      __syncthreads();
      const uint32_t fx = ~((1u << hi) - 1u);
      for (int b = tid; b < nb; b += NT) {
        const uint32_t u = bkey[b];
        if (u != 0u && (u & fx) == prefix) sm.fin[atomicAdd(&sm.nfin, 1u)] = u;
      }
      __syncthreads();
      const uint32_t m = sm.nfin;
      if (static_cast<uint32_t>(tid) < m) {
        const uint32_t v = sm.fin[tid];
        uint32_t gt = 0, eq = 0;
        for (uint32_t j = 0; j < m; ++j) {
          gt += sm.fin[j] > v;
          eq += sm.fin[j] == v;
        }
        if (gt < remaining && remaining <= gt + eq) {  // every thread holding v agrees
          sm.fin_v = v;
          sm.fin_gt = gt;
          sm.fin_eq = eq;
        }
      }
      __syncthreads();
      prefix = sm.fin_v;
      remaining -= sm.fin_gt;
      eq_total = sm.fin_eq;
      __syncthreads();
      break;
    }
  }
  thr = prefix;
  need_eq = remaining;
  if (need_eq == eq_total) {  // every key equal to thr is taken: keep = key >= thr
    thr -= 1u;                // thr >= 1: a positive key
    need_eq = 0u;
  }
}

template <int NT>
__global__ void __launch_bounds__(NT)
candidate_blocks_kernel(const float *__restrict__ scores, int64_t ld, int B, int N_c, int r,
                        const int32_t *__restrict__ q_seq, const int32_t *__restrict__ q_pos, int bs, FastDiv dbs,
                        int topk_blocks, int words, uint32_t *__restrict__ cand, uint32_t *status) {
  constexpr int kWarps = NT / 32;
  extern __shared__ uint32_t bkey[];  // [32 * words] block keys; 0 is never taken
  __shared__ SelectSmem sm;
  __shared__ uint32_t pin_new;
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = static_cast<int>((static_cast<int64_t>(N_c) + bs - 1) / bs);
  for (int i = tid; i < 32 * words; i += NT) bkey[i] = 0u;
  pdl_wait();  // the scores come from the previous kernel
  Token tk;
  const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk, tid == 0);
  const int nv = ok ? tk.nv : 0;
  __syncthreads();

  // block maxima and the reachable count
  uint32_t first = block_maxima<NT>(scores + static_cast<int64_t>(t) * ld, nv, dbs, bkey);
  first = __reduce_add_sync(0xffffffffu, first);
  if (lane == 0) sm.warp_sums[warp] = first;
  __syncthreads();
  if (tid == 0) {
    pin_new = 0u;
    if (nv >= 1) {  // the newest block is pinned
      const int b = (nv - 1) / bs;
      pin_new = bkey[b] == 0u;
      bkey[b] = kKeyPosInf;
    }
  }
  __syncthreads();
  const uint32_t reach = pin_new + sum_parts<NT>(sm.warp_sums, kWarps);
  __syncthreads();

  // keep = key > thr, or key == thr among the first need_eq such blocks
  const uint32_t n = static_cast<uint32_t>(min(topk_blocks, nb));
  uint32_t thr = 0u, need_eq = 0u;  // every reachable block
  if (n == 0u)
    thr = 0xFFFFFFFFu;  // no block
  else if (reach > n)
    select_threshold<NT>(bkey, nb, n, sm, thr, need_eq);

  // warp w writes words [w * per, (w + 1) * per) in order
  const int per = (words + kWarps - 1) / kWarps;
  const int w_begin = min(words, warp * per), w_end = min(words, w_begin + per);
  uint32_t eq_seen = 0;  // blocks equal to thr in lower words
  if (need_eq > 0u) {
    uint32_t eq_cnt = 0;
    for (int w = w_begin; w < w_end; ++w) eq_cnt += __popc(__ballot_sync(0xffffffffu, bkey[32 * w + lane] == thr));
    if (lane == 0) sm.warp_sums[warp] = eq_cnt;
    __syncthreads();
    eq_seen = sum_parts<NT>(sm.warp_sums, warp);
  }
  uint32_t *out = cand + static_cast<int64_t>(t) * words;
  for (int w = w_begin; w < w_end; ++w) {
    const uint32_t u = bkey[32 * w + lane];
    const bool eq = u == thr;
    const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
    const uint32_t rank = eq_seen + __popc(eqm & lanemask_lt());
    const uint32_t take = __ballot_sync(0xffffffffu, u > thr || (eq && rank < need_eq));
    eq_seen += __popc(eqm);
    if (lane == 0) out[w] = take;
  }
}

}  // namespace

int candidate_words(int N_c, int block_size) {
  const int64_t nb = (static_cast<int64_t>(N_c) + block_size - 1) / block_size;
  return static_cast<int>((nb + 31) / 32);
}

cudaError_t launch_candidate_blocks(const float *scores, int64_t ld, const sa_index_args &ia, int block_size,
                                   int topk_blocks, uint32_t *cand, uint32_t *status, cudaStream_t stream) {
  if (ia.T == 0) return cudaSuccess;
  // 1024 threads while each SM holds about one row, 512 when rows outnumber the SMs
  const bool many_rows = ia.T > 2 * sm_count();
  const auto kern = many_rows ? candidate_blocks_kernel<512> : candidate_blocks_kernel<1024>;
  static bool attr_done[2][64] = {};
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), sizeof(uint32_t) * kMaxCandidateBlocks,
                                attr_done[many_rows ? 0 : 1]);
  if (e != cudaSuccess) return e;
  const int words = candidate_words(ia.N_c, block_size);
  return launch_ex(false, kern, dim3(ia.T), dim3(many_rows ? 512 : 1024), sizeof(uint32_t) * 32 * words, stream, 1,
                   scores, ld, ia.B, ia.N_c, ia.r, ia.q_seq, ia.q_pos, block_size,
                   make_fastdiv(static_cast<uint32_t>(block_size)), topk_blocks, words, cand, status);
}

}  // namespace sa
