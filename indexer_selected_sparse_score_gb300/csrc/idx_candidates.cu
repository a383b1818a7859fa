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
// order-preserving keys by shared atomicMax over the visible positions only (a
// chunk of four positions inside one block folds to one atomic); a block that
// is -inf or unreachable keeps key 0, which is never taken.  When more blocks
// are reachable than are taken, an exact radix select (four 8-bit passes over
// the block keys) finds the key of the last block taken; each warp then writes
// its run of 32-block words in order, taking the blocks equal to that key
// lowest-numbered first until the quota is met.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // ordered_key(-inf)
constexpr uint32_t kKeyPosInf = 0xFF800000u;  // ordered_key(+inf)
constexpr int kLoadBatch = 8;                 // float4 loads each thread has in flight

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Block keys into shared memory: bkey[b] = the largest key of a visible
// position of block b above ordered_key(-inf), else 0; the newest block gets
// ordered_key(+inf).
template <int NT>
__device__ __forceinline__ void block_maxima(const float *__restrict__ row, int nv, FastDiv dbs, int bs,
                                             uint32_t *bkey) {
  const int tid = threadIdx.x;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const float ninf = __uint_as_float(0xFF800000u);
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
          if (m > kKeyNegInf) atomicMax(&bkey[b0], m);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (k[j] > kKeyNegInf) atomicMax(&bkey[fast_div(p0 + j, dbs)], k[j]);
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && nv >= 1) bkey[(nv - 1) / bs] = kKeyPosInf;  // the newest block is pinned
  __syncthreads();
}

template <int NT>
__global__ void __launch_bounds__(NT)
candidate_blocks_kernel(const float *__restrict__ scores, int64_t ld, int B, int N_c, int r,
                        const int32_t *__restrict__ q_seq, const int32_t *__restrict__ q_pos, int bs, FastDiv dbs,
                        int topk_blocks, int words, uint32_t *__restrict__ cand, uint32_t *status) {
  constexpr int kWarps = NT / 32;
  extern __shared__ uint32_t bkey[];  // [32 * words] block keys; 0 is never taken
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sums[kWarps];
  __shared__ uint32_t sh_digit, sh_above;
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nb = static_cast<int>((static_cast<int64_t>(N_c) + bs - 1) / bs);
  for (int i = tid; i < 32 * words; i += NT) bkey[i] = 0u;
  pdl_wait();  // the scores come from the previous kernel
  Token tk;
  const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk, tid == 0);
  const int nv = ok ? tk.nv : 0;
  __syncthreads();
  block_maxima<NT>(scores + static_cast<int64_t>(t) * ld, nv, dbs, bs, bkey);

  // reachable blocks (key > 0)
  uint32_t c = 0;
  for (int b = tid; b < nb; b += NT) c += bkey[b] != 0u;
  c = __reduce_add_sync(0xffffffffu, c);
  if (lane == 0) warp_sums[warp] = c;
  __syncthreads();
  uint32_t reach = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) reach += warp_sums[i];
  __syncthreads();

  // keep = key > thr, or key == thr among the first need_eq such blocks
  const uint32_t n = static_cast<uint32_t>(min(topk_blocks, nb));
  uint32_t thr = 0u, need_eq = 0u;  // every reachable block
  if (n == 0u) {
    thr = 0xFFFFFFFFu;  // no block
  } else if (reach > n) {
    uint32_t prefix = 0u, mask = 0u, remaining = n;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += NT) hist[i] = 0u;
      __syncthreads();
      // block maxima crowd into few bins: lanes with the same bin add once
      for (int base = 0; base < nb; base += NT) {
        const int b = base + tid;
        const uint32_t u = b < nb ? bkey[b] : 0u;
        const bool act = b < nb && (u & mask) == prefix;
        const uint32_t bin = act ? (u >> shift) & 255u : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (act && __ffs(peers) - 1 == lane) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 8l .. 8l+7: find the bin where the count of keys
        // at or above it first reaches `remaining`, from the top bin down
        uint32_t cb[8], local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cb[j] = hist[8 * lane + j];
          local += cb[j];
        }
        uint32_t sfx = local;  // keys in this lane's bins and above
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t v = __shfl_down_sync(0xffffffffu, sfx, o);
          if (lane + o < 32) sfx += v;
        }
        const uint32_t above = sfx - local;
        if (above < remaining && remaining <= sfx) {
          uint32_t acc = above;
#pragma unroll
          for (int j = 7; j >= 0; --j) {
            if (acc + cb[j] >= remaining) {
              sh_digit = 8 * lane + j;
              sh_above = acc;
              break;
            }
            acc += cb[j];
          }
        }
      }
      __syncthreads();
      remaining -= sh_above;
      prefix |= sh_digit << shift;
      mask |= 255u << shift;
      __syncthreads();
    }
    thr = prefix;
    need_eq = remaining;
  }

  // warp w writes words [w * per, (w + 1) * per) in order
  const int per = (words + kWarps - 1) / kWarps;
  const int w_begin = min(words, warp * per), w_end = min(words, w_begin + per);
  uint32_t eq_cnt = 0;
  for (int w = w_begin; w < w_end; ++w) eq_cnt += __popc(__ballot_sync(0xffffffffu, bkey[32 * w + lane] == thr));
  if (lane == 0) warp_sums[warp] = eq_cnt;
  __syncthreads();
  uint32_t eq_seen = 0;  // blocks equal to thr in lower words
  for (int i = 0; i < warp; ++i) eq_seen += warp_sums[i];
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
