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
//
// Level two of the two-level top-k ("DeepSeek-V4.1-Flash-NVFP4
// inference/model.py", Indexer.forward in a layer that uses candidates) is the
// same selection on scores masked to -inf outside the kept candidate blocks:
// given a block mask, both kernels apply it as they read the row.
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

// Whether position s lies in a kept block of a candidate mask row (bit b % 32
// of word b / 32 for block b = s / block_size).
__device__ __forceinline__ bool cand_kept(const uint32_t *crow, int s, FastDiv dbs) {
  const uint32_t b = fast_div(static_cast<uint32_t>(s), dbs);
  return (crow[b >> 5] >> (b & 31)) & 1u;
}

constexpr uint32_t kNegInfBits = 0xFF800000u;  // fp32 -inf

__global__ void __launch_bounds__(kTopkThreads)
topk_radix_kernel(const float *__restrict__ scores, int64_t ld, int B, int N_c, int r,
                  const int32_t *__restrict__ q_seq, const int32_t *__restrict__ q_pos, int K,
                  int32_t *__restrict__ idx, uint32_t *status, const uint32_t *__restrict__ cmask,
                  int cand_words, FastDiv dbs) {
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
  const uint32_t *crow = cmask ? cmask + static_cast<int64_t>(t) * cand_words : nullptr;
  auto key_at = [&](int s) {
    return crow && !cand_kept(crow, s, dbs) ? ordered_key(__uint_as_float(kNegInfBits)) : ordered_key(row[s]);
  };
  uint32_t prefix = 0, mask = 0;
  int remaining = K;  // picks still to make among keys matching `prefix`
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int s = tid; s < nv; s += kTopkThreads) {
      const uint32_t u = key_at(s);
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
    const uint32_t u = s < nv ? key_at(s) : 0u;
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
// Register-resident variant for rows of up to kRegMax scores: slot e of
// thread i holds position NT e + i, so the row's loads depend only on N_c and
// go out at once (before the token's visible count is known), any row length
// spreads evenly over the threads, and slot e of a warp covers 32 consecutive
// positions: one word of a position bitmap, formed by one ballot.  The keys are
// first reduced to their range (key - min, an order-preserving shift), so the
// radix digits cover only the L = bit length of (max - min) bits the row
// actually uses: the first pass spreads the row over its bins (plain shared
// atomics, little contention) and a bin of at most kFinish keys is ranked
// directly.  Slots past the visible count hold key 0, the smallest: with more
// than K visible keys they change neither the k-th largest value nor, as they
// sit at the highest positions, which of the keys equal to it are taken, so no
// pass tests them.  The picks go into two position bitmaps in shared memory
// (above the k-th key, equal to it); one block scan over the words then writes
// them in ascending order, the equal ones lowest position first.

constexpr int kRegMax = 32768;
constexpr int kDigitBits = 11;                 // radix digit width
constexpr int kDigitBins = 1 << kDigitBits;
constexpr int kFinish = 256;                   // a bin this small is ranked directly
// The register top-k runs with NT threads: 1024 when each SM holds about one
// row (one row's latency is the step's), 512 when rows outnumber the SMs (two
// CTAs per SM keep more rows in flight); E keys per thread cover E * NT
// positions.

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
    uint32_t w = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0u;
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

// Shared state of one register top-k CTA.
struct RegSel {
  uint32_t warp_sums[33];
  uint32_t digit, above, count;    // the pass's chosen bin
  uint32_t ncand, fin_above;
  uint32_t cand[kFinish];          // the last bin's keys and positions
  int32_t cpos[kFinish];
};

// One radix pass: histogram of digit (key >> shift) & (nbins-1) over the keys
// that match `prefix` under `mask`, then locate the bin holding the
// `remaining`-th largest.  Returns the digit; `remaining` becomes the rank
// within that bin.  kFirst: the first pass, whose keys all match (they are
// below 2^L and shift + log2(nbins) = L) and whose histogram was zeroed before
// the block's first barrier.  kBounded: only slots below `nslots` (the same for
// every thread) are counted.  Each warp sums its threads' bins; every warp then
// finds, from the warp totals, the warp whose bins hold the rank, and that
// warp alone locates the bin.
template <int E, int NT, bool kFirst, bool kBounded = false>
__device__ __forceinline__ uint32_t radix_pass(const uint32_t (&key)[E], uint32_t prefix, uint32_t mask, int shift,
                                               int nbins, uint32_t *hist, RegSel &rs, int &remaining,
                                               uint32_t &in_bin, int nslots = E) {
  constexpr int R = kDigitBins / NT;  // ranks (bins) per thread
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if constexpr (!kFirst) {
    for (int i = tid; i < nbins; i += NT) hist[i] = 0;
    __syncthreads();
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (kBounded && e >= nslots) break;  // kBounded: slots from nslots on hold no key of any thread
    if constexpr (kFirst)
      atomicAdd(&hist[key[e] >> shift], 1u);
    else if ((key[e] & mask) == prefix)
      atomicAdd(&hist[(key[e] >> shift) & static_cast<uint32_t>(nbins - 1)], 1u);
  }
  __syncthreads();
  // bins in descending order: thread t owns ranks R t .. R t + R - 1 (bin nbins-1-rank)
  uint32_t c[R], sum = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int rk = R * tid + k;
    c[k] = rk < nbins ? hist[nbins - 1 - rk] : 0u;
    sum += c[k];
  }
  const uint32_t wsum = __reduce_add_sync(0xffffffffu, sum);
  if (lane == 0) rs.warp_sums[warp] = wsum;
  __syncthreads();
  const uint32_t rem = static_cast<uint32_t>(remaining);
  const uint32_t wv = lane < kWarps ? rs.warp_sums[lane] : 0u;
  uint32_t wincl = wv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += y;
  }
  // the ranks above `rem` exist (rem <= the keys counted), so some warp reaches it
  const int sw = __ffs(__ballot_sync(0xffffffffu, wincl >= rem)) - 1;
  if (warp == sw) {
    const uint32_t before = __shfl_sync(0xffffffffu, wincl - wv, sw);
    uint32_t li = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, li, o);
      if (lane >= o) li += y;
    }
    if (lane == __ffs(__ballot_sync(0xffffffffu, before + li >= rem)) - 1) {
      uint32_t run = before + li - sum;
#pragma unroll
      for (int k = 0; k < R; ++k) {
        if (run < rem && rem <= run + c[k]) {
          rs.digit = static_cast<uint32_t>(nbins - 1 - (R * tid + k));
          rs.above = run;
          rs.count = c[k];
        }
        run += c[k];
      }
    }
  }
  __syncthreads();
  // rs is rewritten only after the next pass's first barrier, which every
  // thread reaches after these reads
  remaining -= static_cast<int>(rs.above);
  in_bin = rs.count;
  return rs.digit;
}

// Resident CTAs per SM the register budget is set for: two at 512 threads
// (while E keys fit in half the register file), else one.
template <int E, int NT>
constexpr int kRegCtasPerSm = (NT <= 512 && E <= 32) ? 2 : 1;

template <int E, int NT, bool kCand>
__global__ void __launch_bounds__(NT, (kRegCtasPerSm<E, NT>))
topk_reg_kernel(const float *__restrict__ scores, int64_t ld, int B, int N_c, int r,
                const int32_t *__restrict__ q_seq, const int32_t *__restrict__ q_pos, int K,
                int32_t *__restrict__ idx, uint32_t *status, const uint32_t *__restrict__ cmask,
                int cand_words, FastDiv dbs) {
  static_assert(E % 8 == 0 && E * NT <= kRegMax, "keys per thread");
  constexpr int kWarps = NT / 32;
  constexpr int kWords = E * NT / 32;                       // bitmap words: one per (slot, warp)
  constexpr int kWordsPerThread = (kWords + NT - 1) / NT;   // in the ordered write-out
  __shared__ uint32_t hist[kDigitBins];
  __shared__ uint32_t sel_gt[kWords], sel_eq[kWords];       // pick bitmaps by position
  __shared__ RegSel rs;
  __shared__ uint32_t wmin[kWarps], wmax[kWarps];
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the token arrays are inputs of the call, not outputs of the previous
  // kernel: read them before waiting for it, so that the score loads can stop
  // at the visible count
  Token tk;
  const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk, tid == 0);
  const int nv = ok ? tk.nv : 0;
  int32_t *out = idx + static_cast<int64_t>(t) * K;
  pdl_wait();  // the scores come from the previous kernel
  if (nv <= K) {  // every visible position is kept
    for (int i = tid; i < K; i += NT) out[i] = i < nv ? i : -1;
    return;
  }
  // the visible slots of a thread are a prefix of its E
  const int cnt = tid < nv ? min(E, (nv - tid + NT - 1) / NT) : 0;
  const float *row = scores + static_cast<int64_t>(t) * ld + tid;
  uint32_t key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) key[e] = e < cnt ? __float_as_uint(row[NT * e]) : 0u;
  // the row's candidate mask (kCand) goes to shared memory with one load per
  // thread, issued beside the score loads
  __shared__ uint32_t cwords[kCand ? kRegMax / 32 : 1];
  if constexpr (kCand) {
    const uint32_t *crow = cmask + static_cast<int64_t>(t) * cand_words;
    for (int i = tid; i < cand_words; i += NT) cwords[i] = crow[i];
  }
  for (int i = tid; i < kDigitBins; i += NT) hist[i] = 0;  // the first pass's histogram
  for (int i = tid; i < kWords; i += NT) sel_eq[i] = 0u;
  if (tid == 0) rs.ncand = 0;
  if constexpr (kCand) {
    // positions outside the kept candidate blocks score -inf
    __syncthreads();  // the mask words are in shared memory
    if (NT % (32 * dbs.d) == 0) {
      // NT a multiple of 32 block sizes: position NT e + tid lies in block
      // NT e / size + tid / size, i.e. the same bit of a mask word that moves
      // NT / (32 size) words per slot
      const uint32_t tb = fast_div(static_cast<uint32_t>(tid), dbs);
      const uint32_t *cw = cwords + (tb >> 5), bit = 1u << (tb & 31u);
      const int step = NT / (32 * static_cast<int>(dbs.d));
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (e < cnt && !(cw[step * e] & bit)) key[e] = kNegInfBits;
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (e < cnt && !cand_kept(cwords, NT * e + tid, dbs)) key[e] = kNegInfBits;
    }
  }
  // the row's key range: keys become key - min (< 2^L)
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (e < cnt) {
      key[e] = ordered_key(__uint_as_float(key[e]));
      kmin = min(kmin, key[e]);
      kmax = max(kmax, key[e]);
    }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    wmin[warp] = kmin;
    wmax[warp] = kmax;
  }
  __syncthreads();
  kmin = __reduce_min_sync(0xffffffffu, lane < kWarps ? wmin[lane] : 0xFFFFFFFFu);
  kmax = __reduce_max_sync(0xffffffffu, lane < kWarps ? wmax[lane] : 0u);
#pragma unroll
  for (int e = 0; e < E; ++e) key[e] = e < cnt ? key[e] - kmin : 0u;
  const int L = kmax > kmin ? 32 - __clz(kmax - kmin) : 0;

  // radix select over bits [0, L), kDigitBits at a time from the top, until
  // the chosen bin holds at most kFinish keys or every bit is fixed
  int remaining = K, hi = L;
  uint32_t thr = 0u, in_bin = 0u;
  if (hi > 0) {
    const int nb = hi < kDigitBits ? hi : kDigitBits, shift = hi - nb;
    thr = radix_pass<E, NT, true>(key, 0u, 0u, shift, 1 << nb, hist, rs, remaining, in_bin) << shift;
    hi = shift;
  }
  while (hi > 0 && in_bin > static_cast<uint32_t>(kFinish)) {
    const int nb = hi < kDigitBits ? hi : kDigitBits, shift = hi - nb;
    const uint32_t mask = ~((1u << hi) - 1u);  // bits already fixed (hi < 32 after the first pass)
    thr |= radix_pass<E, NT, false>(key, thr, mask, shift, 1 << nb, hist, rs, remaining, in_bin) << shift;
    hi = shift;
  }
  uint32_t need_eq;
  if (hi > 0) {
    // keys above the chosen bin are picks: one ballot per slot fills the
    // bitmap word of the warp's 32 positions; the bin's keys (at most
    // kFinish) are gathered with their positions and ranked directly
    const uint32_t fixed = ~((1u << hi) - 1u);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t kf = key[e] & fixed;
      const uint32_t above = __ballot_sync(0xffffffffu, kf > thr);
      if (lane == 0) sel_gt[kWarps * e + warp] = above;
      const uint32_t inb = __ballot_sync(0xffffffffu, kf == thr);
      if (inb != 0u) {
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(&rs.ncand, static_cast<uint32_t>(__popc(inb)));
        base = __shfl_sync(0xffffffffu, base, 0);
        if ((inb >> lane) & 1u) {
          const uint32_t i = base + __popc(inb & lanemask_lt());
          rs.cand[i] = key[e];
          rs.cpos[i] = NT * e + tid;
        }
      }
    }
    __syncthreads();
    // the remaining-th largest among the candidates is the value v with
    // #(> v) < remaining <= #(>= v); candidate i is above it exactly when
    // #(>= its key) < remaining, equal to it when #(> its key) < remaining <=
    // #(>= its key), so each candidate places its own bit
    const uint32_t n = rs.ncand, rem2 = static_cast<uint32_t>(remaining);
    if (static_cast<uint32_t>(tid) < n) {
      const uint32_t v = rs.cand[tid];
      uint32_t gt = 0, ge = 0;
      for (uint32_t j = 0; j < n; ++j) {
        const uint32_t u = rs.cand[j];
        gt += u > v;
        ge += u >= v;
      }
      const int p = rs.cpos[tid];
      if (ge < rem2)
        atomicOr(&sel_gt[p >> 5], 1u << (p & 31));
      else if (gt < rem2) {
        atomicOr(&sel_eq[p >> 5], 1u << (p & 31));
        rs.fin_above = gt;  // the same from every candidate equal to the k-th key
      }
    }
    __syncthreads();
    need_eq = rem2 - rs.fin_above;
  } else {
    // every bit fixed: thr is the k-th largest key itself
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t gt = __ballot_sync(0xffffffffu, key[e] > thr);
      const uint32_t eq = __ballot_sync(0xffffffffu, key[e] == thr);
      if (lane == 0) {
        sel_gt[kWarps * e + warp] = gt;
        sel_eq[kWarps * e + warp] = eq;
      }
    }
    __syncthreads();
    need_eq = static_cast<uint32_t>(remaining);
  }

  // thread i writes the picks among its words of 32 positions, in order
  uint32_t ng = 0, ne = 0;
#pragma unroll
  for (int w = 0; w < kWordsPerThread; ++w) {
    const int wi = kWordsPerThread * tid + w;
    if (wi < kWords) {
      ng += __popc(sel_gt[wi]);
      ne += __popc(sel_eq[wi]);
    }
  }
  uint32_t tot;
  const uint32_t pre = block_excl_scan((ng << 16) | ne, rs.warp_sums, &tot);
  uint32_t eq_seen = pre & 0xFFFFu;  // equal keys at lower positions
  uint32_t o = (pre >> 16) + min(eq_seen, need_eq);
#pragma unroll
  for (int w = 0; w < kWordsPerThread; ++w) {
    const int wi = kWordsPerThread * tid + w;
    if (wi >= kWords) break;
    uint32_t take = sel_gt[wi], x = sel_eq[wi];
    for (; x != 0u && eq_seen < need_eq; ++eq_seen) {  // equal keys, lowest positions first
      take |= x & (0u - x);
      x &= x - 1u;
    }
    eq_seen += __popc(x);  // equal keys past the quota
    while (take != 0u) {
      const int bit = __ffs(take) - 1;
      if (o < static_cast<uint32_t>(K)) out[o] = 32 * wi + bit;
      ++o;
      take &= take - 1u;
    }
  }
}

// ---------------------------------------------------------------------------
// Level two with compaction, for candidate blocks of at least kCompactMinBlock
// positions: the selection runs over the kept visible positions alone, listed
// in ascending order (kept block ids in shared memory; candidate c is position
// list[c / size] * size + c % size), so its slots stop at the row's candidate
// count instead of the row's length.  The row the selection stands for is the
// visible row with -inf outside the kept blocks.  Its k-th largest value is a
// candidate's while at least K candidates score above -inf (nfin >= K): the
// radix select then runs over the candidates' keys, and every other position
// lies below it.  Otherwise it is -inf: every candidate above -inf is a pick,
// and the rest are the lowest-positioned of the positions that score -inf
// (candidates at -inf and the visible positions outside the kept blocks).
// Candidate slots past the count hold key 0 and set no bit: as with the
// register kernel, they sit below every candidate and are never needed to fill
// the picks of the value they may tie.
constexpr int kCompactMinBlock = 4;                    // the block list fits 8192 uint16 entries
constexpr uint32_t kNegInfKey = ~kNegInfBits;          // ordered key of -inf

template <int E, int NT>
__global__ void __launch_bounds__(NT, (kRegCtasPerSm<E, NT>))
topk_cand_kernel(const float *__restrict__ scores, int64_t ld, int B, int N_c, int r,
                 const int32_t *__restrict__ q_seq, const int32_t *__restrict__ q_pos, int K,
                 int32_t *__restrict__ idx, uint32_t *status, const uint32_t *__restrict__ cmask,
                 int cand_words, FastDiv dbs) {
  static_assert(E % 8 == 0 && E * NT <= kRegMax, "keys per thread");
  constexpr int kWarps = NT / 32;
  constexpr int kWords = E * NT / 32;                       // position bitmap words
  constexpr int kWordsPerThread = (kWords + NT - 1) / NT;
  constexpr int kMaxBlocks = kRegMax / kCompactMinBlock;
  __shared__ uint32_t hist[kDigitBins];
  __shared__ uint32_t sel_gt[kWords], sel_eq[kWords];
  __shared__ RegSel rs;
  __shared__ uint32_t wred[3][kWarps];
  __shared__ uint32_t cwords[kRegMax / 32];
  __shared__ uint16_t blist[kMaxBlocks];                    // kept visible blocks, ascending
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Token tk;
  const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk, tid == 0);
  const int nv = ok ? tk.nv : 0;
  int32_t *out = idx + static_cast<int64_t>(t) * K;
  pdl_wait();  // the scores and the block mask come from the previous kernels
  if (nv <= K) {  // every visible position is kept
    for (int i = tid; i < K; i += NT) out[i] = i < nv ? i : -1;
    return;
  }
  const uint32_t bs = dbs.d;
  const int nbv = static_cast<int>(fast_div(static_cast<uint32_t>(nv) + bs - 1u, dbs));  // blocks holding a visible position
  const int nwv = (nbv + 31) >> 5;                                                      // their mask words
  const uint32_t *crow = cmask + static_cast<int64_t>(t) * cand_words;
  for (int i = tid; i < kDigitBins; i += NT) hist[i] = 0;  // the first pass's histogram
  for (int i = tid; i < kWords; i += NT) {
    sel_gt[i] = 0u;
    sel_eq[i] = 0u;
  }
  if (tid == 0) rs.ncand = 0;
  // the kept visible blocks in ascending order: a block scan of the mask words'
  // counts, then each thread lists its words' blocks (one word per thread per round)
  uint32_t listed = 0;  // blocks listed by earlier rounds
  for (int w0 = 0; w0 < nwv; w0 += NT) {
    const int w = w0 + tid;
    uint32_t m = 0u;
    if (w < nwv) {
      m = crow[w];
      if (w == nwv - 1 && (nbv & 31)) m &= (1u << (nbv & 31)) - 1u;  // blocks past the visible end
      cwords[w] = m;
    }
    uint32_t tot;
    uint32_t o = listed + block_excl_scan(static_cast<uint32_t>(__popc(m)), rs.warp_sums, &tot);
    for (uint32_t x = m; x != 0u; x &= x - 1u) blist[o++] = static_cast<uint16_t>(32 * w + __ffs(x) - 1);
    listed += tot;
  }
  __syncthreads();  // the list and the mask words are in shared memory
  const int nkept = static_cast<int>(listed);
  // candidate count: the kept blocks' positions below nv (only the block
  // holding position nv - 1 can be cut short, and it is listed last)
  int ncv = nkept * static_cast<int>(bs);
  if (nkept > 0 && static_cast<int>(blist[nkept - 1]) == nbv - 1) ncv -= nbv * static_cast<int>(bs) - nv;
  ncv = min(ncv, E * NT);
  const int nslots = (ncv + NT - 1) / NT;                   // slots holding a candidate of some thread
  const float *row = scores + static_cast<int64_t>(t) * ld;
  uint32_t key[E];
#pragma unroll
  for (int e = 0; e < E; ++e) key[e] = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (e >= nslots) break;
    const int c = NT * e + tid;
    if (c < ncv) {
      const uint32_t kb = fast_div(static_cast<uint32_t>(c), dbs);
      const int pos = static_cast<int>(blist[kb] * bs + (static_cast<uint32_t>(c) - kb * bs));
      key[e] = __float_as_uint(row[pos]);
    }
  }
  auto pos_of = [&](int c) -> int {
    const uint32_t kb = fast_div(static_cast<uint32_t>(c), dbs);
    return static_cast<int>(blist[kb] * bs + (static_cast<uint32_t>(c) - kb * bs));
  };
  // keys, the candidates' range, and how many score above -inf
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u, nf = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (e >= nslots) break;
    if (NT * e + tid < ncv) {
      key[e] = ordered_key(__uint_as_float(key[e]));
      kmin = min(kmin, key[e]);
      kmax = max(kmax, key[e]);
      nf += key[e] > kNegInfKey;
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  nf = __reduce_add_sync(0xffffffffu, nf);
  if (lane == 0) {
    wred[0][warp] = kmin;
    wred[1][warp] = kmax;
    wred[2][warp] = nf;
  }
  __syncthreads();
  kmin = __reduce_min_sync(0xffffffffu, lane < kWarps ? wred[0][lane] : 0xFFFFFFFFu);
  kmax = __reduce_max_sync(0xffffffffu, lane < kWarps ? wred[1][lane] : 0u);
  const uint32_t nfin = __reduce_add_sync(0xffffffffu, lane < kWarps ? wred[2][lane] : 0u);
  uint32_t need_eq;
  if (nfin < static_cast<uint32_t>(K)) {
    // the k-th value is -inf: candidates above it are picks; the rest come,
    // lowest position first, from the candidates at -inf and the visible
    // positions outside the kept blocks
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (e >= nslots) break;
      const int c = NT * e + tid;
      if (c < ncv) {
        const int p = pos_of(c);
        atomicOr(key[e] > kNegInfKey ? &sel_gt[p >> 5] : &sel_eq[p >> 5], 1u << (p & 31));
      }
    }
    const int nwp = (nv + 31) >> 5;  // words of visible positions
    for (int w = tid; w < nwp; w += NT) {
      uint32_t outside = 0u;
      for (int b = 0; b < 32; ++b) {
        const int p = 32 * w + b;
        if (p < nv) {
          const uint32_t blk = fast_div(static_cast<uint32_t>(p), dbs);
          if (!((cwords[blk >> 5] >> (blk & 31)) & 1u)) outside |= 1u << b;
        }
      }
      atomicOr(&sel_eq[w], outside);
    }
    __syncthreads();
    need_eq = static_cast<uint32_t>(K) - nfin;
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (e >= nslots) break;
      key[e] = NT * e + tid < ncv ? key[e] - kmin : 0u;
    }
    const int L = kmax > kmin ? 32 - __clz(kmax - kmin) : 0;
    int remaining = K, hi = L;
    uint32_t thr = 0u, in_bin = 0u;
    if (hi > 0) {
      const int nb = hi < kDigitBits ? hi : kDigitBits, shift = hi - nb;
      thr = radix_pass<E, NT, true, true>(key, 0u, 0u, shift, 1 << nb, hist, rs, remaining, in_bin, nslots) << shift;
      hi = shift;
    }
    while (hi > 0 && in_bin > static_cast<uint32_t>(kFinish)) {
      const int nb = hi < kDigitBits ? hi : kDigitBits, shift = hi - nb;
      const uint32_t mask = ~((1u << hi) - 1u);
      thr |= radix_pass<E, NT, false, true>(key, thr, mask, shift, 1 << nb, hist, rs, remaining, in_bin, nslots)
             << shift;
      hi = shift;
    }
    if (hi > 0) {
      // the chosen bin's keys (at most kFinish) are gathered with their
      // positions and rank themselves; keys above the bin are picks
      const uint32_t fixed = ~((1u << hi) - 1u);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (e >= nslots) break;
        const int c = NT * e + tid;
        const uint32_t kf = key[e] & fixed;
        if (c < ncv) {
          if (kf > thr) {
            const int p = pos_of(c);
            atomicOr(&sel_gt[p >> 5], 1u << (p & 31));
          } else if (kf == thr) {
            const uint32_t i = atomicAdd(&rs.ncand, 1u);
            rs.cand[i] = key[e];
            rs.cpos[i] = pos_of(c);
          }
        }
      }
      __syncthreads();
      const uint32_t n = rs.ncand, rem2 = static_cast<uint32_t>(remaining);
      if (static_cast<uint32_t>(tid) < n) {
        const uint32_t v = rs.cand[tid];
        uint32_t gt = 0, ge = 0;
        for (uint32_t j = 0; j < n; ++j) {
          const uint32_t u = rs.cand[j];
          gt += u > v;
          ge += u >= v;
        }
        const int p = rs.cpos[tid];
        if (ge < rem2)
          atomicOr(&sel_gt[p >> 5], 1u << (p & 31));
        else if (gt < rem2) {
          atomicOr(&sel_eq[p >> 5], 1u << (p & 31));
          rs.fin_above = gt;  // the same from every candidate equal to the k-th key
        }
      }
      __syncthreads();
      need_eq = rem2 - rs.fin_above;
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (e >= nslots) break;
        const int c = NT * e + tid;
        if (c < ncv && key[e] >= thr) {
          const int p = pos_of(c);
          atomicOr(key[e] > thr ? &sel_gt[p >> 5] : &sel_eq[p >> 5], 1u << (p & 31));
        }
      }
      __syncthreads();
      need_eq = static_cast<uint32_t>(remaining);
    }
  }

  // thread i writes the picks among its words of 32 positions, in order
  uint32_t ng = 0, ne = 0;
#pragma unroll
  for (int w = 0; w < kWordsPerThread; ++w) {
    const int wi = kWordsPerThread * tid + w;
    if (wi < kWords) {
      ng += __popc(sel_gt[wi]);
      ne += __popc(sel_eq[wi]);
    }
  }
  uint32_t tot;
  const uint32_t pre = block_excl_scan((ng << 16) | ne, rs.warp_sums, &tot);
  uint32_t eq_seen = pre & 0xFFFFu;
  uint32_t o = (pre >> 16) + min(eq_seen, need_eq);
#pragma unroll
  for (int w = 0; w < kWordsPerThread; ++w) {
    const int wi = kWordsPerThread * tid + w;
    if (wi >= kWords) break;
    uint32_t take = sel_gt[wi], x = sel_eq[wi];
    for (; x != 0u && eq_seen < need_eq; ++eq_seen) {
      take |= x & (0u - x);
      x &= x - 1u;
    }
    eq_seen += __popc(x);
    while (take != 0u) {
      const int bit = __ffs(take) - 1;
      if (o < static_cast<uint32_t>(K)) out[o] = 32 * wi + bit;
      ++o;
      take &= take - 1u;
    }
  }
}

using RegKern = void (*)(const float *, int64_t, int, int, int, const int32_t *, const int32_t *, int, int32_t *,
                         uint32_t *, const uint32_t *, int, FastDiv);

template <bool kCand>
RegKern pick_reg_kernel(int N_c, bool many_rows) {
  constexpr int kE = kRegMax / 1024;  // 32 keys per thread at most with 1024 threads
  if (many_rows)
    return N_c <= kRegMax / 4 ? topk_reg_kernel<kE / 2, 512, kCand>
         : N_c <= kRegMax / 2 ? topk_reg_kernel<kE, 512, kCand>
                              : topk_reg_kernel<2 * kE, 512, kCand>;
  return N_c <= kRegMax / 4 ? topk_reg_kernel<kE / 4, 1024, kCand>
       : N_c <= kRegMax / 2 ? topk_reg_kernel<kE / 2, 1024, kCand>
                            : topk_reg_kernel<kE, 1024, kCand>;
}

template <int Dummy = 0>
RegKern pick_cand_kernel(int N_c, bool many_rows) {
  constexpr int kE = kRegMax / 1024;
  if (many_rows)
    return N_c <= kRegMax / 4 ? topk_cand_kernel<kE / 2, 512>
         : N_c <= kRegMax / 2 ? topk_cand_kernel<kE, 512>
                              : topk_cand_kernel<2 * kE, 512>;
  return N_c <= kRegMax / 4 ? topk_cand_kernel<kE / 4, 1024>
       : N_c <= kRegMax / 2 ? topk_cand_kernel<kE / 2, 1024>
                            : topk_cand_kernel<kE, 1024>;
}

}  // namespace

cudaError_t launch_topk(const float *scores, int64_t ld, const sa_index_args &ia, int K,
                        int32_t *idx, uint32_t *status, cudaStream_t stream, const uint32_t *cand,
                        int cand_words, int block_size, bool programmatic) {
  if (ia.T == 0 || K == 0) return cudaSuccess;
  const FastDiv dbs = make_fastdiv(static_cast<uint32_t>(block_size));
  // a row holds at most N_c visible scores
  if (ia.N_c > kRegMax)
    return launch_ex(programmatic, topk_radix_kernel, dim3(ia.T), dim3(kTopkThreads), 0, stream, 1, scores, ld, ia.B,
                     ia.N_c, ia.r, ia.q_seq, ia.q_pos, K, idx, status, cand, cand_words, dbs);
  const bool many_rows = ia.T > 2 * sm_count();
  // level two: blocks of kCompactMinBlock positions or more are compacted
  // (the selection runs over the kept positions), smaller ones masked in place
  const RegKern kern = !cand ? pick_reg_kernel<false>(ia.N_c, many_rows)
                       : block_size >= kCompactMinBlock ? pick_cand_kernel(ia.N_c, many_rows)
                                                        : pick_reg_kernel<true>(ia.N_c, many_rows);
  // programmatic (after the scoring kernel of the fused step): the CTAs take
  // SMs as the scoring kernel's CTAs finish (they all started before any of
  // these can) and wait for it before reading the scores
  return launch_ex(programmatic, kern, dim3(ia.T), dim3(many_rows ? 512 : 1024), 0, stream, 1, scores, ld, ia.B, ia.N_c, ia.r,
                   ia.q_seq, ia.q_pos, K, idx, status, cand, cand_words, dbs);
}

}  // namespace sa
