// Index scores on the 5th-generation tensor cores (tcgen05), for fp8-e4m3
// keys of dim 128 ("DeepSeek-V3.2-Exp inference/model.py", Indexer.forward /
// fp8_index: fp8 k_cache with one fp32 scale per position;
// "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Indexer.forward: einsum,
// relu_(), times weights, sum over heads).
//
// Per key tile of 128 positions the tensor core forms D[key, head] =
// sum_d k[key, d] * q[head, d] (M = 128 keys, N = H_I heads, K = 128) with
// e4m3 operands and an fp32 accumulator in tensor memory; the epilogue applies
// ReLU, the head weights and the key scale.
//
// Queries that are bf16 are split exactly into two e4m3 pieces per head:
// with a power-of-two head scale 2^e (max|q_h| 2^-e in (224, 448]),
// q 2^-e = p1 + p2 where p1 = e4m3(q 2^-e) and p2 = e4m3(q 2^-e - p1).  Every
// element within 2^-10.8 of the head's largest is represented exactly (its
// 8 significant bits split 4 + 4); smaller ones carry an error below
// 2^-10 * 2^e, i.e. below 2^-18.8 of the head's largest element.  Both pieces
// accumulate into the same tensor-memory columns (two passes of K = 128), so
// D = q 2^-e . k, and 2^e moves into the head weight.  fp8 queries need one
// piece.  The products of e4m3 values are exact and the tensor core
// accumulates them in fp32.
//
// The main kernel is persistent: every CTA takes a contiguous range of the
// flattened (token, key tile) list, and four roles run as warps:
//   warp 0     TMA producer: key tiles (6-stage ring) and each token's packed
//              queries and weights (double buffered);
//   warp 1     MMA issuer (one thread) and tensor-memory owner;
//   warps 2-5  epilogue: tensor memory -> registers -> score.
// Every wait is bounded (about a second); on expiry the kernel flags the
// workspace status word and drains its in-flight copies and MMAs before it
// returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace sa {
namespace {

using namespace umma;

constexpr int kTileKeys = 128;                   // M
constexpr int kAccStages = 4;
constexpr int kKeyTileBytes = kTileKeys * 128;   // 128 keys x 128 fp8
constexpr int kMaxStages = 8;                    // key-tile ring depth, as far as shared memory allows

// Two CTAs share an SM when their tensor memory fits (kAccStages * NH columns
// each): one CTA's MMA and epilogue latency then overlaps the other's copies.
template <int NH>
constexpr int kCtasPerSm = kAccStages * NH <= 256 ? 2 : 1;
// Shared memory a CTA may lay out (less the 1 KB the driver reserves per CTA
// and the 1 KB alignment slack): 228 KB per SM, 227 KB per CTA.
template <int NH>
constexpr size_t kSmemBudget = kCtasPerSm<NH> == 2 ? 233472 / 2 - 2048 : 232448 - 1024;
constexpr int kMainThreads = 224;
constexpr int kPrepThreads = 256;

// Work split of the main kernel.  The first part of the flattened (token, key
// tile) list is cut into one contiguous range per CTA; the rest is a pool that
// CTAs claim one chunk at a time from a global counter once their own work
// runs low, so CTAs on SMs that stream slower than others end up with fewer
// tiles and all finish together.  The pool goes out in chunks of kPoolChunk
// tiles (a chunk that starts a token reloads its queries, so smaller chunks
// cost more than their finer finish saves), except its last kTailPerCta tiles
// per CTA, which go in chunks of kTailChunk so that the CTAs finish closer
// together (c2 step 61.8 -> 61.0 us; single tiles there cost more than they
// saved).
constexpr int kPoolChunk = 4;
constexpr int kTailPerCta = 2, kTailChunk = 2;
constexpr int kClaimAhead = 4;  // claim when at most this many queued tiles are left to issue
constexpr int kSegQ = 4;        // segments queued between the scheduler and the producer warp
__device__ __forceinline__ int static_tiles(int total) {
  return total - static_cast<int>(total / 4);
}
// Tiles [first, end) of pool chunk c (first >= total: the pool is exhausted)
// for a grid of `ctas` CTAs.
struct PoolChunk {
  int first, end;
};
__device__ __forceinline__ PoolChunk pool_chunk(int total, int c, int ctas) {
  const int S = static_tiles(total), P = total - S;
  const int tail = min(P, kTailPerCta * ctas);
  const int n_big = (P - tail) / kPoolChunk;
  if (c < n_big) return {S + c * kPoolChunk, S + (c + 1) * kPoolChunk};
  const int f = S + n_big * kPoolChunk + (c - n_big) * kTailChunk;
  return {f, min(total, f + kTailChunk)};
}

template <int NH, int P>
struct ScoreSmem {
  static constexpr int kQBytes = P * NH * 128;
  static constexpr int kInfoMax = kMaxStages + kAccStages;
  // everything but the key ring: two query buffers, two weight vectors, the
  // tile records and their key scales, the segment queue, barriers (at most
  // 2 * kMaxStages + 13 + 2 * kSegQ of them) and the misc words
  static constexpr size_t kFixed = 2 * static_cast<size_t>(kQBytes) + 2 * NH * sizeof(float) +
                                   kInfoMax * (kTileKeys * sizeof(float) + 16) + kSegQ * 32 +
                                   (2 * kMaxStages + 13 + 2 * kSegQ) * sizeof(uint64_t) + 128 + 8;
  static constexpr int kStages = static_cast<int>(
      (kSmemBudget<NH> - kFixed) / kKeyTileBytes < kMaxStages ? (kSmemBudget<NH> - kFixed) / kKeyTileBytes
                                                                : kMaxStages);
  // tile records live until the epilogue has read them: the producer reuses
  // record n % kInfo for tile n only after the MMA of tile n + kAccStages - kInfo
  // freed its smem stage, and that MMA waited for the epilogue to release tile n - kInfo
  static constexpr int kInfo = kStages + kAccStages;
  static constexpr size_t keys = 0;
  static constexpr size_t qbuf = keys + static_cast<size_t>(kStages) * kKeyTileBytes;
  static constexpr size_t wq = qbuf + 2 * static_cast<size_t>(kQBytes);
  static constexpr size_t ksc = wq + 2 * NH * sizeof(float);
  static constexpr size_t info = ksc + static_cast<size_t>(kInfo) * kTileKeys * sizeof(float);
  static constexpr size_t seg = info + static_cast<size_t>(kInfo) * 16;
  static constexpr size_t bars = seg + kSegQ * 32;
  static constexpr int kBars = 2 * kStages + 4 + 2 * kAccStages + 1 + 2 * kSegQ;
  static constexpr size_t misc = bars + kBars * sizeof(uint64_t);
  // tmem base, abort flag, tiles issued; plan words at misc + 64
  static constexpr size_t total = misc + 128;
  static_assert(total <= kSmemBudget<NH>, "shared memory budget");
  static_assert(kInfo <= kInfoMax, "tile records");
};

// ---------------------------------------------------------------- prep ----

// Key tiles of a token of sequence b at position pos (0 for an invalid token).
__device__ __forceinline__ int tiles_of(int B, int N_c, int r, int b, int pos) {
  if (b < 0 || b >= B || pos < 0) return 0;
  const int nv = min(n_vis_of(pos, r), N_c);
  return (nv + kTileKeys - 1) / kTileKeys;
}

// Block-wide inclusive scan (kPrepThreads threads) of one int per thread.
__device__ __forceinline__ int plan_block_scan(int v, int *warp_sums) {
  constexpr int kWarps = kPrepThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_sums[lane] : 0, wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) warp_sums[lane] = wi - w;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl;
  __syncthreads();
  return r;
}

// Blocks 0..T-1: pack token t's index queries into the K-major
// 128-byte-swizzled layout the MMA reads (piece p, head h at rows p*H_I + h),
// write the folded head weights wq[t, h] = w * q_scale * 2^e, and (optionally)
// -inf into the masked tail of the score row.
// Block T: prefix[t] = key tiles of the tokens before t (prefix[T] = all
// tiles), which the main kernel reads when a CTA crosses into a later token
// (each CTA computes its own starting point from the inputs), and resets the
// main kernel's pool counter.
template <int NH, bool QFP8>
__global__ void __launch_bounds__(kPrepThreads)
idx_qprep_kernel(int B, int T, int N_c, int r, const int32_t *__restrict__ q_seq,
                 const int32_t *__restrict__ q_pos, const void *__restrict__ q_I,
                 const float *__restrict__ q_scale, const float *__restrict__ w,
                 uint8_t *__restrict__ qpack, float *__restrict__ wq, float *__restrict__ scores,
                 int64_t ld, int write_masked, int32_t *__restrict__ prefix, int *__restrict__ pool,
                 uint32_t *status) {
  constexpr int P = QFP8 ? 1 : 2;
  constexpr int kHeadsPerWarp = NH / (kPrepThreads / 32);
  pdl_trigger();
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (t == T) {
    // (no large shared array: prep blocks must fit beside the main kernel's
    // CTAs, which start early and fill the SMs' shared memory)
    __shared__ int warp_sums[32];
    if (threadIdx.x == 0) *pool = 0;  // no pool chunk handed out yet
    if (T <= 4 * kPrepThreads) {
      // up to four tokens per thread, in order: the counts stay in registers
      // (one round trip for the inputs, one block scan)
      const int base = 4 * static_cast<int>(threadIdx.x);
      int sq[4], ps[4], cnt[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int tt = min(base + k, T - 1);
        sq[k] = q_seq[tt];
        ps[k] = q_pos[tt];
      }
      int sum = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cnt[k] = base + k < T ? tiles_of(B, N_c, r, sq[k], ps[k]) : 0;
        sum += cnt[k];
      }
      const int incl = plan_block_scan(sum, warp_sums);
      int run = incl - sum;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (base + k < T) {
          prefix[base + k] = run;
          run += cnt[k];
        }
      if (threadIdx.x == kPrepThreads - 1) prefix[T] = incl;
      return;
    }
    int *cnt_s = prefix;  // tile counts, then their prefix, staged in global memory
    // (a) tile count of every token, one token per thread, coalesced, four loads in flight
    for (int t0 = threadIdx.x; t0 < T; t0 += 4 * kPrepThreads) {
      int sq[4], ps[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int tt = min(t0 + k * kPrepThreads, T - 1);
        sq[k] = q_seq[tt];
        ps[k] = q_pos[tt];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (t0 + k * kPrepThreads < T) cnt_s[t0 + k * kPrepThreads] = tiles_of(B, N_c, r, sq[k], ps[k]);
    }
    __syncthreads();
    // (b) exclusive prefix: each thread scans a contiguous chunk
    const int chunk = (T + kPrepThreads - 1) / kPrepThreads;
    const int c0 = min(T, static_cast<int>(threadIdx.x) * chunk), c1 = min(T, c0 + chunk);
    int sum = 0;
    for (int base = c0; base < c1; base += 8) {  // eight loads in flight per round
      int v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = cnt_s[min(base + k, c1 - 1)];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (base + k < c1) sum += v[k];
    }
    const int incl = plan_block_scan(sum, warp_sums);
    int run = incl - sum;
    for (int base = c0; base < c1; base += 8) {
      int v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = cnt_s[min(base + k, c1 - 1)];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (base + k < c1) {
          cnt_s[base + k] = run;
          run += v[k];
        }
    }
    __shared__ int carry;
    if (threadIdx.x == kPrepThreads - 1) carry = incl;
    __syncthreads();
    if (threadIdx.x == 0) prefix[T] = carry;
    return;
  }

  uint8_t *dst = qpack + static_cast<size_t>(t) * P * NH * 128;
  // every global load first (one round trip): lane i < kHeadsPerWarp holds the
  // weight and query scale of the warp's head i
  float w_pre = 0.f, qs_pre = 1.f;
  if (lane < kHeadsPerWarp) {
    const int64_t hi = static_cast<int64_t>(t) * NH + warp + (kPrepThreads / 32) * lane;
    w_pre = w[hi];
    if (q_scale) qs_pre = q_scale[hi];
  }
  if (QFP8) {
    uint32_t v[kHeadsPerWarp];
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
      const int h = warp + (kPrepThreads / 32) * i;
      v[i] = reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(q_I) +
                                                (static_cast<int64_t>(t) * NH + h) * 128)[lane];
    }
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
      const int h = warp + (kPrepThreads / 32) * i;
      *reinterpret_cast<uint32_t *>(dst + umma::sw128_offset(h, 4 * lane)) = v[i];
      const float wh = __shfl_sync(0xffffffffu, w_pre, i), qh = __shfl_sync(0xffffffffu, qs_pre, i);
      if (lane == 0) wq[static_cast<int64_t>(t) * NH + h] = wh * qh;
    }
  } else {
    uint2 raw[kHeadsPerWarp];
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
      const int h = warp + (kPrepThreads / 32) * i;
      raw[i] = reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(q_I) +
                                               (static_cast<int64_t>(t) * NH + h) * 128)[lane];
    }
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
      const int h = warp + (kPrepThreads / 32) * i;
      const float x[4] = {__uint_as_float(raw[i].x << 16), __uint_as_float(raw[i].x & 0xFFFF0000u),
                          __uint_as_float(raw[i].y << 16), __uint_as_float(raw[i].y & 0xFFFF0000u)};
      float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // e such that amax 2^-e is in (224, 448]: for a normal amax = 1.f 2^E,
      // e = E - 8, plus one when 1.f > 1.75 (so the scaled max is <= 448)
      int e = 0;
      const uint32_t abits = __float_as_uint(amax), ebits = abits >> 23;
      if (amax > 0.f) {
        if (ebits != 0u && ebits != 0xFFu) {
          e = static_cast<int>(ebits) - 135 + ((abits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
        } else {
          int ex;
          frexpf(amax, &ex);  // amax = m 2^ex, m in [0.5, 1)
          e = ex - 9;         // amax 2^-e in [256, 512)
          if (ldexpf(amax, -e) > 448.f) ++e;
        }
      }
      // 2^-e as a normal float when it is one (an exact scaling, as ldexpf)
      const bool pow2_ok = e >= -126 && e <= 126;
      const float inv2e = __uint_as_float(static_cast<uint32_t>(pow2_ok ? 127 - e : 127) << 23);
      uint32_t w1 = 0, w2 = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float y = pow2_ok ? x[k] * inv2e : ldexpf(x[k], -e);
        const __nv_fp8_storage_t p1 = __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
        const float rest = y - e4m3_bits_to_float(p1);
        const __nv_fp8_storage_t p2 = __nv_cvt_float_to_fp8(rest, __NV_SATFINITE, __NV_E4M3);
        w1 |= static_cast<uint32_t>(p1) << (8 * k);
        w2 |= static_cast<uint32_t>(p2) << (8 * k);
      }
      *reinterpret_cast<uint32_t *>(dst + umma::sw128_offset(h, 4 * lane)) = w1;
      *reinterpret_cast<uint32_t *>(dst + NH * 128 + umma::sw128_offset(h, 4 * lane)) = w2;
      const float wh = __shfl_sync(0xffffffffu, w_pre, i), qh = __shfl_sync(0xffffffffu, qs_pre, i);
      if (lane == 0) {
        const float f = wh * qh;
        wq[static_cast<int64_t>(t) * NH + h] =
            pow2_ok ? f * __uint_as_float(static_cast<uint32_t>(127 + e) << 23) : ldexpf(f, e);
      }
    }
  }
  if (write_masked) {
    Token tk;
    const bool ok = load_token(q_seq, q_pos, t, B, N_c, r, status, tk, threadIdx.x == 0);
    const int nv = ok ? tk.nv : 0;
    float *row = scores + static_cast<int64_t>(t) * ld;
    for (int s2 = nv + threadIdx.x; s2 < N_c; s2 += kPrepThreads) row[s2] = -INFINITY;
  }
}

// --------------------------------------------------------------- main -----

struct ScoreParams {
  int B, T, N_c, r;
  int kseq;  // key rows between consecutive sequences (k_I and k_scale)
  const int32_t *q_seq, *q_pos;
  const int32_t *prefix;  // tiles before each token, written by the prep kernel
  const uint8_t *qpack;
  const float *wq;
  const float *k_scale;
  float *scores;
  int64_t ld;
  uint32_t *status;
  int *pool;        // pool chunks claimed so far (zeroed by the prep kernel)
  int evict_first;  // nonzero: key rows are read once per call (at most one token per sequence)
};

template <int NH, int P>
__global__ void __launch_bounds__(kMainThreads, kCtasPerSm<NH>)
idx_score_umma_kernel(const __grid_constant__ CUtensorMap kmap, const ScoreParams p) {
  using L = ScoreSmem<NH, P>;
  constexpr int kQBytes = L::kQBytes;
  constexpr int kStages = L::kStages;
  constexpr int kInfo = L::kInfo;
  constexpr uint32_t kTmemCols = kAccStages * NH;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the swizzle atoms need 1024-byte alignment: align the base explicitly
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *keys = smem + L::keys;
  uint8_t *qbuf = smem + L::qbuf;
  float *wqs = reinterpret_cast<float *>(smem + L::wq);
  float *ksc = reinterpret_cast<float *>(smem + L::ksc);  // [kInfo][128] key scales of a tile
  int4 *info = reinterpret_cast<int4 *>(smem + L::info);  // [kInfo] {token (-1: end), first position, n_vis, query buffer}
  int *segq = reinterpret_cast<int *>(smem + L::seg);     // [kSegQ][8] {tile, end tile, token, first tile, b, n_vis}
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *kfull = bars, *kempty = bars + kStages;
  uint64_t *qfull = bars + 2 * kStages, *qempty = qfull + 2;
  uint64_t *afull = qempty + 2, *aempty = afull + kAccStages;
  uint64_t *done = aempty + kAccStages;
  uint64_t *segfull = done + 1, *segempty = segfull + kSegQ;
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem + L::misc);
  int *abort_s = reinterpret_cast<int *>(smem + L::misc + 8);
  int *issued_s = reinterpret_cast<int *>(smem + L::misc + 16);  // key tiles the producer has issued

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();

  // The tile plan below starts from every token's sequence and position.
  // Their loads go out first, so that their latency (the first touch of
  // these inputs in the step) overlaps the set-up; each thread keeps the
  // first eight tokens of its chunk in registers.
  constexpr int kW = kMainThreads / 32;
  const int chunk = (p.T + kMainThreads - 1) / kMainThreads;
  const int c0 = min(p.T, tid * chunk), c1 = min(p.T, c0 + chunk);
  int sq[8], ps[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int tt = min(c0 + k, p.T - 1);
    sq[k] = p.q_seq[tt];
    ps[k] = p.q_pos[tt];
  }

  // ---- set-up: barriers, tensor memory
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kfull[i], 1 + 32);  // the key tile's copy (with its record) + the 32 key-scale copies
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1 + 4);  // MMA commit + four epilogue warps
    }
    for (int i = 0; i < kAccStages; ++i) {
      mbar_init(&afull[i], 2);  // MMA commit + the issuing lane, which passes the tile record on
      mbar_init(&aempty[i], 4);
    }
    mbar_init(done, 1);
    for (int i = 0; i < kSegQ; ++i) {
      mbar_init(&segfull[i], 1);
      mbar_init(&segempty[i], 1);
    }
    *abort_s = 0;
    *issued_s = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_s, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;

  // This CTA's own tile range and its first token, from the inputs alone (the
  // prep kernel's prefix is the same plan; the scheduler reads it for later
  // tokens), so key tiles can stream before the prep kernel ends.
  int *plan_s = reinterpret_cast<int *>(smem + L::misc + 64);  // [8]
  {
    int *wsum_s = plan_s + 8;  // [kW + 1]
    int sum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (c0 + k < c1) sum += tiles_of(p.B, p.N_c, p.r, sq[k], ps[k]);
    for (int base = c0 + 8; base < c1; base += 8) {  // longer chunks: eight loads in flight per round
      int sq2[8], ps2[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int tt = min(base + k, c1 - 1);
        sq2[k] = p.q_seq[tt];
        ps2[k] = p.q_pos[tt];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (base + k < c1) sum += tiles_of(p.B, p.N_c, p.r, sq2[k], ps2[k]);
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum_s[warp] = incl;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int w2 = 0; w2 < kW; ++w2) {
        const int v = wsum_s[w2];
        wsum_s[w2] = run;
        run += v;
      }
      wsum_s[kW] = run;
    }
    __syncthreads();
    const int pre = wsum_s[warp] + incl - sum, total = wsum_s[kW];
    const int S = static_tiles(total);
    const int begin0 = static_cast<int>(static_cast<long long>(S) * blockIdx.x / gridDim.x);
    const int end0 = static_cast<int>(static_cast<long long>(S) * (blockIdx.x + 1) / gridDim.x);
    if (tid == 0) {
      plan_s[0] = begin0;
      plan_s[1] = end0;
      plan_s[7] = total;
    }
    if (begin0 < end0 && pre <= begin0 && begin0 < pre + sum) {  // this chunk holds tile begin0
      int run = pre, tt = c0, b = 0, pos = 0, tl = 0;
      bool found = false;
#pragma unroll
      for (int k = 0; k < 8; ++k)  // the first eight tokens from registers
        if (!found && c0 + k < c1) {
          tt = c0 + k;
          b = sq[k];
          pos = ps[k];
          tl = tiles_of(p.B, p.N_c, p.r, b, pos);
          found = begin0 < run + tl;
          if (!found) run += tl;
        }
      for (int t2 = c0 + 8; !found && t2 < c1; ++t2) {  // the rest reloaded
        tt = t2;
        b = p.q_seq[t2];
        pos = p.q_pos[t2];
        tl = tiles_of(p.B, p.N_c, p.r, b, pos);
        found = begin0 < run + tl;
        if (!found) run += tl;
      }
      if (found) {
        plan_s[2] = tt;
        plan_s[3] = run;
        plan_s[4] = run + tl;
        plan_s[5] = b;
        plan_s[6] = min(n_vis_of(pos, p.r), p.N_c);
      }
    }
    __syncthreads();
  }
  const int begin = plan_s[0], end = plan_s[1], total = plan_s[7];
  // the first token of the own range (meaningful only when begin < end)
  const int t0 = plan_s[2], first0 = plan_s[3], next0 = plan_s[4], b0 = plan_s[5], nv0 = plan_s[6];
  auto fail = [&]() {
    raise_flag(p.status, kFlagTimeout);
    atomicExch(abort_s, 1);
  };
  auto aborted = [&]() { return __any_sync(0xffffffffu, *(volatile int *)abort_s != 0); };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    // The whole warp walks its tiles segment by segment (a run of tiles of
    // one token): lane 0 writes the tile record and issues the key tile,
    // every lane copies four of the tile's 128 key scales.
    if (lane == 0) prefetch_tmap(&kmap);
    const uint64_t kpol = l2_policy(p.evict_first != 0);
    int n = 0, qn = -1, prev_t = -1, si = 0;
    bool ok = true;
    // current segment: tiles [i, i1) of token t (first tile `first`, sequence b, nv visible)
    int i = begin, i1 = begin < end ? min(end, next0) : begin;
    int t = t0, first = first0, b = b0, nv = nv0;
    auto issue = [&]() {
      const int s = n % kStages, k = n % kInfo;
      const int s0 = (i - first) * kTileKeys;
      if (lane == 0) {
        info[k] = make_int4(t, s0, nv, qn);
        mbar_expect_tx(&kfull[s], kKeyTileBytes);
        tma_load_2d_hint(keys + s * kKeyTileBytes, &kmap, &kfull[s], 0, b * p.kseq + s0, kpol);
      }
      if (p.k_scale) {
        const int pos = s0 + 4 * lane;
        const float *src = p.k_scale + static_cast<int64_t>(b) * p.kseq + pos;
        float *dst = ksc + k * kTileKeys + 4 * lane;
        if (pos + 3 < nv && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
          cp_async16(dst, src, kpol);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (pos + e < nv) cp_async4(dst + e, src + e);
        }
      }
      cp_async_mbar_arrive(&kfull[s]);
      ++n;
      ++i;
    };
    auto load_q = [&]() -> bool {  // the current token's packed queries and weights
      ++qn;
      const int qb = qn & 1;
      if (!mbar_wait_warp(&qempty[qb], ((qn >> 1) & 1) ^ 1)) return false;
      if (lane == 0) {
        mbar_expect_tx(&qfull[qb], kQBytes + NH * 4);
        bulk_load(qbuf + qb * kQBytes, p.qpack + static_cast<size_t>(t) * kQBytes, kQBytes, &qfull[qb]);
        bulk_load(wqs + qb * NH, p.wq + static_cast<size_t>(t) * NH, NH * 4, &qfull[qb]);
      }
      prev_t = t;
      return true;
    };
    // the first key tiles of the own range (up to the ring size) do not
    // depend on the prep kernel: issue them first, then wait for its queries
    const int n_pre = min(i1 - i, kStages);
    if (n_pre > 0) qn = 0;
    while (n < n_pre) issue();
    pdl_wait();
    if (n_pre > 0) {
      qn = -1;
      ok = load_q();
    }
    while (ok) {
      if (aborted()) {
        ok = false;
        break;
      }
      if (i >= i1) {  // next segment from the scheduler
        const int q = si % kSegQ;
        if (!mbar_wait_warp(&segfull[q], (si / kSegQ) & 1)) {
          ok = false;
          break;
        }
        const int *e = segq + q * 8;
        i = e[0];
        i1 = e[1];
        t = e[2];
        first = e[3];
        b = e[4];
        nv = e[5];
        __syncwarp();
        if (lane == 0) mbar_arrive(&segempty[q]);
        ++si;
        if (i < 0) break;  // no more work
        continue;
      }
      if (t != prev_t && !load_q()) {
        ok = false;
        break;
      }
      const int s = n % kStages;
      if (!mbar_wait_warp(&kempty[s], ((n / kStages) & 1) ^ 1)) {
        ok = false;
        break;
      }
      issue();
      if (lane == 0) *(volatile int *)issued_s = n;
    }
    if (ok) {  // end of work: a record with token -1, passed on by the MMA warp to the epilogue
      const int s = n % kStages;
      if (mbar_wait_warp(&kempty[s], ((n / kStages) & 1) ^ 1)) {
        if (lane == 0) {
          info[n % kInfo] = make_int4(-1, 0, 0, 0);
          mbar_arrive(&kfull[s]);
        }
        cp_async_mbar_arrive(&kfull[s]);
        ++n;
      } else {
        ok = false;
      }
    }
    if (!ok && lane == 0) fail();
    // drain: every issued copy lands before the CTA may exit
    cp_async_wait_all();
    if (lane == 0) {
      for (int m = max(0, n - kStages); m < n; ++m) mbar_wait(&kfull[m % kStages], (m / kStages) & 1);
      if (qn >= 0) mbar_wait(&qfull[qn & 1], (qn >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    // The whole warp walks the tile records and waits; one elected lane
    // issues the MMAs and commits from operands the warp computed uniformly.
    constexpr uint32_t idesc = idesc_e4m3(kTileKeys, NH);
    const bool leader = elect_one();
    int qn = -1;
    bool ok = true;
    for (int n = 0;; ++n) {
      if (aborted()) break;
      const int s = n % kStages, a = n % kAccStages;
      if (!mbar_wait_warp(&kfull[s], (n / kStages) & 1) ||
          !mbar_wait_warp(&aempty[a], ((n / kAccStages) & 1) ^ 1)) {
        ok = false;
        break;
      }
      const int4 ti = info[n % kInfo];
      if (ti.x < 0) {  // end of work: pass the record on
        if (leader) {
          mbar_arrive(&afull[a]);
          mbar_arrive(&afull[a]);
        }
        break;
      }
      if (ti.w != qn) {
        if (qn >= 0 && leader) mma_commit(&qempty[qn & 1]);
        qn = ti.w;
        if (!mbar_wait_warp(&qfull[qn & 1], (qn >> 1) & 1)) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      const uint32_t d = tmem + a * NH;
      const uint32_t a0 = smem_u32(keys + s * kKeyTileBytes);
      const uint32_t b0 = smem_u32(qbuf + (qn & 1) * kQBytes);
      if (leader) {
#pragma unroll
        for (int pc = 0; pc < P; ++pc)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8f6f4(d, desc_sw128_kmajor(a0 + 32 * k), desc_sw128_kmajor(b0 + pc * NH * 128 + 32 * k),
                       idesc, (pc | k) != 0);
        mma_commit(&kempty[s]);
        mma_commit(&afull[a]);
        mbar_arrive(&afull[a]);  // releases the tile record and key scales the epilogue reads
      }
      __syncwarp();
    }
    if (!ok && lane == 0) fail();
    if (leader) {
      if (qn >= 0) mma_commit(&qempty[qn & 1]);
      mma_commit(done);
      if (!mbar_wait(done, 0)) raise_flag(p.status, kFlagTimeout);
    }
    __syncwarp();
  } else if (warp < 6) {
    // --------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int qn = -1;
    for (int n = 0;; ++n) {
      if (aborted()) break;
      const int a = n % kAccStages, k = n % kInfo;
      if (!mbar_wait_warp(&afull[a], (n / kAccStages) & 1)) {
        if (lane == 0) fail();
        break;
      }
      const int4 ti = info[k];
      if (ti.x < 0) break;
      if (ti.w != qn) {
        if (qn >= 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&qempty[qn & 1]);
        }
        qn = ti.w;
        if (!mbar_wait_warp(&qfull[qn & 1], (qn >> 1) & 1)) {
          if (lane == 0) fail();
          break;
        }
      }
      tc_fence_after();
      uint32_t v[NH];
#pragma unroll
      for (int c = 0; c < NH / 32; ++c)
        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * NH + 32 * c,
                           *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
      // the record and the scale are read before the stage is released (the
      // producer reuses them once the stage's next MMA has run)
      const float ks = p.k_scale ? ksc[k * kTileKeys + row] : 1.f;
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[a]);
      const int s = ti.y + row;
      if (s < ti.z) {
        // sum_h w_h relu(d_h): eight independent partial sums (short chains),
        // weights read four at a time
        const float4 *wv4 = reinterpret_cast<const float4 *>(wqs + (qn & 1) * NH);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
        for (int h4 = 0; h4 < NH / 4; ++h4) {
          const float4 w4 = wv4[h4];
          float *a2 = &acc[(h4 & 1) * 4];
          a2[0] = fmaf(w4.x, fmaxf(__uint_as_float(v[4 * h4]), 0.f), a2[0]);
          a2[1] = fmaf(w4.y, fmaxf(__uint_as_float(v[4 * h4 + 1]), 0.f), a2[1]);
          a2[2] = fmaf(w4.z, fmaxf(__uint_as_float(v[4 * h4 + 2]), 0.f), a2[2]);
          a2[3] = fmaf(w4.w, fmaxf(__uint_as_float(v[4 * h4 + 3]), 0.f), a2[3]);
        }
        const float tot = ((acc[0] + acc[4]) + (acc[1] + acc[5])) + ((acc[2] + acc[6]) + (acc[3] + acc[7]));
        p.scores[static_cast<int64_t>(ti.x) * p.ld + s] = tot * ks;
      }
    }
    if (qn >= 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qn & 1]);
    }
  } else {
    // -------------------------------------------------------- scheduler
    // Hands the producer its tiles as segments (runs of one token's tiles):
    // the rest of the own range first, then pool chunks, each claimed only
    // when the producer has at most kClaimAhead queued tiles left to issue.
    pdl_wait();  // the token prefix and the pool counter come from the prep kernel
    // token cursor: token ct holds tiles [cfirst, cnext)
    int ct = -1, cfirst = 0, cnext = 0, cb = 0, cnv = 0;
    if (begin < end) {
      ct = t0;
      cfirst = first0;
      cnext = next0;
      cb = b0;
      cnv = nv0;
    }
    int i = begin < end ? min(end, next0) : begin;
    int pushed = i - begin, si = 0;
    bool ok = true;
    // moves the cursor forward to the token holding tile `tile` (< total):
    // 32 tokens' boundaries per round, one load each
    auto seek = [&](int tile) -> bool {
      if (tile < cnext) return true;
      for (int base = ct + 1; base < p.T; base += 32) {
        const int cand = base + lane;
        const int nx = cand < p.T ? p.prefix[cand + 1] : 0x7FFFFFFF;
        const uint32_t hit = __ballot_sync(0xffffffffu, nx > tile);
        if (hit) {
          const int l = __ffs(hit) - 1;
          ct = base + l;
          if (ct >= p.T) return false;
          cnext = __shfl_sync(0xffffffffu, nx, l);
          int f = 0, bb = 0, pp = 0;
          if (lane == 0) {
            f = p.prefix[ct];
            bb = p.q_seq[ct];
            pp = p.q_pos[ct];
          }
          cfirst = __shfl_sync(0xffffffffu, f, 0);
          cb = __shfl_sync(0xffffffffu, bb, 0);
          cnv = min(n_vis_of(__shfl_sync(0xffffffffu, pp, 0), p.r), p.N_c);
          return true;
        }
      }
      return false;
    };
    auto push = [&](int i0, int i1) -> bool {
      const int q = si % kSegQ;
      if (!mbar_wait_warp(&segempty[q], ((si / kSegQ) & 1) ^ 1)) return false;
      if (lane == 0) {
        int *e = segq + q * 8;
        e[0] = i0;
        e[1] = i1;
        e[2] = ct;
        e[3] = cfirst;
        e[4] = cb;
        e[5] = cnv;
        mbar_arrive(&segfull[q]);
      }
      __syncwarp();
      ++si;
      return true;
    };
    // the rest of the own range
    while (ok && i < end) {
      const int i1 = seek(i) ? min(end, cnext) : -1;
      if (i1 < 0 || !push(i, i1)) {
        ok = false;
        break;
      }
      pushed += i1 - i;
      i = i1;
    }
    // pool chunks
    while (ok) {
      const long long w0 = clock64();
      for (;;) {  // until the producer has at most kClaimAhead queued tiles left
        int wait = 0;
        if (lane == 0)
          wait = pushed - *(volatile int *)issued_s > kClaimAhead && !*(volatile int *)abort_s &&
                 clock64() - w0 < kWaitBudgetCycles;
        if (!__shfl_sync(0xffffffffu, wait, 0)) break;
        __nanosleep(200);
      }
      if (aborted() || clock64() - w0 >= kWaitBudgetCycles) {
        ok = false;
        break;
      }
      int c = 0;
      if (lane == 0) c = atomicAdd(p.pool, 1);
      c = __shfl_sync(0xffffffffu, c, 0);
      const PoolChunk pc = pool_chunk(total, c, static_cast<int>(gridDim.x));
      if (pc.first >= total) break;  // pool exhausted
      int i0 = pc.first;
      const int ie = pc.end;
      while (i0 < ie) {
        const int i1 = seek(i0) ? min(ie, cnext) : -1;
        if (i1 < 0 || !push(i0, i1)) {
          ok = false;
          break;
        }
        pushed += i1 - i0;
        i0 = i1;
      }
    }
    if (!ok && lane == 0) fail();
    push(-1, -1);  // end of work
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host --

template <int NH, bool QFP8>
cudaError_t launch_umma_impl(const sa_index_args &ia, float *scores, int64_t ld, bool write_masked,
                             uint8_t *qpack, float *wq, int32_t *prefix, int *pool, uint32_t *status,
                             cudaStream_t stream) {
  constexpr int P = QFP8 ? 1 : 2;
  using L = ScoreSmem<NH, P>;
  const int grid = sm_count() * kCtasPerSm<NH>;
  // The prep kernel takes the largest shared-memory carveout, as the main
  // kernel does: an SM holding a prep CTA configured for less shared memory
  // could not take a main-kernel CTA until the prep CTA had left, and the main
  // kernel's CTAs start while the prep kernel runs.
  {
    static bool carveout_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 && !carveout_done[dev]) {
      cudaError_t ce = cudaFuncSetAttribute(reinterpret_cast<const void *>(idx_qprep_kernel<NH, QFP8>),
                                            cudaFuncAttributePreferredSharedMemoryCarveout,
                                            cudaSharedmemCarveoutMaxShared);
      if (ce != cudaSuccess) return ce;
      carveout_done[dev] = true;
    }
  }
  idx_qprep_kernel<NH, QFP8><<<ia.T + 1, kPrepThreads, 0, stream>>>(
      ia.B, ia.T, ia.N_c, ia.r, ia.q_seq, ia.q_pos, ia.q_I, ia.q_scale, ia.w, qpack, wq, scores, ld,
      write_masked ? 1 : 0, prefix, pool, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap kmap;
  // rows of the last sequence end at (B - 1) * kseq + N_c; a tile reaching
  // past that reads zeros (and past a token's visible rows is never used)
  const int64_t kseq = k_rows_per_seq(ia);
  if ((static_cast<int64_t>(ia.B) - 1) * kseq + ia.N_c + kTileKeys >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>((static_cast<int64_t>(ia.B) - 1) * kseq + ia.N_c)};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, kTileKeys};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ia.k_I), dims,
                       strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;

  ScoreParams sp{ia.B,  ia.T,   ia.N_c, ia.r,   static_cast<int>(kseq), ia.q_seq, ia.q_pos, prefix, qpack,
                 wq,    ia.k_scale, scores, ld, status, pool, ia.T <= ia.B ? 1 : 0};
  auto kern = idx_score_umma_kernel<NH, P>;
  const size_t smem = L::total + 1024;  // + alignment slack for the 1024-byte swizzle atoms
  static bool attr_done[64] = {};
  e = set_smem_once(reinterpret_cast<const void *>(kern), smem, attr_done);
  if (e != cudaSuccess) return e;
  // the prep kernel is short: overlapping this kernel's launch and set-up
  // with it pays
  return launch_ex(true, kern, dim3(grid), dim3(kMainThreads), smem, stream, 1, kmap, sp);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

cudaError_t set_smem_once(const void *func, size_t bytes, bool *done_per_device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done_per_device[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done_per_device[dev] = true;
  return e;
}

bool idx_score_umma_supported(const sa_index_args &ia) {
  return ia.k_dtype == SA_FP8_E4M3 && ia.D_I == 128 && (ia.H_I == 32 || ia.H_I == 64 || ia.H_I == 128);
}

namespace {
struct UmmaScratch {
  size_t qpack, wq, prefix, pool, total;
};
UmmaScratch umma_scratch_layout(const sa_index_args &ia) {
  const int P = ia.q_dtype == SA_FP8_E4M3 ? 1 : 2;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  UmmaScratch L{};
  L.qpack = 0;
  L.wq = up(static_cast<size_t>(ia.T) * P * ia.H_I * 128);
  L.prefix = L.wq + up(static_cast<size_t>(ia.T) * ia.H_I * 4);
  L.pool = L.prefix + up(static_cast<size_t>(ia.T + 1) * 4);
  L.total = L.pool + 256;
  return L;
}
}  // namespace

size_t idx_score_umma_scratch(const sa_index_args &ia) { return umma_scratch_layout(ia).total; }

cudaError_t launch_idx_score_umma(const sa_index_args &ia, float *scores, int64_t ld, bool write_masked,
                                  void *scratch, uint32_t *status, cudaStream_t stream) {
  if (ia.T == 0) return cudaSuccess;
  const UmmaScratch L = umma_scratch_layout(ia);
  uint8_t *base = static_cast<uint8_t *>(scratch);
  uint8_t *qpack = base + L.qpack;
  float *wq = reinterpret_cast<float *>(base + L.wq);
  int32_t *prefix = reinterpret_cast<int32_t *>(base + L.prefix);
  int *pool = reinterpret_cast<int *>(base + L.pool);
  const bool qf8 = ia.q_dtype == SA_FP8_E4M3;
#define SA_UMMA_CASE(NH, QF)                                                                              \
  if (ia.H_I == NH && qf8 == QF)                                                                          \
    return launch_umma_impl<NH, QF>(ia, scores, ld, write_masked, qpack, wq, prefix, pool, status, stream);
  SA_UMMA_CASE(32, false)
  SA_UMMA_CASE(32, true)
  SA_UMMA_CASE(64, false)
  SA_UMMA_CASE(64, true)
  SA_UMMA_CASE(128, false)
  SA_UMMA_CASE(128, true)
#undef SA_UMMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace sa
