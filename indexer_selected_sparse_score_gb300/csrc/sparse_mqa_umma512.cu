// Sparse MQA on the 5th-generation tensor cores (tcgen05) at the released
// V4.1 attention shape: 64 query heads of dim 512 over one kv tensor used as
// both K and V ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
// Attention.forward: sparse_attn(q, kv, attn_sink, topk_idxs, softmax_scale)
// over the window rows and the index-selected compressed rows; head_dim 512
// in the released config).
//
// O for 64 heads x 512 dims in fp32 needs 512 tensor-memory columns when the
// heads sit in the lanes, leaving none for the logits.  So every product is
// taken transposed, with the long dimension in the lanes:
//   S^T = KV Q^T   M = 128 rows of the kv tile (64 keys; the other 64 rows only
//                  feed accumulator lanes nobody reads), N = 64 heads, K = 512
//                  dims: lanes 0-63 hold the tile's keys, one column per head;
//   softmax        one thread per (key, half of the heads): all four warps of
//                  the softmax warpgroup, each over 32 heads (warps 0 and 1,
//                  which reach lanes 0-63, hand heads 32-63 over to warps 2
//                  and 3 in shared memory): p = 2^(scale s - m_ref[h]) with a
//                  lazily raised reference max per head; P^T is written to
//                  shared memory as a bf16 hi + lo pair, each thread half a
//                  row (the MN-major layout of the second product's B);
//   O^T += V^T P^T four products of M = 128 dims, N = 64 heads, K = 64 keys,
//                  hi and lo: O^T takes 4 x 64 = 256 columns, dims in lanes.
// The kv tile lands once, by TMA gather4, in the 128-byte-swizzled layout that
// is K-major for the first product (rows = keys) and MN-major for the second
// (dims contiguous along a row), so one copy serves both.  Per-head maxima
// and sums over a warp's 32 keys are one reduce-scatter (31 shuffles for 32
// heads).
//
// Warps: 0-3 the softmax warpgroup (P, and the rescale and read-out of O^T,
// whose lanes they split); 4 MMA issuer and tensor-memory owner; 5-15 copy kv
// rows (warp 5 also loads each token's Q and writes the tile's key mask).  A
// CTA takes whole tokens, or, when every token can have a 2-CTA cluster of
// its own, half of one token's tiles: the two CTAs then exchange, over
// distributed shared memory (bulk copies into the upper half of the other's
// kv ring, free once its last product is done), their per-head reference
// maxima and sums and the unnormalised O^T of the other's half of the dims;
// each merges the parts against the larger of the two maxima and writes its
// 256 dims of the output.  When every input but the indices is known to be
// complete at launch, the queries and the window rows load before the wait
// for the previous kernel.  Every wait is bounded; on expiry the kernel flags
// the status word, drains its copies and MMAs and returns, and the softmax
// warpgroup's named barriers are reached by all four warps on every path.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace sa {
namespace {

using namespace umma;

constexpr int kH = 64;            // query heads
constexpr int kD = 512;           // head dim
constexpr int kTk = 64;           // keys per tile
constexpr int kChunks = kD / 64;  // 64-dim chunks of a row (128 bytes each)
constexpr int kSlots = 2;         // kv ring slots
constexpr int kSBufs = 3;         // S^T buffers in tensor memory
constexpr int kPBufs = 2;         // P^T buffers in shared memory
constexpr int kMaskSlots = 4;
constexpr int kThreads = 512;
constexpr int kMmaWarp = 4;
constexpr int kCopyWarp0 = 5, kCopyWarps = 11;
constexpr int kCopies = kTk / 4 * kChunks;  // gather4 copies per tile: 16 groups of 4 keys x 8 chunks
constexpr float kLazyRescale = 8.f;         // log2 units
constexpr uint32_t kColS = 256;             // S^T buffer b at 256 + 64 b; O^T block mb at 64 mb
constexpr int kSSteps = kD / 16;            // k-steps of a logit product
// hand-off between the two CTAs of a split token, each way: O^T of the
// partner's two dim blocks and (m_ref, sum) per head, in bulk copies of
// kXferChunk bytes
constexpr uint32_t kXferChunk = 16384;
constexpr int kXferChunks = 65536 / kXferChunk;                // 64 KB: two dim blocks of O^T
constexpr uint32_t kXferBytes = 65536 + kH * 8;
// Registers per thread: built for 128 (512 threads); the softmax warpgroup
// raises its limit and the other three lower theirs, 192 + 3 * 104 <= 4 * 128.
constexpr int kLaunchRegs = 128, kSoftmaxRegs = 192, kOtherRegs = 104;
static_assert(kSoftmaxRegs + 3 * kOtherRegs <= 4 * kLaunchRegs, "register split exceeds the launch allocation");

struct Smem512 {
  static constexpr size_t q = 0;                               // [8 chunk][64 heads][128 B]
  static constexpr size_t kv = q + 65536;                      // [slot][8 chunk][64 keys][128 B]
  static constexpr size_t pt = kv + kSlots * 65536;            // [buf][hi, lo][64 keys][128 B]
  static constexpr size_t mask = pt + kPBufs * 16384;          // [slot][4] u32
  static constexpr size_t red = mask + kMaskSlots * 16;        // [4][32] f32: per-warp partial max / sum
  static constexpr size_t mref = red + 2 * kH * 4;             // [64] f32: reference max per head (log2 units)
  static constexpr size_t fac = mref + kH * 4;                 // [64] f32: rescale factor / output scale per head
  static constexpr size_t flags = fac + kH * 4;                // [4] i32: abort (slot 3); [2][4] votes at +16
  static constexpr size_t bars = (flags + 48 + 7) & ~size_t(7);
  static constexpr int kBars = 2 * kSlots + 2 + 2 * kSBufs + 2 * kPBufs + 1 + kMaskSlots + 1 + 2;
  static constexpr size_t misc = bars + kBars * 8;
  static constexpr size_t total = misc + 16;
};
static_assert(Smem512::total + 1024 <= 232448, "shared memory budget");

struct Attn512Params {
  int B, T, N_c, r, W, R, K;
  int WT, TPT;       // window tiles per token, tiles per token
  int split, PT0;    // CTAs per token (1, or a 2-CTA cluster with one token), tiles of rank 0's part
  int wseq, cseq;    // rows between consecutive sequences of the ring and of the compressed cache
  int evict_first;   // nonzero: rows are read once per call (at most one token per sequence)
  int early;         // nonzero: every input but idx is complete at launch, so only idx waits for the predecessor
  long long budget;  // SM cycles a pipeline wait may take before the kernel gives up (drains keep the full budget)
  const int32_t *q_seq, *q_pos, *idx;
  const float *sink;
  float qk_scale;    // scale * log2(e)
  __nv_bfloat16 *out;
  uint32_t *status;
};

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void gather4(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y0, int y1,
                                        int y2, int y3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
      "l"(policy)
      : "memory");
}

// 2^x by the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// MN-major 128-byte-swizzled operand: rows = K (8-row atoms 1024 B apart),
// 64 M or N values per row, blocks of 64 `lbo` bytes apart.
__device__ __forceinline__ uint64_t desc_sw128_mnmajor(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Reduces 32 values per lane over the warp, the result for value l landing in
// lane l: five halving rounds, in the round of offset o each lane keeps the
// half of its remaining values picked by bit o of its lane number and
// combines it with the partner lane's copy of that half (31 shuffles for all
// 32 values).  `v` is overwritten.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float keep = up ? v[i + o] : v[i];
      const float send = up ? v[i] : v[i + o];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// Named barrier of the softmax warpgroup (warps 0-3).
__device__ __forceinline__ void group_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// kShort: the waits between stages take the bound of sa_set_wait_budget (and
// the copy warps vote on stopping); otherwise the default bound, a constant
template <bool kShort>
__global__ void __launch_bounds__(kThreads, 1)
sparse_mqa_umma512_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                          const __grid_constant__ CUtensorMap cmap, const Attn512Params p) {
  using L = Smem512;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *qs = smem + L::q, *kvs = smem + L::kv, *pts = smem + L::pt;
  uint32_t *mask_s = reinterpret_cast<uint32_t *>(smem + L::mask);
  float *red_s = reinterpret_cast<float *>(smem + L::red);
  float *mref_s = reinterpret_cast<float *>(smem + L::mref);
  float *fac_s = reinterpret_cast<float *>(smem + L::fac);
  volatile int *flags_s = reinterpret_cast<volatile int *>(smem + L::flags);
  // votes of the softmax warpgroup for tile n, slot n % 2 (a warp can be at
  // most one group barrier ahead of another): bit 0 = a logit passed its
  // reference by the lazy margin, bit 1 = this warp saw a failure or an abort
  volatile int *votes_s = flags_s + 4;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *kvfull = bars, *kvempty = bars + kSlots;
  uint64_t *qfull = bars + 2 * kSlots, *qempty = qfull + 1;
  uint64_t *sfull = qempty + 1, *sempty = sfull + kSBufs;  // S^T written; S^T read (buffer free)
  // pempty[b]: the P.V product that read P^T buffer b is done.  Its phases
  // also tell the softmax when O^T holds a given tile's product: the buffer's
  // next product needs P of two tiles later, so a wait on it can never be
  // satisfied by a phase other than the one meant (a barrier of its own with
  // a phase per tile could run two phases ahead of a waiter)
  uint64_t *pfull = sempty + kSBufs, *pempty = pfull + kPBufs;
  uint64_t *oempty = pempty + kPBufs;  // O^T of the previous token read out
  uint64_t *mfull = oempty + 1;       // [kMaskSlots]
  uint64_t *done = mfull + kMaskSlots;
  // split hand-off: xempty (rank 1) = rank 0's kv ring is free to take rank
  // 1's part; xfull (rank 0) = the part is there
  uint64_t *xempty = done + 1, *xfull = xempty + 1;
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem + L::misc);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long budget = kShort ? p.budget : kWaitBudgetCycles;  // bound of a wait between stages
  // cluster c (of G) takes tokens [T c / G, T (c + 1) / G); with a 2-CTA
  // cluster (one token each), rank 0 takes tiles [0, PT0) and rank 1 the rest
  const int split = p.split;
  const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int G = gridDim.x / split, cl = blockIdx.x / split;
  const int t0 = static_cast<int>(static_cast<long long>(p.T) * cl / G);
  const int t1 = static_cast<int>(static_cast<long long>(p.T) * (cl + 1) / G);
  const int J0 = rank * p.PT0;
  const int PT = split == 1 ? p.TPT : (rank == 0 ? p.PT0 : p.TPT - p.PT0);
  const int count = (t1 - t0) * PT;  // tile n is tile J0 + n % PT of token t0 + n / PT

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&kvfull[i], kCopyWarps);
      mbar_init(&kvempty[i], 1);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, 1);
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 2);
    }
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(&pfull[i], 4);
      mbar_init(&pempty[i], 1);
    }
    mbar_init(oempty, 4);
    for (int i = 0; i < kMaskSlots; ++i) mbar_init(&mfull[i], 1);
    mbar_init(done, 1);
    mbar_init(xempty, 1);
    mbar_init(xfull, 1);
    for (int i = 0; i < 12; ++i) flags_s[i] = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_base_s, 512);
    tmem_relinquish();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  if (split > 1) cluster_sync();  // the partner's barriers are initialised before any remote arrival
  tc_fence_after();
  // The selected indices come from the previous kernel.  When every other
  // input is known complete at launch, only the reads of idx wait for it, so
  // the queries and the window rows load while the previous kernel finishes.
  if (!p.early) pdl_wait();
  const uint32_t tmem = *tmem_base_s;
  auto fail = [&]() {
    raise_flag(p.status, kFlagTimeout);
    flags_s[3] = 1;
  };
  auto aborted = [&]() { return flags_s[3] != 0; };

  if (warp >= 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp >= kCopyWarp0) {
      // ------------------------------------------------------------ copy warps
      const int pw = warp - kCopyWarp0;
      const uint64_t rpol = l2_policy(p.evict_first != 0);
      if (count > 0) {
        if (warp == kCopyWarp0 && lane == 0) {
          prefetch_tmap(&qmap);
          prefetch_tmap(&wmap);
          prefetch_tmap(&cmap);
        }
        // rows of absent keys are multiplied by P = 0 but must be finite: an
        // absent key of a copied group holds a present key's row, and a group
        // with no present key is not copied and keeps what the slot held
        // before, so the ring starts zeroed
        for (int i = pw * 32 + lane; i < kSlots * 65536 / 16; i += 32 * kCopyWarps)
          reinterpret_cast<uint4 *>(kvs)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async();
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kCopyWarps) : "memory");
        int prev_t = -1, issued = 0, qn = -1;
        Token tk{0, 0, 0};
        bool tok_ok = false, waited = !p.early;
        int n_w = 0;
        const int g_own = lane & 15;  // the 4-key group whose rows this lane computes
        // idx entries of keys 4 g_own .. +3 of a compressed tile, one tile ahead
        auto load_idx = [&](int n, int32_t (&cc)[4]) {
          const int t = t0 + n / PT, j = J0 + n % PT;
          if (j >= p.WT && !waited) {
            pdl_wait();
            waited = true;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            cc[e] = -1;
            const int k = (j - p.WT) * kTk + 4 * g_own + e;
            if (j >= p.WT && k < p.K) cc[e] = p.idx[static_cast<int64_t>(t) * p.K + k];
          }
        };
        // a new token: its (sequence, position), and its queries into the Q buffer
        auto begin_token = [&](int t) -> bool {
          tok_ok = load_token(p.q_seq, p.q_pos, t, p.B, p.N_c, p.r, p.status, tk, warp == kCopyWarp0 && lane == 0);
          n_w = tok_ok ? min(p.W, tk.pos + 1) : 0;
          ++qn;
          prev_t = t;
          if (warp != kCopyWarp0) return true;
          bool ok = true;
          if (lane == 0) {
            ok = mbar_wait(qempty, (qn & 1) ^ 1, budget);
            if (ok) {
              mbar_expect_tx(qfull, kH * kD * 2);
#pragma unroll
              for (int kc = 0; kc < kChunks; ++kc) tma_load_2d(qs + kc * 8192, &qmap, qfull, 64 * kc, t * kH);
            } else {
              fail();
            }
          }
          return __shfl_sync(0xffffffffu, ok, 0);
        };
        bool run = begin_token(t0);
        int32_t cnext[4];
        load_idx(0, cnext);
        for (int n = 0; n < count; ++n) {
          const int t = t0 + n / PT, j = J0 + n % PT;
          int32_t cidx[4] = {cnext[0], cnext[1], cnext[2], cnext[3]};
          bool ok = run;
          if (ok && t != prev_t) ok = begin_token(t);
          // rows and presence of keys 4 g_own .. 4 g_own + 3
          const bool window = j < p.WT;
          int rows[4];
          bool valid[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            rows[e] = 0;
            valid[e] = false;
            if (!tok_ok) continue;
            if (window) {
              const int q = j * kTk + 4 * g_own + e;
              if (q < n_w) {
                const int pos = tk.pos - n_w + 1 + q;
                rows[e] = tk.b * p.wseq + pos % p.R;
                valid[e] = true;
              }
            } else if (cidx[e] >= 0 && cidx[e] < tk.nv) {
              rows[e] = tk.b * p.cseq + cidx[e];
              valid[e] = true;
            } else if (cidx[e] != -1 && warp == kCopyWarp0 && lane < 16) {
              raise_flag(p.status, kFlagBadIndex);
            }
          }
          const int s = n % kSlots;
          if (ok) ok = mbar_wait_warp(&kvempty[s], ((n / kSlots) & 1) ^ 1, budget);
          if (!ok && lane == 0) fail();
          // Under a short wait bound every copy warp takes the same decision (a
          // reducing barrier per tile), so that a tile's copies are issued by
          // all of them or by none: its barrier then completes and the drain
          // below ends as soon as they land.  At the default bound (a stop is
          // then all but impossible) each warp decides alone, and a drain may
          // wait out its own bound.
          const bool stop = kShort ? barrier_any(1, 32 * kCopyWarps, !ok || aborted())
                                   : __any_sync(0xffffffffu, !ok || aborted());
          if (stop) break;
          if (warp == kCopyWarp0) {  // key mask: bit g of word e = key 4g+e exists
            uint32_t m4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = __ballot_sync(0xffffffffu, valid[e]) & 0xFFFFu;
            if (lane == 0) {
#pragma unroll
              for (int e = 0; e < 4; ++e) mask_s[(n % kMaskSlots) * 4 + e] = m4[e];
              mbar_arrive(&mfull[n % kMaskSlots]);
            }
          }
          {
            // this warp's copies c = lane * kCopyWarps + pw < 128: group g = c % 16
            // (keys 4g..4g+3), chunk kc = c / 16 (dims 64 kc .. 64 kc + 63).
            // Absent keys of a group read a present key's row; a group with none
            // is not copied (its rows keep what the slot held: finite values --
            // the ring starts zeroed -- multiplied by P = 0 and masked out of
            // the logits).
            const bool any4 = valid[0] || valid[1] || valid[2] || valid[3];
            const int fill = valid[0] ? rows[0] : valid[1] ? rows[1] : valid[2] ? rows[2] : rows[3];
            const int c = lane * kCopyWarps + pw;
            const int g = c & 15, kc = c >> 4;
            int gr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) gr[e] = __shfl_sync(0xffffffffu, valid[e] ? rows[e] : fill, g);
            const bool gany = __shfl_sync(0xffffffffu, any4, g);
            const bool mine = c < kCopies && gany;
            const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, mine)) * 512u;
            if (lane == 0) mbar_expect_tx(&kvfull[s], bytes);
            __syncwarp();
            if (mine) {
              uint8_t *dst = kvs + s * 65536 + kc * 8192 + 4 * g * 128;
              gather4(dst, window ? &wmap : &cmap, &kvfull[s], 64 * kc, gr[0], gr[1], gr[2], gr[3], rpol);
            }
          }
          ++issued;
          // the next tile's indices load while this tile's rows are in flight
          if (n + 1 < count) load_idx(n + 1, cnext);
        }
        if (lane == 0) {  // drain: every copy this warp issued lands before the CTA exits
          for (int n = max(0, issued - kSlots); n < issued; ++n) mbar_wait(&kvfull[n % kSlots], (n / kSlots) & 1);
          if (warp == kCopyWarp0 && qn >= 0) mbar_wait(qfull, qn & 1);
        }
      }
    } else {
      // ------------------------------------------------------------- MMA issuer
      // S^T runs a tile ahead of the P.V product: after S(n), S(n + 1) and
      // O(n) go out in whichever order their inputs complete (the rows of
      // tile n + 1, or P(n)), so that a late tile does not hold back the
      // product whose completion frees a ring slot.  The whole warp waits; one
      // elected lane tests and issues.  Each instruction reads its whole A
      // operand (128 rows x 16 values) from shared memory, so a product costs
      // about the same per instruction for N = 32 as for N = 64: S is taken
      // as one N = 64 product per 16 dims.
      if (count > 0) {
        const bool leader = elect_one();
        const int leader_lane = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
        constexpr uint32_t idesc_s = idesc_bf16(128, kH);                           // K-major A and B
        constexpr uint32_t idesc_o = idesc_bf16(128, kH) | (1u << 15) | (1u << 16);  // MN-major A and B
        int tok_s = -1, prev_t_s = -1, tok_o = -1;
        bool ok = true;
        auto issue_s = [&](int n) -> bool {
          const int t = t0 + n / PT;
          const int s = n % kSlots, b = n % kSBufs;
          if (t != prev_t_s) {
            ++tok_s;
            prev_t_s = t;
            if (!mbar_wait_warp(qfull, tok_s & 1, budget)) return false;
          }
          if (!mbar_wait_warp(&kvfull[s], (n / kSlots) & 1, budget) ||
              !mbar_wait_warp(&sempty[b], ((n / kSBufs) & 1) ^ 1, budget))
            return false;
          tc_fence_after();
          if (leader) {
            // the descriptors of k-step kk are the base descriptors plus its
            // byte offset / 16 (addresses stay below 256 KB, so the start
            // address field does not carry)
            const uint64_t da = desc_sw128_kmajor(smem_u32(kvs + s * 65536)), db = desc_sw128_kmajor(smem_u32(qs));
            const uint32_t d0 = tmem + kColS + 64 * b;
#pragma unroll
            for (int kk = 0; kk < kSSteps; ++kk) {  // 16 dims at a time
              const uint64_t c = static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
              mma_f16(d0, da + c, db + c, idesc_s, kk > 0);
            }
            mma_commit(&sfull[b]);
            if (n % PT == PT - 1) mma_commit(qempty);
          }
          __syncwarp();
          return true;
        };
        auto issue_o = [&](int n) -> bool {
          const bool first = n % PT == 0;
          const int s = n % kSlots, pb = n % kPBufs;
          if (first && tok_o >= 0 && !mbar_wait_warp(oempty, tok_o & 1, budget)) return false;
          if (!mbar_wait_warp(&pfull[pb], (n / kPBufs) & 1, budget)) return false;
          if (first) ++tok_o;
          tc_fence_after();
          if (leader) {
            // base descriptors plus byte offset / 16, as for S
            const uint64_t dv = desc_sw128_mnmajor(smem_u32(kvs + s * 65536), 8192);
            const uint64_t dp = desc_sw128_mnmajor(smem_u32(pts + pb * 16384), 8192);
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {  // dims 128 mb .. 128 mb + 127: chunks 2 mb, 2 mb + 1
#pragma unroll
              for (int kk = 0; kk < kTk / 16; ++kk) {  // keys 16 kk .. 16 kk + 15
                const uint64_t a = dv + static_cast<uint64_t>((2 * mb * 8192 + kk * 2048) >> 4);
                const uint64_t ph = dp + static_cast<uint64_t>((kk * 2048) >> 4);
                mma_f16(tmem + 64 * mb, a, ph, idesc_o, !(first && kk == 0));
                mma_f16(tmem + 64 * mb, a, ph + (8192 >> 4), idesc_o, 1);
              }
            }
            mma_commit(&kvempty[s]);
            mma_commit(&pempty[pb]);
          }
          __syncwarp();
          return true;
        };
        // non-blocking readiness tests, taken by the issuing lane and shared
        auto ready_s = [&](int n) -> bool {
          bool r = false;
          if (leader) {
            const int t = t0 + n / PT;
            r = (t == prev_t_s || mbar_test_wait(qfull, (tok_s + 1) & 1)) &&
                mbar_test_wait(&kvfull[n % kSlots], (n / kSlots) & 1) &&
                mbar_test_wait(&sempty[n % kSBufs], ((n / kSBufs) & 1) ^ 1);
          }
          return __shfl_sync(0xffffffffu, r, leader_lane);
        };
        auto ready_o = [&](int n) -> bool {
          bool r = false;
          if (leader)
            r = (n % PT != 0 || tok_o < 0 || mbar_test_wait(oempty, tok_o & 1)) &&
                mbar_test_wait(&pfull[n % kPBufs], (n / kPBufs) & 1);
          return __shfl_sync(0xffffffffu, r, leader_lane);
        };
        int s_next = 0;  // S(s_next) is the next logit product to issue
        for (int n = 0; ok && n < count; ++n) {
          // S up to n + 1 and O(n), S(n) first (P(n) needs it)
          bool o_left = true;
          long long t_idle = clock64();
          while (ok) {
            const bool s_left = s_next < count && s_next <= n + 1;
            if (!s_left && !o_left) break;
            if (__any_sync(0xffffffffu, aborted())) {
              ok = false;
            } else if (s_left && ready_s(s_next)) {
              ok = issue_s(s_next);
              ++s_next;
              t_idle = clock64();
            } else if (o_left && ready_o(n)) {
              ok = issue_o(n);
              o_left = false;
              t_idle = clock64();
            } else if (__shfl_sync(0xffffffffu, clock64() - t_idle > budget, leader_lane)) {
              ok = false;
            } else if (leader) {
              // nothing ready: sleep in the barrier of P(n) (or of tile
              // n + 1's rows once O(n) is out) until it completes, 200 ns at most
              if (o_left)
                mbar_try_wait_ns(&pfull[n % kPBufs], (n / kPBufs) & 1, 200);
              else
                mbar_try_wait_ns(&kvfull[s_next % kSlots], (s_next / kSlots) & 1, 200);
            }
            __syncwarp();
          }
        }
        if (!ok && lane == 0) fail();
        if (leader) {
          mma_commit(done);
          if (!mbar_wait(done, 0)) raise_flag(p.status, kFlagTimeout);
        }
        __syncwarp();
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ----------------------------------------------------------------- softmax
    // Thread (warp w, lane) = key 32 (w & 1) + lane of the tile for heads
    // 32 (w >> 1) .. + 31.  The tile's logits sit in S^T lanes 0-63, which
    // only warps 0 and 1 reach: they read all 64 heads and hand heads 32-63
    // to warps 2 and 3 through shared memory.  For O^T every warp holds lanes
    // 32 w .. 32 w + 31 of each dim block (dims 128 mb + 32 w + lane), all 64
    // heads.
    const int hg = warp >> 1;  // head group: heads 32 hg .. 32 hg + 31
    const int key = 32 * (warp & 1) + lane;
    const bool keyw = warp < 2;  // warps 0 and 1 reach the S^T lanes (0-63) of the tile's keys
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const float *mref_g = mref_s + 32 * hg;
    float l[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) l[h] = 0.f;
    bool bad = false;  // a wait of this warp gave up (the group leaves together after a barrier)
    // thread 0 of a split token's CTA, once it has told the partner that its
    // ring may take the partner's hand-off: the partner may then be copying
    // into this CTA, so this CTA does not leave before the copy has landed
    bool x_armed = false;
    int jj = 0, tok = 0;
    for (int n = 0; n < count; ++n, jj = (jj + 1 == PT) ? 0 : jj + 1, tok += jj == 0) {
      const bool first = jj == 0, last = jj == PT - 1;
      const int b = n % kSBufs, pb = n % kPBufs;
      uint32_t sv[32];  // this key's logits (raw dot products) for the warp's 32 heads
      bool present = false;
      if (!mbar_wait_warp(&mfull[n % kMaskSlots], (n / kMaskSlots) & 1, budget)) {
        bad = true;
      } else {
        const uint32_t mw = mask_s[(n % kMaskSlots) * 4 + (key & 3)];
        present = ((mw >> (key >> 2)) & 1u) != 0;
      }
      // P^T buffer pb (its previous product done) first carries the logits of
      // heads 32-63 from the key warps, which alone reach the S^T lanes, to
      // warps 2 and 3: fp32 [64 keys][32 heads] in its lower half, 16-byte
      // chunk c of key k's row at chunk position c ^ (k & 7)
      if (!bad && !mbar_wait_warp(&pempty[pb], ((n / kPBufs) & 1) ^ 1, budget)) bad = true;
      uint8_t *xrow = pts + pb * 16384 + 8192 + 128 * key;
      bool over = false;  // does a present logit pass its head's reference by the lazy margin?
      if (keyw && !bad) {
        if (!mbar_wait_warp(&sfull[b], (n / kSBufs) & 1, budget)) {
          bad = true;
        } else {
          tc_fence_after();
          uint32_t s2[32];
          tmem_ld_32x32b_x32(tmem + lane_base + kColS + 64 * b, sv);
          tmem_ld_32x32b_x32(tmem + lane_base + kColS + 64 * b + 32, s2);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sempty[b]);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(xrow + 16 * (c ^ (key & 7))) =
                make_uint4(s2[4 * c], s2[4 * c + 1], s2[4 * c + 2], s2[4 * c + 3]);
          if (!first && present) {
#pragma unroll
            for (int h = 0; h < 32; ++h)
              over |= fmaxf(__uint_as_float(sv[h]) * p.qk_scale - mref_s[h],
                            __uint_as_float(s2[h]) * p.qk_scale - mref_s[32 + h]) > kLazyRescale;
          }
        }
      }
      if (bad && lane == 0) fail();
      over = __any_sync(0xffffffffu, over);
      // every warp votes, then all read the same four votes: the group leaves
      // the loop, or not, together
      if (lane == 0) votes_s[(n & 1) * 4 + warp] = (over ? 1 : 0) | ((bad || aborted()) ? 2 : 0);
      group_sync();  // (1) the votes, and the hand-over of heads 32-63
      const int vote = votes_s[(n & 1) * 4] | votes_s[(n & 1) * 4 + 1] | votes_s[(n & 1) * 4 + 2] |
                       votes_s[(n & 1) * 4 + 3];
      if (vote & 2) break;
      if (!keyw) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4 *>(xrow + 16 * (c ^ (key & 7)));
          sv[4 * c] = v.x;
          sv[4 * c + 1] = v.y;
          sv[4 * c + 2] = v.z;
          sv[4 * c + 3] = v.w;
        }
      }
      if (first || (vote & 1) != 0) {
        // the tile's max per head over its present keys: reduced within each
        // warp (lane l ends with head 32 hg + l), the two key halves combined
        // through shared memory
        float x[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) x[h] = present ? __uint_as_float(sv[h]) * p.qk_scale : -INFINITY;
        red_s[32 * warp + lane] = warp_reduce_scatter32<true>(x, lane);
        group_sync();  // (2) the partial maxima
        // new reference per head (thread h of the group); the factor O^T and
        // the sums take
        if (tid < kH) {
          const int g = tid >> 5, i = tid & 31;
          const float mo = first ? -INFINITY : mref_s[tid];
          const float mn = fmaxf(mo, fmaxf(red_s[64 * g + i], red_s[64 * g + 32 + i]));
          fac_s[tid] = (mo == -INFINITY || mn == -INFINITY) ? 1.f : exp2f(mo - mn);
          mref_s[tid] = mn;
        }
        group_sync();  // (3) references and factors
        if (!first) {
          // O^T holds the products of tiles up to n - 1: wait for the last, then
          // scale this warp's lanes of every block, column h by factor h
          if (!mbar_wait_warp(&pempty[(n - 1) % kPBufs], ((n - 1) / kPBufs) & 1, budget)) {
            if (lane == 0) fail();
          } else {
            tc_fence_after();
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb)
#pragma unroll 1
              for (int half = 0; half < 2; ++half) {
                uint32_t o[32];
                const uint32_t ta = tmem + lane_base + 64 * mb + 32 * half;
                tmem_ld_32x32b_x32(ta, o);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * fac_s[32 * half + q]);
                tmem_st_32x32b_x32(ta, o);
              }
            tmem_st_wait();
            tc_fence_before();
          }
#pragma unroll
          for (int h = 0; h < 32; ++h) l[h] *= fac_s[32 * hg + h];
        }
        group_sync();  // (4) O^T rescaled before any further product is issued
      } else {
        group_sync();  // (1b) the hand-over read before P^T is written over it
      }
      // ---- P^T row of this key, heads 32 hg .. + 31: p = 2^(scale s - m_ref)
      // as bf16 hi + lo (over the hand-over area: every read of it precedes
      // the barriers (2)-(4) or (1b))
      if (!bad) {
        uint8_t *hi_row = pts + pb * 16384, *lo_row = hi_row + 8192;
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // heads 8c .. 8c + 7 of the group: one 16-byte chunk of the row
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int h = 8 * c + 2 * q;
            const float pa = present ? ex2_approx(fmaf(__uint_as_float(sv[h]), p.qk_scale, -mref_g[h])) : 0.f;
            const float pb2 = present ? ex2_approx(fmaf(__uint_as_float(sv[h + 1]), p.qk_scale, -mref_g[h + 1])) : 0.f;
            l[h] += pa;
            l[h + 1] += pb2;
            const uint32_t ua = __float_as_uint(pa), ub = __float_as_uint(pb2);
            const float la = pa - __uint_as_float(ua & 0xFFFF0000u);
            const float lb = pb2 - __uint_as_float(ub & 0xFFFF0000u);
            hw[q] = __byte_perm(ua, ub, 0x7632);
            lw[q] = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
          }
          const uint32_t off = sw128_offset(static_cast<uint32_t>(key), 16u * (4 * hg + c));
          *reinterpret_cast<uint4 *>(hi_row + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4 *>(lo_row + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async();  // the rows are read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[pb]);
      }
      if (last) {
        // ---- end of the token: O^T complete once the tile's product is done
        if (!bad && !mbar_wait_warp(&pempty[pb], (n / kPBufs) & 1, budget)) {
          if (lane == 0) fail();
          bad = true;
        }
        tc_fence_after();
        // a split token's part: every product of this CTA is done, so the
        // upper half of its kv ring and its P^T area may take the partner's
        // hand-off
        if (split > 1 && tid == 0 && !bad) {
          mbar_expect_tx(xfull, kXferBytes);
          mbar_arrive_remote(xempty, rank ^ 1);
          x_armed = true;
        }
        // the sums per head (lane l: head 32 hg + l over the warp's keys)
        red_s[32 * warp + lane] = warp_reduce_scatter32<false>(l, lane);
#pragma unroll
        for (int h = 0; h < 32; ++h) l[h] = 0.f;
        group_sync();  // (5) the sums
        // this part's (m_ref, sum) per head at 8 h of the P^T area
        if (tid < kH) {
          const int g = tid >> 5, i = tid & 31;
          *reinterpret_cast<float2 *>(pts + 8 * tid) =
              make_float2(mref_s[tid], red_s[64 * g + i] + red_s[64 * g + 32 + i]);
        }
        // a split token: each CTA writes dims 256 rank .. + 255 of the output
        // and hands the partner its O^T for the partner's dims (blocks
        // 2 (rank ^ 1), + 1) through the lower half of the ring: 4-column
        // chunk c (c = 16 i + column / 4 of the i-th block) of thread t at
        // 16 (128 c + t), so a warp's store covers 512 contiguous bytes
        if (split > 1 && !bad) {
#pragma unroll 1
          for (int i = 0; i < 2; ++i)
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(tmem + lane_base + 64 * (2 * (rank ^ 1) + i) + 32 * half, o);
              tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(kvs + 16 * (128 * (16 * i + 8 * half + q) + tid)) =
                    make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            }
        }
        fence_proxy_async();  // the bulk copies read what this thread wrote
        tc_fence_before();
        group_sync();  // (6) the part's (m_ref, sum) and the hand-off staged, or a failure flagged
        if (split > 1) {
          if (tid == 0) {
            if (!aborted() && mbar_wait_cluster(xempty, 0, budget)) {
              const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
              const uint32_t bar = cluster_map(xfull, peer);
#pragma unroll 1
              for (int i = 0; i < kXferChunks; ++i)
                bulk_copy_to_cluster(cluster_map(kvs + 65536 + i * kXferChunk, peer), kvs + i * kXferChunk,
                                     kXferChunk, bar);
              bulk_copy_to_cluster(cluster_map(pts + 8 * kH, peer), pts, 8 * kH, bar);
            } else {
              fail();
            }
          }
          if (!mbar_wait_cluster_warp(xfull, 0, budget) && lane == 0) fail();
        }
        // O = (a0 O0 + a1 O1) / L against M = max(m0, m1), L = a0 l0 + a1 l1
        // (part 0 = this CTA's, part 1 = the partner's, absent for a whole token)
        if (tid < kH) {
          const float2 own = *reinterpret_cast<const float2 *>(pts + 8 * tid);
          float2 other = make_float2(-INFINITY, 0.f);
          if (split > 1) other = *reinterpret_cast<const float2 *>(pts + 8 * kH + 8 * tid);
          const float M = fmaxf(own.x, other.x);
          const float a0 = own.x == -INFINITY ? 0.f : exp2f(own.x - M);
          const float a1 = other.x == -INFINITY ? 0.f : exp2f(other.x - M);
          const float Ls = own.y * a0 + other.y * a1;
          // 1 / (sum of weights, plus the sink's term when given)
          float Lden = Ls, a = 1.f;
          if (p.sink) {
            const float s2 = p.sink[tid] * kLog2e;
            const float Mf = fmaxf(M, s2);
            a = (M == -INFINITY) ? 0.f : exp2f(M - Mf);
            Lden = Ls * a + exp2f(s2 - Mf);
          }
          const float inv = Lden > 0.f ? a / Lden : 0.f;
          fac_s[tid] = a0 * inv;
          red_s[tid] = a1 * inv;
        }
        group_sync();  // (7) output scales
        {
          const int64_t tbase = static_cast<int64_t>(t0 + tok) * kH;
          // the scales are read where they are used (volatile: hoisting all 128
          // out of the loop would take registers the loop over tiles holds)
          const volatile float *f0v = fac_s, *f1v = red_s;
          const int nblk = split > 1 ? 2 : 4, mb0 = split > 1 ? 2 * rank : 0;
#pragma unroll 1
          for (int i = 0; i < nblk; ++i) {
            const int mb = mb0 + i;
            const int d = 128 * mb + 32 * warp + lane;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(tmem + lane_base + 64 * mb + 32 * half, o);
              tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 v4 = split > 1 ? *reinterpret_cast<const float4 *>(
                                                  kvs + 65536 + 16 * (128 * (16 * i + 8 * half + q) + tid))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                const float x[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int h = 32 * half + 4 * q + e;
                  const float y = fmaf(__uint_as_float(o[4 * q + e]), f0v[h], x[e] * f1v[h]);
                  p.out[(tbase + h) * kD + d] = __float2bfloat16_rn(y);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(oempty);
      }
    }
    // the hand-off into this CTA has landed, or (partner failed) a second has passed
    if (x_armed && !mbar_wait_cluster(xfull, 0)) raise_flag(p.status, kFlagTimeout);
  }

  // a CTA whose part had no compressed tile never waited for the previous
  // kernel: it does so before leaving, so that this kernel completes after it
  if (p.early) pdl_wait();
  tc_fence_before();
  __syncthreads();
  // neither CTA of a cluster leaves while the other may still write to or
  // arrive on its shared memory
  if (split > 1) cluster_sync();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// 2-D tensor map over `rows` rows of 512 bf16 (1 KB apart), a box of 64
// values and `box_rows` rows, 128-byte swizzle.
bool encode_rows512(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {kD, rows};
  const cuuint64_t strides[1] = {kD * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t attn512_smem_bytes() { return Smem512::total + 1024; }

// 2-CTA clusters of this kernel that fit on the GPU at once (0 if unknown).
int max_pair_clusters512() {
  static int cached[64];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!done[dev]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = attn512_smem_bytes();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mqa_umma512_kernel<false>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[dev] = n;
    done[dev] = true;
  }
  return cached[dev];
}

}  // namespace

bool attn_umma512_supported(const sa_attn_args &aa) {
  return aa.H == kH && aa.D == kD && aa.Kw == aa.Vw && aa.Kc == aa.Vc;
}

cudaError_t launch_sparse_mqa_umma512(const sa_index_args &ia, const sa_attn_args &aa, const int32_t *idx, int K,
                                      void *out, bool inputs_ready, uint32_t *status, cudaStream_t stream) {
  const long long budget = attn_wait_budget();
  if (ia.T == 0) return cudaSuccess;
  Attn512Params p;
  p.B = ia.B;
  p.T = ia.T;
  p.N_c = ia.N_c;
  p.r = ia.r;
  p.W = aa.W;
  p.R = aa.R;
  p.K = K;
  p.WT = (aa.W + kTk - 1) / kTk;
  p.TPT = p.WT + (K + kTk - 1) / kTk;
  p.wseq = static_cast<int>(w_rows_per_seq(aa));
  p.cseq = static_cast<int>(c_rows_per_seq(ia, aa));
  p.evict_first = ia.T <= ia.B ? 1 : 0;
  p.early = inputs_ready ? 1 : 0;
  const bool short_budget = budget > 0 && budget < kWaitBudgetCycles;
  auto kern = short_budget ? sparse_mqa_umma512_kernel<true> : sparse_mqa_umma512_kernel<false>;
  p.budget = short_budget ? budget : kWaitBudgetCycles;
  p.q_seq = ia.q_seq;
  p.q_pos = ia.q_pos;
  p.idx = idx;
  p.sink = aa.sink;
  p.qk_scale = aa.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.status = status;
  CUtensorMap qmap, wmap, cmap;
  if (!encode_rows512(&qmap, aa.Q, static_cast<uint64_t>(ia.T) * kH, 64) ||
      !encode_rows512(&wmap, aa.Kw, static_cast<uint64_t>(ia.B - 1) * p.wseq + aa.R, 1) ||
      !encode_rows512(&cmap, aa.Kc, static_cast<uint64_t>(ia.B - 1) * p.cseq + ia.N_c, 1))
    return cudaErrorInvalidValue;
  // the register split assumes kLaunchRegs registers per thread at launch;
  // anything else could leave a raise waiting forever
  static int regs[2] = {-1, -1};
  if (regs[short_budget] < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(kern));
    if (e != cudaSuccess) return e;
    regs[short_budget] = fa.numRegs;
  }
  if (regs[short_budget] != kLaunchRegs) return cudaErrorInvalidConfiguration;
  const size_t smem = attn512_smem_bytes();
  static bool attr_done[2][64] = {};
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), smem, attr_done[short_budget]);
  if (e != cudaSuccess) return e;
  if (short_budget) {  // the occupancy query below runs on the default kernel
    static bool attr_done_default[64] = {};
    e = set_smem_once(reinterpret_cast<const void *>(sparse_mqa_umma512_kernel<false>), smem, attr_done_default);
    if (e != cudaSuccess) return e;
  }
  // a 2-CTA cluster per token when every token can have one at once (each CTA
  // half of the token's tiles), else whole tokens with at most one CTA per SM
  p.split = (p.TPT >= 2 && ia.T <= max_pair_clusters512()) ? 2 : 1;
  // rank 0 takes the larger half, window first (in the fused step its rows
  // load before the wait for the indices)
  p.PT0 = (p.TPT + 1) / 2;
  const int sms = sm_count();
  const int grid = p.split == 1 ? (ia.T < sms ? ia.T : sms) : 2 * ia.T;
  return launch_ex(true, kern, dim3(grid), dim3(kThreads), smem, stream, p.split, qmap, wmap, cmap, p);
}

}  // namespace sa
