// Sparse MQA on the 5th-generation tensor cores (tcgen05) for 64 query heads
// of dim 128 sharing one KV head ("DeepSeek-V4.1-Flash-NVFP4
// inference/model.py", Attention.forward: sparse_attn over the window rows
// and the index-selected compressed rows).
//
// Each token's key list is its window (padded to a multiple of 128) followed
// by its K index slots (padded likewise), i.e. TPT tiles of 128 keys.  Every
// CTA takes whole tokens (a contiguous token range), so no token is split.
// Per tile:
//   S = Q K^T      M = 128, N = 128 keys, K = 128, bf16 x bf16 -> f32 in
//                  tensor memory.  Head 16w+i (w = 0..3, i = 0..15) is A row
//                  and accumulator lane 32w+i, so each quarter of tensor
//                  memory (one per SM sub-partition) holds 16 heads; the
//                  other 64 rows are not used;
//   softmax        four warps, one per sub-partition; a thread takes one head
//                  and 64 of the tile's 128 keys (the 16x32bx2 access shape:
//                  threads 0-15 keys 0-63, threads 16-31 keys 64-127 of the
//                  same 16 heads): the tile max, then p = 2^(scale s - m) with
//                  a lazily raised reference max (O is rescaled only when a
//                  tile's max exceeds it by more than 2^8);
//   O += P V       P written over the logits it came from, as a bf16 hi + lo
//                  pair (two MMAs into the same accumulator); V read MN-major
//                  from the gathered tile; M = 128, N = 128 (d), K = 128 keys.
// Three S/P buffers let S run two tiles ahead of P.V, so the softmax waits for
// the tensor core only to rescale O and at a token's end.
// K and V rows are gathered by index with TMA gather4 (4 rows of 128 bytes per
// instruction) into the 128-byte-swizzled layout both MMAs read, in two
// separate rings: a K slot is free once S is done, a V slot once P.V is done.
//
// Warps: 0-3 softmax; 4 MMA issuer and tensor-memory owner; 5-10 copy K rows
// (warp 5 also loads each token's Q and writes the tile's key mask); 11-15
// copy V rows.  Issuing gather4 copies is the limit of a single warp, hence
// eleven issuers.  Every wait is bounded; on expiry the kernel flags the
// status word, drains its copies and MMAs, and returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace sa {
namespace {

using namespace umma;

constexpr int kH = 64;            // query heads handled by this kernel
constexpr int kD = 128;           // head dim
constexpr int kTile = 128;        // keys per tile
constexpr int kStages = 3;        // slots of the K ring and of the V ring
constexpr int kMaskSlots = 6;     // key masks; written up to 3 tiles ahead of their reader
constexpr int kThreads = 512;
constexpr int kMmaWarp = 4;
constexpr int kKWarp0 = 5, kKWarps = 6;   // warps 5-10
constexpr int kVWarp0 = 11, kVWarps = 5;  // warps 11-15
constexpr float kLazyRescale = 8.f;  // log2 units
// Registers per thread: the kernel is built for 128 (512 threads on 64K
// registers); the softmax warpgroup (warps 0-3) raises its limit and the other
// three lower theirs, 184 + 3 * 104 <= 4 * 128 so the raise can always be met.
constexpr int kLaunchRegs = 128, kSoftmaxRegs = 184, kOtherRegs = 104;
static_assert(kSoftmaxRegs + 3 * kOtherRegs <= 4 * kLaunchRegs, "register split exceeds the launch allocation");

constexpr int kSBufs = 3;          // S/P buffers in tensor memory (P overwrites its S in place)
constexpr uint32_t kColO = 384;    // tensor-memory columns: S/P buffer b at 128 b, O at 384

// Q: two token buffers share one 32 KB region [kblk][128 rows][128 B]: head
// 16w+i of buffer qb is row 32w+16qb+i.  The S MMA of buffer qb reads 128 rows
// from row 16qb, so A row 32w+i is head 16w+i; the rows in between (the other
// buffer, or past the region) only feed unused accumulator rows.
struct AttnSmem {
  static constexpr size_t q = 0;                                   // [2 kblk][128 rows][128 B]
  static constexpr size_t k = q + 32768;                           // [slot][2 kblk][128 rows][128 B]
  static constexpr size_t v = k + kStages * 32768;
  static constexpr size_t mask = v + kStages * 32768;              // [slot][4] u32
  static constexpr size_t bars = (mask + kMaskSlots * 16 + 7) & ~size_t(7);
  static constexpr int kBars = 4 * kStages + 4 + 3 * kSBufs + 2 + kMaskSlots + 2;
  static constexpr size_t misc = bars + kBars * 8;
  static constexpr size_t total = misc + 64;
};

struct AttnUmmaParams {
  int B, T, N_c, r, W, R, K;
  int wseq, cseq;                 // rows between consecutive sequences of the ring and of the compressed cache
  int WT, TPT;                    // window tiles per token, tiles per token
  int split, PT0;                 // CTAs per token (1, or a 2-CTA cluster with one token), tiles of rank 0's part
  int early;                      // nonzero: every input but idx is complete at launch, so only idx waits for the predecessor
  long long budget;               // SM cycles a pipeline wait may take before the kernel gives up (drains keep the full budget)
  int evict_first;                // nonzero: K/V rows are read once per call (at most one token per sequence)
  const int32_t *q_seq, *q_pos, *idx;
  const __nv_bfloat16 *Vw, *Vc;   // V rows (window ring, compressed), 128 bf16 each
  const float *sink;
  float qk_scale;                 // scale * log2(e)
  __nv_bfloat16 *out;
  uint32_t *status;
};

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16x32bx2 shape with a half offset of 64 columns: thread t of the warp
// accesses lane (warp quarter) + t % 16, columns col + 64 (t / 16) + j.
__device__ __forceinline__ void tmem_ld_16x2_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], 64;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_16x2_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16], 64;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st_16x2_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], 64, "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_16x2_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.16x32bx2.x8.b32 [%0], 64, {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// O[tmem] (+)= A[tmem] . B[smem]
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

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
// 64 N values per row, N blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t desc_sw128_mnmajor(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Key q (0..63) of a thread's 64 keys is present iff bit q/4 of mw[q%4] is
// set, mw = the tile's mask words shifted to the thread's half (bit g of word
// e = key 4g+e of the tile).
__device__ __forceinline__ bool key_present(const uint32_t (&mw)[4], int q) {
  return ((mw[q & 3] >> (q >> 2)) & 1u) != 0;
}

// Max of the present logits among 64 (eight independent partial maxima, so
// the compare chain is eight deep instead of 64).
template <bool MASKED>
__device__ __forceinline__ float max64(const uint32_t (&v)[64], const uint32_t (&mw)[4]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = -INFINITY;
#pragma unroll
  for (int q = 0; q < 64; ++q) {
    float x = __uint_as_float(v[q]);
    if (MASKED) x = key_present(mw, q) ? x : -INFINITY;
    m[q & 7] = fmaxf(m[q & 7], x);
  }
#pragma unroll
  for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}

// p = 2^(c s - m) of the 16 logits v[16G .. 16G+15] (absent keys give 0),
// added into four partial sums, and split into P = hi + lo: hi = p truncated
// to bf16, lo = (p - hi) truncated to bf16 (|p - hi - lo| < 2^-16 p); pairs of
// keys packed per 32-bit word by byte permutes.
template <bool MASKED, int G>
__device__ __forceinline__ void exp_split16(const uint32_t (&v)[64], const uint32_t (&mw)[4], float c, float neg_m,
                                            uint32_t (&hi)[8], uint32_t (&lo)[8], float (&s4)[4]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int k = 16 * G + 2 * q;
    float pa = ex2_approx(fmaf(__uint_as_float(v[k]), c, neg_m));
    float pb = ex2_approx(fmaf(__uint_as_float(v[k + 1]), c, neg_m));
    if (MASKED) {
      pa = key_present(mw, k) ? pa : 0.f;
      pb = key_present(mw, k + 1) ? pb : 0.f;
    }
    s4[q & 3] += pa + pb;
    const uint32_t ua = __float_as_uint(pa), ub = __float_as_uint(pb);
    const float la = pa - __uint_as_float(ua & 0xFFFF0000u);
    const float lb = pb - __uint_as_float(ub & 0xFFFF0000u);
    hi[q] = __byte_perm(ua, ub, 0x7632);
    lo[q] = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
  }
}

// The thread's 64 keys, 16 at a time: group G (keys 16G .. 16G+15 of the
// thread's half) goes to columns 32(G/2) + 8(G%2) (hi) and 16 more (lo) of the
// thread's half of the S/P buffer, over logits already in registers.
template <bool MASKED>
__device__ __forceinline__ void exp_store64(const uint32_t (&v)[64], const uint32_t (&mw)[4], float c, float neg_m,
                                            uint32_t s_col, float (&s4)[4]) {
  uint32_t hi[8], lo[8];
  exp_split16<MASKED, 0>(v, mw, c, neg_m, hi, lo, s4);
  tmem_st_16x2_x8(s_col + 0, hi);
  tmem_st_16x2_x8(s_col + 16, lo);
  exp_split16<MASKED, 1>(v, mw, c, neg_m, hi, lo, s4);
  tmem_st_16x2_x8(s_col + 8, hi);
  tmem_st_16x2_x8(s_col + 24, lo);
  exp_split16<MASKED, 2>(v, mw, c, neg_m, hi, lo, s4);
  tmem_st_16x2_x8(s_col + 32, hi);
  tmem_st_16x2_x8(s_col + 48, lo);
  exp_split16<MASKED, 3>(v, mw, c, neg_m, hi, lo, s4);
  tmem_st_16x2_x8(s_col + 40, hi);
  tmem_st_16x2_x8(s_col + 56, lo);
}

// kShort: the waits between stages take the bound of sa_set_wait_budget (and
// the copy warps vote on stopping); otherwise the default bound, a constant
template <bool kShort>
__global__ void __launch_bounds__(kThreads, 1)
sparse_mqa_umma_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kwmap,
                       const __grid_constant__ CUtensorMap kcmap, const __grid_constant__ CUtensorMap vwmap,
                       const __grid_constant__ CUtensorMap vcmap, const AttnUmmaParams p) {
  using L = AttnSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *ks = smem + L::k, *vs = smem + L::v, *qs = smem + L::q;
  uint32_t *mask_s = reinterpret_cast<uint32_t *>(smem + L::mask);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *kfull = bars, *kempty = bars + kStages;
  uint64_t *vfull = bars + 2 * kStages, *vempty = bars + 3 * kStages;
  uint64_t *qfull = bars + 4 * kStages, *qempty = qfull + 2;
  // per S/P buffer: S written (sfull), P written (pfull), P.V done = buffer free (sempty)
  uint64_t *sfull = qempty + 2, *pfull = sfull + kSBufs, *sempty = pfull + kSBufs;
  uint64_t *oempty = sempty + kSBufs;  // O of the previous token read out
  uint64_t *done = oempty + 1;
  uint64_t *mfull = done + 1;  // [kMaskSlots]: the slot's key mask is written
  // split handoff: xempty (rank 1) = rank 0's K ring is free to take rank 1's partial;
  // xfull (rank 0) = the partial is there
  uint64_t *xfull = mfull + kMaskSlots, *xempty = xfull + 1;
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem + L::misc);
  int *abort_s = reinterpret_cast<int *>(smem + L::misc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long budget = kShort ? p.budget : kWaitBudgetCycles;  // bound of a wait between stages
  // Work: cluster c (of G) takes whole tokens [T*c/G, T*(c+1)/G); with a
  // 2-CTA cluster, rank 0 takes tiles [0, PT0) of each and rank 1 the rest.
  const int split = p.split;
  const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int G = gridDim.x / split, c = blockIdx.x / split;
  const int t0 = static_cast<int>(static_cast<long long>(p.T) * c / G);
  const int t1 = static_cast<int>(static_cast<long long>(p.T) * (c + 1) / G);
  const int J0 = rank * p.PT0;
  const int PT = split == 1 ? p.TPT : (rank == 0 ? p.PT0 : p.TPT - p.PT0);
  const int count = (t1 - t0) * PT;  // tiles of this CTA; tile n is tile J0 + n % PT of token t0 + n / PT

  static_assert(L::total + 1024 <= 232448, "shared memory budget");
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kfull[i], kKWarps);
      mbar_init(&kempty[i], 1);
      mbar_init(&vfull[i], kVWarps);
      mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], 4);
      mbar_init(&sempty[i], 1);
    }
    mbar_init(oempty, 4);
    mbar_init(done, 1);
    for (int i = 0; i < kMaskSlots; ++i) mbar_init(&mfull[i], 1);
    mbar_init(xfull, 4);
    mbar_init(xempty, 4);
    *abort_s = 0;
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
    atomicExch(abort_s, 1);
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int *>(abort_s) != 0; };

  if (warp >= 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp >= kKWarp0) {
      // --------------------------------------------------------------- producers
      const bool is_k = warp < kVWarp0;
      const int pw = is_k ? warp - kKWarp0 : warp - kVWarp0;  // rank among its ring's warps
      const int nw = is_k ? kKWarps : kVWarps;
      uint64_t *ring_full = is_k ? kfull : vfull;
      uint64_t *ring_empty = is_k ? kempty : vempty;
      const uint64_t rpol = l2_policy(p.evict_first != 0);
      uint8_t *ring = is_k ? ks : vs;
      if (count > 0) {
        if (warp == kKWarp0 && lane == 0) {
          prefetch_tmap(&qmap);
          prefetch_tmap(&kwmap);
          prefetch_tmap(&kcmap);
          prefetch_tmap(&vwmap);
          prefetch_tmap(&vcmap);
        }
        if (!is_k) {
          // V rows of absent keys are multiplied by P = 0 but must be finite:
          // an absent key of a copied group holds a present key's row, and a
          // group with no present key is not copied and keeps what the slot
          // held before, so the ring starts zeroed.  (Absent K rows only reach
          // logits the softmax masks; unused Q rows only reach accumulator
          // lanes nobody reads.)
          for (int i = pw * 32 + lane; i < kStages * 32768 / 16; i += 32 * kVWarps)
            reinterpret_cast<uint4 *>(vs)[i] = make_uint4(0, 0, 0, 0);
          fence_proxy_async();
          asm volatile("bar.sync 1, %0;" ::"n"(32 * kVWarps) : "memory");
        }
        int qn = -1, prev_t = -1, issued = 0;
        Token tk{0, 0, 0};
        bool tok_ok = false, waited = !p.early;
        int n_w = 0;
        // idx entries of keys 4*lane .. 4*lane+3 of a compressed tile, loaded one
        // tile ahead so their latency overlaps the current tile's copies
        auto load_idx = [&](int n, int32_t (&cc)[4]) {
          const int t = t0 + n / PT, j = J0 + n % PT;
          if (j >= p.WT && !waited) {
            pdl_wait();
            waited = true;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            cc[e] = -1;
            const int k = (j - p.WT) * kTile + 4 * lane + e;
            if (j >= p.WT && k < p.K) cc[e] = p.idx[static_cast<int64_t>(t) * p.K + k];
          }
        };
        // a new token: its (sequence, position), and its queries into a Q buffer
        auto begin_token = [&](int t) -> bool {
          tok_ok = load_token(p.q_seq, p.q_pos, t, p.B, p.N_c, p.r, p.status, tk, warp == kKWarp0 && lane == 0);
          n_w = tok_ok ? min(p.W, tk.pos + 1) : 0;
          ++qn;
          prev_t = t;
          if (warp != kKWarp0) return true;
          const int qb = qn & 1;
          bool ok = true;
          if (lane == 0) {
            ok = mbar_wait(&qempty[qb], ((qn >> 1) & 1) ^ 1, budget);
            if (ok) {
              // heads 16w..16w+15 -> rows 32w+16qb .. +15, both 64-column halves
              mbar_expect_tx(&qfull[qb], 2 * kH * 128);
#pragma unroll
              for (int w = 0; w < 4; ++w)
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
                  tma_load_2d(qs + kb * 16384 + (32 * w + 16 * qb) * 128, &qmap, &qfull[qb], 64 * kb,
                              t * kH + 16 * w);
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
          // rows and presence of keys 4*lane .. 4*lane+3
          const bool window = j < p.WT;
          int rows[4];
          bool valid[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            rows[e] = 0;
            valid[e] = false;
            if (!tok_ok) continue;
            if (window) {
              const int q = j * kTile + 4 * lane + e;
              if (q < n_w) {
                const int pos = tk.pos - n_w + 1 + q;
                rows[e] = tk.b * p.wseq + pos % p.R;
                valid[e] = true;
              }
            } else if (cidx[e] >= 0 && cidx[e] < tk.nv) {
              rows[e] = tk.b * p.cseq + cidx[e];
              valid[e] = true;
            } else if (cidx[e] != -1 && warp == kKWarp0) {
              raise_flag(p.status, kFlagBadIndex);
            }
          }
          const int s = n % kStages;
          if (ok) ok = mbar_wait_warp(&ring_empty[s], ((n / kStages) & 1) ^ 1, budget);
          if (!ok && lane == 0) fail();
          // Under a short wait bound the warps of a ring take the same
          // decision (a reducing barrier per tile), so that a tile's copies are
          // issued by all of them or by none: its barrier then completes and
          // the drain below ends as soon as they land.  At the default bound
          // (a stop is then all but impossible) each warp decides alone, and a
          // drain may wait out its own bound.
          const bool stop = kShort ? (is_k ? barrier_any(3, 32 * kKWarps, !ok || aborted())
                                           : barrier_any(1, 32 * kVWarps, !ok || aborted()))
                                   : __any_sync(0xffffffffu, !ok || aborted());
          if (stop) break;
          if (warp == kKWarp0) {  // key mask of the tile: bit g of word e = key 4g+e exists
            uint32_t m4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = __ballot_sync(0xffffffffu, valid[e]);
            if (lane == 0) {
#pragma unroll
              for (int e = 0; e < 4; ++e) mask_s[(n % kMaskSlots) * 4 + e] = m4[e];
              mbar_arrive(&mfull[n % kMaskSlots]);
            }
          }
          {
            // K or V rows by TMA gather4.  This warp's share of the tile's 64
            // copies: copy c = (half, group): half = columns 0-63 / 64-127 of
            // the rows, group g = keys 4g..4g+3 (absent keys of a group read a
            // present key's row; a group with none is not copied)
            const bool any4 = valid[0] || valid[1] || valid[2] || valid[3];
            const int fill = valid[0] ? rows[0] : valid[1] ? rows[1] : valid[2] ? rows[2] : rows[3];
            const int c0 = lane * nw + pw;
            const int g = c0 & 31, half = c0 >> 5;
            int gr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) gr[e] = __shfl_sync(0xffffffffu, valid[e] ? rows[e] : fill, g);
            const bool gany = __shfl_sync(0xffffffffu, any4, g);
            const bool mine = c0 < 64 && gany;
            const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, mine)) * 512u;
            if (lane == 0) mbar_expect_tx(&ring_full[s], bytes);
            __syncwarp();
            if (mine) {
              const CUtensorMap *map = is_k ? (window ? &kwmap : &kcmap) : (window ? &vwmap : &vcmap);
              uint8_t *dst = ring + s * 32768 + half * 16384 + 4 * g * 128;
              gather4(dst, map, &ring_full[s], half * 64, gr[0], gr[1], gr[2], gr[3], rpol);
            }
          }
          ++issued;
          // the next tile's indices load while this tile's rows are in flight
          if (n + 1 < count) load_idx(n + 1, cnext);
        }
        if ((warp == kKWarp0 || warp == kVWarp0) && lane == 0) {  // drain: every issued copy lands before the CTA exits
          for (int n = max(0, issued - kStages); n < issued; ++n)
            mbar_wait(&ring_full[n % kStages], (n / kStages) & 1);
          if (warp == kKWarp0)
            for (int q = max(0, qn - 1); q <= qn; ++q) mbar_wait(&qfull[q & 1], (q >> 1) & 1);
        }
      }
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------------- MMA issuer
      // Fixed order S(0), S(1), P.V(0), S(2), P.V(1), S(3), ...: S runs two
      // tiles ahead of P.V, and S(n+2) (which waits for P.V(n-1) to free its
      // buffer) is issued after P.V(n), so the tensor core always has P.V(n)
      // queued while the issuer waits.  Every input of each step is produced by
      // work issued earlier in this order, so the blocking waits cannot deadlock.
      // The whole warp waits; one elected lane issues from warp-uniform operands.
      if (count > 0) {
        const bool leader = elect_one();
        constexpr uint32_t idesc_s = idesc_bf16(128, kTile);              // K-major A, K-major B
        constexpr uint32_t idesc_o = idesc_bf16(128, kD) | (1u << 16);     // K-major A (tmem), MN-major B
        int qn_s = -1, prev_t_s = -1;  // token ordinal as seen by the S stage
        int tok_pv = -1;               // tokens started by the P.V stage
        bool ok = true;
        // S(n): Q of its token, its K tile and a free S/P buffer
        auto issue_s = [&](int n) -> bool {
          const int t = t0 + n / PT, j = J0 + n % PT;
          const int s = n % kStages, b = n % kSBufs;
          if (t != prev_t_s) {
            ++qn_s;
            prev_t_s = t;
            if (!mbar_wait_warp(&qfull[qn_s & 1], (qn_s >> 1) & 1, budget)) return false;
          }
          if (!mbar_wait_warp(&kfull[s], (n / kStages) & 1, budget) ||
              !mbar_wait_warp(&sempty[b], ((n / kSBufs) & 1) ^ 1, budget))
            return false;
          tc_fence_after();
          const uint32_t a0 = smem_u32(qs + (qn_s & 1) * 2048), b0 = smem_u32(ks + s * 32768);
          const uint32_t d = tmem + 128 * b;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_f16(d, desc_sw128_kmajor(a0 + off), desc_sw128_kmajor(b0 + off), idesc_s, kk > 0);
            }
            mma_commit(&sfull[b]);
            mma_commit(&kempty[s]);
            if (j == J0 + PT - 1) mma_commit(&qempty[qn_s & 1]);
          }
          __syncwarp();
          return true;
        };
        // P.V(n): P of the tile (in its S/P buffer: keys 32c..32c+31 as hi in
        // columns 32c..32c+15 and lo in 32c+16..32c+31), its V tile, and O read
        // out after the previous token
        auto issue_pv = [&](int n) -> bool {
          const bool first = n % PT == 0;
          const int s = n % kStages, b = n % kSBufs;
          if (first && tok_pv >= 0 && !mbar_wait_warp(oempty, tok_pv & 1, budget)) return false;
          if (!mbar_wait_warp(&pfull[b], (n / kSBufs) & 1, budget) ||
              !mbar_wait_warp(&vfull[s], (n / kStages) & 1, budget))
            return false;
          if (first) ++tok_pv;
          tc_fence_after();
          const uint32_t v0 = smem_u32(vs + s * 32768), pb = tmem + 128 * b;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // keys 16kk .. 16kk+15
              const uint64_t bdesc = desc_sw128_mnmajor(v0 + kk * 2048, 16384);
              const uint32_t col = 32 * (kk >> 1) + 8 * (kk & 1);
              mma_f16_ta(tmem + kColO, pb + col, bdesc, idesc_o, !(first && kk == 0));
              mma_f16_ta(tmem + kColO, pb + col + 16, bdesc, idesc_o, 1);
            }
            mma_commit(&vempty[s]);
            mma_commit(&sempty[b]);
          }
          __syncwarp();
          return true;
        };
        for (int n = 0; ok && n < 2 && n < count; ++n) ok = issue_s(n);
        for (int n = 0; ok && n < count; ++n) {
          if (__any_sync(0xffffffffu, aborted()) || !issue_pv(n) || (n + 2 < count && !issue_s(n + 2))) ok = false;
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
    // Warp w, thread t: head 16w + t%16 (tensor-memory lane 32w + t%16),
    // keys 64u .. 64u+63 of each tile with u = t/16 (also O columns 64u ..
    // 64u+63).  The two threads of a head combine their maxima by one shuffle
    // per tile and their sums at the token's end.  P overwrites the logits it
    // came from; O is touched only to rescale it (after waiting for the
    // previous P.V) and to read it out at a token's end.
    const int hq = lane & 15, u = lane >> 4;
    const int h = 16 * warp + hq;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    float m_ref = -INFINITY, l = 0.f;
    int jj = 0, tok = 0;  // tile within the token's part, token ordinal
    for (int n = 0; n < count; ++n, jj = (jj + 1 == PT) ? 0 : jj + 1, tok += jj == 0) {
      const bool first = jj == 0, last = jj == PT - 1;
      if (first) {
        m_ref = -INFINITY;
        l = 0.f;
      }
      const int b = n % kSBufs;
      if (!(mbar_wait_warp(&mfull[n % kMaskSlots], (n / kMaskSlots) & 1, budget) &&
            mbar_wait_warp(&sfull[b], (n / kSBufs) & 1, budget))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      // rank 0, last tile: S is done, so the K ring is free to take rank 1's part
      if (split > 1 && rank == 0 && last && lane == 0) mbar_arrive_remote(xempty, 1);
      const uint32_t s_col = tmem + lane_base + 128 * b;
      uint32_t v[64];
      tmem_ld_16x2_x32(s_col, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld_16x2_x32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      uint32_t mw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) mw[e] = mask_s[(n % kMaskSlots) * 4 + e];
      const bool all_keys = (mw[0] & mw[1] & mw[2] & mw[3]) == 0xFFFFFFFFu;  // warp-uniform
#pragma unroll
      for (int e = 0; e < 4; ++e) mw[e] >>= 16 * u;
      tmem_ld_wait();
      // ---- the tile's max over the raw dot products (scale > 0)
      float mx = all_keys ? max64<false>(v, mw) : max64<true>(v, mw);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      mx *= p.qk_scale;
      float factor = 1.f;
      bool rescale = false;
      if (first) {
        m_ref = mx;
      } else if (mx > m_ref + kLazyRescale) {
        factor = exp2f(m_ref - mx);
        m_ref = mx;
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O holds P.V of tiles up to n-1: wait for P.V(n-1), then scale this
        // warp's rows (factor 1 for heads that keep their reference)
        const int pn = n - 1;
        if (!mbar_wait_warp(&sempty[pn % kSBufs], (pn / kSBufs) & 1, budget)) {
          if (lane == 0) fail();
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t o[32];
          tmem_ld_16x2_x32(tmem + lane_base + kColO + 32 * c2, o);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * factor);
          tmem_st_16x2_x32(tmem + lane_base + kColO + 32 * c2, o);
        }
      }
      // with no key seen yet (m_ref = -inf) every key of the tile is absent
      // and masked to 0; any finite reference serves
      const float neg_m = m_ref != -INFINITY ? -m_ref : 0.f;
      // ---- P = 2^(scale * s - m_ref) as bf16 hi + lo, written over the logits
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
      if (all_keys)
        exp_store64<false>(v, mw, p.qk_scale, neg_m, s_col, s4);
      else
        exp_store64<true>(v, mw, p.qk_scale, neg_m, s_col, s4);
      tmem_st_wait();
      l = l * factor + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[b]);

      if (last) {
        // O is complete once P.V(n) is done
        if (!mbar_wait_warp(&sempty[b], (n / kSBufs) & 1, budget)) {
          if (lane == 0) fail();
          break;
        }
        tc_fence_after();
        const float l_all = l + __shfl_xor_sync(0xffffffffu, l, 16);
        const int64_t row = static_cast<int64_t>(t0 + tok) * kH + h;
        if (rank == 1) {
          // second part of a split token: (m, l, O) go to rank 0's K ring once
          // it is free, laid out by softmax thread (the same thread of rank 0
          // reads them): O chunk q (4 columns) of thread i at 16 (128 q + i),
          // so a warp's store covers 512 contiguous bytes; (m, l) at 32 KB + 8 i
          if (!mbar_wait_cluster_warp(xempty, 0, budget)) {
            if (lane == 0) fail();
            break;
          }
          const uint32_t xo = cluster_map(ks + tid * 16, 0);
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {  // once per token: a short loop, not unrolled
            uint32_t o[16];
            tmem_ld_16x2_x16(tmem + lane_base + kColO + 16 * c4, o);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_cluster_f4(xo + 2048 * (4 * c4 + q), __uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                            __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
          }
          {
            const uint32_t xml = cluster_map(ks + 32768 + tid * 8, 0);
            asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(xml), "f"(m_ref), "f"(l_all) : "memory");
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_remote(xfull, 0);
            mbar_arrive(oempty);
          }
        } else {
          // whole token, or the first part merged with rank 1's:
          // O = a0 O0 + a1 O1, l = a0 l0 + a1 l1 against M = max(m0, m1)
          float m1 = -INFINITY, l1 = 0.f;
          const float4 *xo = reinterpret_cast<const float4 *>(ks) + tid;  // chunk q at xo[128 q]
          if (split > 1) {
            if (!mbar_wait_cluster_warp(xfull, 0, budget)) {
              if (lane == 0) fail();
              break;
            }
            const float2 ml = *reinterpret_cast<const float2 *>(ks + 32768 + tid * 8);
            m1 = ml.x;
            l1 = ml.y;
          }
          const float M = fmaxf(m_ref, m1);
          const float a0 = m_ref == -INFINITY ? 0.f : exp2f(m_ref - M);
          const float a1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
          const float Lsum = l_all * a0 + l1 * a1;
          float Lden = Lsum, a = 1.f;
          if (p.sink) {
            const float s2 = p.sink[h] * kLog2e;
            const float Mf = fmaxf(M, s2);
            a = (M == -INFINITY) ? 0.f : exp2f(M - Mf);
            Lden = Lsum * a + exp2f(s2 - Mf);
          }
          const float inv = Lden > 0.f ? a / Lden : 0.f;
          const float f0 = a0 * inv, f1 = a1 * inv;
          uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kD + 64 * u);
          // 16 columns at a time (columns 64u + 16c4 ..): merge with the
          // partner's part, round, store.  Runs once per token, so it is kept
          // as a short loop (its code runs cold) rather than unrolled.
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t o[16];
            tmem_ld_16x2_x16(tmem + lane_base + kColO + 16 * c4, o);
            float x[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 v4 = split > 1 ? xo[128 * (4 * c4 + q)] : make_float4(0.f, 0.f, 0.f, 0.f);
              x[4 * q] = v4.x;
              x[4 * q + 1] = v4.y;
              x[4 * q + 2] = v4.z;
              x[4 * q + 3] = v4.w;
            }
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int d = 8 * q + 2 * e;
                const float y0 = fmaf(__uint_as_float(o[d]), f0, x[d] * f1);
                const float y1 = fmaf(__uint_as_float(o[d + 1]), f0, x[d + 1] * f1);
                pk[e] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y0))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(y1))) << 16);
              }
              dst[2 * c4 + q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(oempty);
        }
      }
    }
  }

  // a CTA whose part had no compressed tile never waited for the previous
  // kernel: it does so before leaving, so that this kernel completes after it
  if (p.early) pdl_wait();
  tc_fence_before();
  __syncthreads();
  // neither CTA of a cluster leaves while the other may still arrive on its barriers
  if (split > 1) cluster_sync();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

bool encode_rows(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows) {
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

size_t attn_smem_bytes() { return AttnSmem::total + 1024; }

// 2-CTA clusters of this kernel that fit on the GPU at once (0 if unknown).
int max_pair_clusters() {
  static int cached[64];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!done[dev]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = attn_smem_bytes();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mqa_umma_kernel<false>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cached[dev] = n;
    done[dev] = true;
  }
  return cached[dev];
}

// CTAs per token: 2 (a cluster pair, each CTA half of the token's tiles) when
// every token can have its own pair at once, else 1 (whole tokens, one CTA per
// SM at most).
int attn_split(const sa_index_args &ia, int TPT) {
  if (TPT < 2) return 1;
  return ia.T <= max_pair_clusters() ? 2 : 1;
}

}  // namespace

bool attn_umma_supported(const sa_attn_args &aa) { return aa.H == kH && aa.D == kD; }

// The tensor-core attention keeps no scratch in global memory (split tokens
// hand their partials over in distributed shared memory).
size_t attn_umma_scratch(const sa_index_args &, const sa_attn_args &, int) { return 0; }

cudaError_t launch_sparse_mqa_umma(const sa_index_args &ia, const sa_attn_args &aa, const int32_t *idx, int K,
                                   void *out, void *, bool inputs_ready, uint32_t *status, cudaStream_t stream) {
  if (ia.T == 0) return cudaSuccess;
  AttnUmmaParams p;
  p.B = ia.B;
  p.T = ia.T;
  p.N_c = ia.N_c;
  p.r = ia.r;
  p.W = aa.W;
  p.R = aa.R;
  p.K = K;
  p.wseq = static_cast<int>(w_rows_per_seq(aa));
  p.cseq = static_cast<int>(c_rows_per_seq(ia, aa));
  p.WT = (aa.W + kTile - 1) / kTile;
  p.TPT = p.WT + (K + kTile - 1) / kTile;
  p.q_seq = ia.q_seq;
  p.q_pos = ia.q_pos;
  p.idx = idx;
  p.sink = aa.sink;
  p.qk_scale = aa.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.Vw = static_cast<const __nv_bfloat16 *>(aa.Vw);
  p.Vc = static_cast<const __nv_bfloat16 *>(aa.Vc);
  p.status = status;
  CUtensorMap qmap, kwmap, kcmap, vwmap, vcmap;
  if (!encode_rows(&qmap, aa.Q, static_cast<uint64_t>(ia.T) * kH, 16) ||
      !encode_rows(&kwmap, aa.Kw, static_cast<uint64_t>(ia.B - 1) * p.wseq + aa.R, 1) ||
      !encode_rows(&kcmap, aa.Kc, static_cast<uint64_t>(ia.B - 1) * p.cseq + ia.N_c, 1) ||
      !encode_rows(&vwmap, aa.Vw, static_cast<uint64_t>(ia.B - 1) * p.wseq + aa.R, 1) ||
      !encode_rows(&vcmap, aa.Vc, static_cast<uint64_t>(ia.B - 1) * p.cseq + ia.N_c, 1))
    return cudaErrorInvalidValue;
  const size_t smem = attn_smem_bytes();
  const long long budget = attn_wait_budget();
  const bool short_budget = budget > 0 && budget < kWaitBudgetCycles;
  auto kern = short_budget ? sparse_mqa_umma_kernel<true> : sparse_mqa_umma_kernel<false>;
  // the register split above assumes the kernel launches with kLaunchRegs
  // registers per thread; anything else could leave a raise waiting forever
  static int regs[2] = {-1, -1};
  if (regs[short_budget] < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void *>(kern));
    if (e != cudaSuccess) return e;
    regs[short_budget] = fa.numRegs;
  }
  if (regs[short_budget] != kLaunchRegs) return cudaErrorInvalidConfiguration;
  static bool attr_done[2][64] = {};
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), smem, attr_done[short_budget]);
  if (e != cudaSuccess) return e;
  if (short_budget) {  // the occupancy query of attn_split runs on the default kernel
    static bool attr_done_default[64] = {};
    e = set_smem_once(reinterpret_cast<const void *>(sparse_mqa_umma_kernel<false>), smem, attr_done_default);
    if (e != cudaSuccess) return e;
  }
  p.split = attn_split(ia, p.TPT);
  p.evict_first = ia.T <= ia.B ? 1 : 0;
  p.early = inputs_ready ? 1 : 0;
  p.budget = short_budget ? budget : kWaitBudgetCycles;
  p.PT0 = (p.TPT + 1) / 2;  // rank 0 takes the larger half (window included); rank 1's hand-off costs about its merge
  const int sms = sm_count();
  // whole tokens (at most one CTA per SM), or one cluster pair per token
  const int grid = p.split == 1 ? (ia.T < sms ? ia.T : sms) : 2 * ia.T;
  // a programmatic dependent launch: CTAs that find a free SM set up (barriers,
  // tensor memory) while the top-k kernel finishes, and wait for it before
  // reading the indices
  return launch_ex(true, kern, dim3(grid), dim3(kThreads), smem, stream, p.split, qmap, kwmap, kcmap, vwmap, vcmap, p);
}

}  // namespace sa
