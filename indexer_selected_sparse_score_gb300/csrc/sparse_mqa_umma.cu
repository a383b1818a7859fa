// Sparse MQA on the 5th-generation tensor cores (tcgen05) for 64 query heads
// of dim 128 sharing one KV head ("DeepSeek-V4.1-Flash-NVFP4
// inference/model.py", Attention.forward: sparse_attn over the window rows
// and the index-selected compressed rows).
//
// Each token's key list is its window (padded to a multiple of 128) followed
// by its K index slots (padded likewise); every token therefore has the same
// number of 128-key tiles, and the persistent CTAs split the flattened
// (token, tile) list evenly.  Per tile:
//   S = Q K^T      M = 128 (the 64 heads; rows 64..127 unused), N = 128 keys,
//                  K = 128, bf16 x bf16 -> f32 in tensor memory;
//   softmax        one thread per (head, half of the keys), exp2 in fp32 with a
//                  lazily raised running maximum (rescale O only when the
//                  tile maximum exceeds the reference by more than 2^8);
//   O += P V       P from tensor memory as a bf16 hi + lo pair (two MMAs into
//                  the same accumulator, p = hi + lo to 2^-16), V read
//                  MN-major from the gathered tile, M = 128, N = 128 (d),
//                  K = 128 keys.
// K and V rows are gathered by index with TMA gather4 (4 rows of 128 bytes per
// instruction) into the 128-byte-swizzled layout both MMAs read.
//
// Warps: 0, 1, 4, 5 softmax (heads 0-31 / 32-63 x key halves 0-63 / 64-127);
// 3 MMA issuer and tensor-memory owner; 2 and 6-11 producers: each of these
// seven warps resolves the rows of its share of a tile's 128 gather4 copies
// and issues them (one warp alone issues gathers at well under the HBM rate,
// seven together come close to it); warp 2 also loads each token's Q and
// writes the tile's key mask.  A token whose tiles all fall in one CTA is finished there; a token
// split across CTAs leaves one (m, l, O) record per piece for the combine
// kernel.  Every wait is bounded; on expiry the kernel flags the status word,
// drains its copies and MMAs, and returns.
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
constexpr int kStages = 3;        // K/V tile stages
constexpr int kThreads = 384;
constexpr int kGatherWarps = 7;   // warp 2 and warps 6..11
constexpr float kLazyRescale = 8.f;  // log2 units
constexpr int kRecFloats = 2 * kH + kH * kD;

constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP = 384;  // tensor-memory columns

// Q: two token buffers of 64 rows share one 32 KB region, [kblk][buf][64 rows
// x 128 B]: the MMA reads 128 rows (M = 128) from each buffer's base, and rows
// 64..127 (the other buffer, or the first K stage right after) only feed the
// unused accumulator rows 64..127.
struct AttnSmem {
  static constexpr size_t q = 0;                                   // [2 kblk][2 buf][64 rows][128 B]
  static constexpr size_t k = q + 32768;                           // [stage][2 kblk][128 rows][128 B]
  static constexpr size_t v = k + kStages * 32768;
  static constexpr size_t mask = v + kStages * 32768;              // [stage][4] u32
  static constexpr size_t xchg = mask + kStages * 4 * 4;           // [2 parity][2 halves][64] f32
  static constexpr size_t bars = (xchg + 4 * kH * 4 + 7) & ~size_t(7);
  static constexpr int kBars = 2 * kStages + 4 + 4 + 2 + 2 + 1 + 2;
  static constexpr size_t misc = bars + kBars * 8;
  static constexpr size_t total = misc + 64;
};

struct AttnUmmaParams {
  int B, T, N_c, r, W, R, K;
  int WT, TPT;                    // window tiles per token, tiles per token
  const int32_t *q_seq, *q_pos, *idx;
  const float *sink;
  float qk_scale;                 // scale * log2(e)
  __nv_bfloat16 *out;
  float *rec;                     // [grid][2][kRecFloats]
  uint32_t *status;
};

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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
                                        int y2, int y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
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

__device__ __forceinline__ int tile_begin(long long total, int c, int G) {
  return static_cast<int>(total * c / G);
}

// Record slot of the piece of token-range [t0, t1) that CTA c processed.
__device__ __forceinline__ float *record(const AttnUmmaParams &p, int c, int slot) {
  return p.rec + (static_cast<size_t>(c) * 2 + slot) * kRecFloats;
}

__global__ void __launch_bounds__(kThreads, 1)
sparse_mqa_umma_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kwmap,
                       const __grid_constant__ CUtensorMap vwmap, const __grid_constant__ CUtensorMap kcmap,
                       const __grid_constant__ CUtensorMap vcmap, const AttnUmmaParams p) {
  using L = AttnSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *ks = smem + L::k, *vs = smem + L::v, *qs = smem + L::q;
  uint32_t *mask_s = reinterpret_cast<uint32_t *>(smem + L::mask);
  float *xchg = reinterpret_cast<float *>(smem + L::xchg);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
  uint64_t *kvfull = bars, *kvempty = bars + kStages;
  uint64_t *qfull = bars + 2 * kStages, *qempty = qfull + 2;
  uint64_t *sfull = qempty + 2, *sempty = sfull + 2;
  uint64_t *pfull = sempty + 2, *pempty = pfull + 1;
  uint64_t *ofull = pempty + 1, *oempty = ofull + 1;
  uint64_t *done = oempty + 1;
  uint64_t *xbar = done + 1;  // [2]: one per head quarter, pairs the two key-half warps
  uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem + L::misc);
  int *abort_s = reinterpret_cast<int *>(smem + L::misc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long total = static_cast<long long>(p.T) * p.TPT;
  const int G = gridDim.x, c = blockIdx.x;
  const int begin = tile_begin(total, c, G), end = tile_begin(total, c + 1, G);

  // zero the operand buffers once: rows never written by a copy stay finite
  for (int i = tid; i < static_cast<int>(L::mask / 16); i += kThreads)
    reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
  static_assert(L::total + 1024 <= 232448, "shared memory budget");
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kvfull[i], kGatherWarps);
      mbar_init(&kvempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], 1);
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], 4);
    }
    mbar_init(pfull, 4);
    mbar_init(pempty, 1);
    mbar_init(ofull, 1);
    mbar_init(oempty, 4);
    mbar_init(done, 1);
    mbar_init(&xbar[0], 2);
    mbar_init(&xbar[1], 2);
    *abort_s = 0;
    fence_barrier_init();
  }
  if (warp == 3) {
    tmem_alloc(tmem_base_s, 512);
    tmem_relinquish();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  auto fail = [&]() {
    raise_flag(p.status, kFlagTimeout);
    atomicExch(abort_s, 1);
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int *>(abort_s) != 0; };

  if (warp == 2 || warp >= 6) {
    // --------------------------------------------------------------- producers
    const int pw = (warp == 2) ? 0 : warp - 5;  // 0 .. 6
    if (begin < end) {
      if (warp == 2 && lane == 0) {
        prefetch_tmap(&qmap);
        prefetch_tmap(&kwmap);
        prefetch_tmap(&vwmap);
        prefetch_tmap(&kcmap);
        prefetch_tmap(&vcmap);
      }
      int qn = -1, prev_t = -1, issued = 0;
      Token tk{0, 0, 0};
      bool tok_ok = false;
      int n_w = 0;
      // the key of slot kk (0..127) of tile j: its row and whether it exists
      auto resolve = [&](int t, int j, int kk, int &row) -> bool {
        if (!tok_ok) return false;
        if (j < p.WT) {
          const int q = j * kTile + kk;
          if (q >= n_w) return false;
          const int pos = tk.pos - n_w + 1 + q;
          row = tk.b * p.R + pos % p.R;
          return true;
        }
        const int k = (j - p.WT) * kTile + kk;
        if (k >= p.K) return false;
        const int cidx = p.idx[static_cast<int64_t>(t) * p.K + k];
        if (cidx >= 0 && cidx < tk.nv) {
          row = tk.b * p.N_c + cidx;
          return true;
        }
        if (cidx != -1 && warp == 2) raise_flag(p.status, kFlagBadIndex);
        return false;
      };
      for (int i = begin; i < end && !aborted(); ++i) {
        const int t = i / p.TPT, j = i % p.TPT, n = i - begin;
        if (t != prev_t) {
          tok_ok = load_token(p.q_seq, p.q_pos, t, p.B, p.N_c, p.r, p.status, tk,
                              warp == 2 && lane == 0 && j == 0);
          n_w = tok_ok ? min(p.W, tk.pos + 1) : 0;
          ++qn;
          if (warp == 2) {
            const int qb = qn & 1;
            bool ok = true;
            if (lane == 0) {
              ok = mbar_wait(&qempty[qb], ((qn >> 1) & 1) ^ 1);
              if (ok) {
                mbar_expect_tx(&qfull[qb], 2 * kH * 128);
                tma_load_2d(qs + qb * 8192, &qmap, &qfull[qb], 0, t * kH);
                tma_load_2d(qs + 16384 + qb * 8192, &qmap, &qfull[qb], 64, t * kH);
              } else {
                fail();
              }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
          }
          prev_t = t;
        }
        const int s = n % kStages;
        if (!mbar_wait_warp(&kvempty[s], ((n / kStages) & 1) ^ 1)) {
          if (lane == 0) fail();
          break;
        }
        const bool window = j < p.WT;
        if (warp == 2) {  // key mask of the tile: bit g of word e = key 4g+e exists
          int row_unused = 0;
          uint32_t m4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) m4[e] = __ballot_sync(0xffffffffu, resolve(t, j, 4 * lane + e, row_unused));
          if (lane == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) mask_s[s * 4 + e] = m4[e];
          }
        }
        // this warp's share of the 128 copies: copy c = (part, group), part =
        // K lo / K hi / V lo / V hi, group g = keys 4g..4g+3
        uint32_t bytes = 0;
        const int c0 = lane * kGatherWarps + pw;
        int rows[4] = {0, 0, 0, 0};
        bool any = false;
        if (c0 < 128) {
          const int g = c0 & 31;
          bool valid[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) valid[e] = resolve(t, j, 4 * g + e, rows[e]);
          any = valid[0] || valid[1] || valid[2] || valid[3];
          const int fill = valid[0] ? rows[0] : valid[1] ? rows[1] : valid[2] ? rows[2] : rows[3];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (!valid[e]) rows[e] = fill;
        }
        bytes = __popc(__ballot_sync(0xffffffffu, any)) * 512u;
        if (lane == 0) mbar_expect_tx(&kvfull[s], bytes);
        __syncwarp();
        if (any) {
          const int g = c0 & 31, part = c0 >> 5;
          const CUtensorMap *map = (part < 2) ? (window ? &kwmap : &kcmap) : (window ? &vwmap : &vcmap);
          uint8_t *dst = ((part < 2) ? ks : vs) + s * 32768 + (part & 1) * 16384 + 4 * g * 128;
          gather4(dst, map, &kvfull[s], (part & 1) * 64, rows[0], rows[1], rows[2], rows[3]);
        }
        ++issued;
      }
      if (warp == 2 && lane == 0) {  // drain: every issued copy lands before the CTA exits
        for (int n = max(0, issued - kStages); n < issued; ++n) mbar_wait(&kvfull[n % kStages], (n / kStages) & 1);
        for (int q = max(0, qn - 1); q <= qn; ++q) mbar_wait(&qfull[q & 1], (q >> 1) & 1);
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------- MMA issuer
    // Issues S for tile n+1 and P.V for tile n in whichever order their inputs
    // become ready (polling), so P.V never waits for the next tile's data.
    if (lane == 0 && begin < end) {
      constexpr uint32_t idesc_s = idesc_bf16(128, kTile);              // K-major A, K-major B
      constexpr uint32_t idesc_o = idesc_bf16(128, kD) | (1u << 16);     // K-major A (tmem), MN-major B
      const int count = end - begin;
      int ns = 0, np = 0;            // next S to issue, next P.V to issue
      int qn_s = -1, prev_t_s = -1;  // token ordinal as seen by the S stage
      int sg = -1;                   // segment ordinal as seen by the P.V stage
      bool q_ready = false;
      long long idle_since = clock64();
      bool ok = true;
      while (np < count) {
        if (aborted()) { ok = false; break; }
        bool progressed = false;
        // ---- S(ns): Q of its token, its K tile and a free S buffer
        if (ns < count && ns <= np + 1) {
          const int i = begin + ns, t = i / p.TPT, j = i % p.TPT;
          if (t != prev_t_s) {
            if (!q_ready && mbar_try_wait(&qfull[(qn_s + 1) & 1], ((qn_s + 1) >> 1) & 1)) q_ready = true;
          }
          const bool q_ok = (t == prev_t_s) || q_ready;
          const int s = ns % kStages, sb = ns & 1;
          if (q_ok && mbar_try_wait(&kvfull[s], (ns / kStages) & 1) &&
              mbar_try_wait(&sempty[sb], ((ns >> 1) & 1) ^ 1)) {
            if (t != prev_t_s) {
              ++qn_s;
              prev_t_s = t;
              q_ready = false;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(qs + (qn_s & 1) * 8192), b0 = smem_u32(ks + s * 32768);
            const uint32_t d = tmem + (sb ? kColS1 : kColS0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_f16(d, desc_sw128_kmajor(a0 + off), desc_sw128_kmajor(b0 + off), idesc_s, kk > 0);
            }
            mma_commit(&sfull[sb]);
            if ((j == p.TPT - 1) || (i == end - 1)) mma_commit(&qempty[qn_s & 1]);
            ++ns;
            progressed = true;
          }
        }
        // ---- P.V(np): P from the softmax (and O read out after the previous segment)
        if (np < ns) {
          const int i = begin + np, j = i % p.TPT;
          const bool first = (j == 0) || (np == 0);
          const bool last = (j == p.TPT - 1) || (i == end - 1);
          const bool o_ok = !first || sg < 0 || mbar_try_wait(oempty, sg & 1);
          if (o_ok && mbar_try_wait(pfull, np & 1)) {
            if (first) ++sg;
            tc_fence_after();
            const int s = np % kStages;
            const uint32_t v0 = smem_u32(vs + s * 32768);
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_f16_ta(tmem + kColO, tmem + kColP + 64 * half + 8 * kk,
                           desc_sw128_mnmajor(v0 + kk * 2048, 16384), idesc_o, !(first && half == 0 && kk == 0));
            mma_commit(&kvempty[s]);
            mma_commit(pempty);
            if (last) mma_commit(ofull);
            ++np;
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = clock64();
        } else if (clock64() - idle_since > kWaitBudgetCycles) {
          ok = false;
          break;
        }
      }
      if (!ok) fail();
      mma_commit(done);
      if (!mbar_wait(done, 0)) raise_flag(p.status, kFlagTimeout);
    }
  } else {
    // ----------------------------------------------------------------- softmax
    const int hq = warp & 1;                 // head quarter: 0 -> heads 0..31, 1 -> 32..63
    const int kh = warp >> 2;                // key half: 0 -> keys 0..63, 1 -> 64..127
    const int h = 32 * hq + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * hq) << 16;
    // value exchange with the partner warp (same heads, other key half):
    // double-buffered slots, one mbarrier phase per exchange, bounded wait
    int xk = 0;
    auto swap = [&](float val, float &partner) -> bool {
      xchg[((xk & 1) * 2 + kh) * kH + h] = val;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[hq]);
      const bool ok = mbar_wait_warp(&xbar[hq], xk & 1);
      partner = xchg[((xk & 1) * 2 + (kh ^ 1)) * kH + h];
      ++xk;
      return ok;
    };
    float m_ref = -INFINITY, l_part = 0.f;
    int sg = -1, seg_start = 0;
    for (int i = begin; i < end; ++i) {
      const int n = i - begin, t = i / p.TPT, j = i % p.TPT;
      const bool first = (j == 0) || (n == 0);
      const bool last = (j == p.TPT - 1) || (i == end - 1);
      if (first) {
        ++sg;
        seg_start = i;
        m_ref = -INFINITY;
        l_part = 0.f;
      }
      const int s = n % kStages, sb = n & 1;
      const bool ok = mbar_wait_warp(&kvfull[s], (n / kStages) & 1) && mbar_wait_warp(&sfull[sb], (n >> 1) & 1);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      uint32_t v[64];  // raw dot products Q.K of this thread's head and keys
      tmem_ld_32x32b_x32(tmem + lane_base + (sb ? kColS1 : kColS0) + 64 * kh,
                         *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld_32x32b_x32(tmem + lane_base + (sb ? kColS1 : kColS0) + 64 * kh + 32,
                         *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      uint32_t m4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) m4[e] = mask_s[s * 4 + e];
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[sb]);
      // Masked keys -> -inf.  The max runs on the raw dot products (the
      // softmax scale is positive) and each logit is scaled and shifted by one
      // FMA inside exp2.  Mask words stride by 4 keys: bit g of word e is key
      // 4g+e; a half of the tile whose 16 groups are all present skips it.
      float mx = -INFINITY;
      const uint32_t all4 = m4[0] & m4[1] & m4[2] & m4[3];
      const uint32_t half_mask = kh ? 0xFFFF0000u : 0x0000FFFFu;
      if ((all4 & half_mask) != half_mask) {
#pragma unroll
        for (int q = 0; q < 64; ++q) {
          const int key = 64 * kh + q;
          if (!((m4[key & 3] >> (key >> 2)) & 1u)) v[q] = 0xFF800000u;  // -inf
        }
      }
#pragma unroll
      for (int q = 0; q < 64; ++q) mx = fmaxf(mx, __uint_as_float(v[q]));
      mx *= p.qk_scale;
      float other;
      if (!swap(mx, other)) {
        if (lane == 0) fail();
        break;
      }
      const float tile_max = fmaxf(mx, other);
      float factor = 1.f;
      bool rescale = false;
      if (first) {
        m_ref = tile_max;
      } else if (tile_max > m_ref + kLazyRescale) {
        factor = exp2f(m_ref - tile_max);
        m_ref = tile_max;
        rescale = true;
      }
      // p = 2^(scale * s - m_ref); P = hi + lo with hi = p truncated to bf16
      // and lo = (p - hi) truncated to bf16 (|p - hi - lo| < 2^-14 p), packed
      // in pairs with byte permutes: no conversion instructions.
      float sum = 0.f;
      uint32_t phi[32], plo[32];
      const float neg_m = -m_ref;
      const bool live = m_ref != -INFINITY;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        float pa = 0.f, pb = 0.f;
        if (live) {
          pa = ex2_approx(fmaf(__uint_as_float(v[2 * q]), p.qk_scale, neg_m));
          pb = ex2_approx(fmaf(__uint_as_float(v[2 * q + 1]), p.qk_scale, neg_m));
        }
        sum += pa + pb;
        const uint32_t ua = __float_as_uint(pa), ub = __float_as_uint(pb);
        const float la = pa - __uint_as_float(ua & 0xFFFF0000u);
        const float lb = pb - __uint_as_float(ub & 0xFFFF0000u);
        phi[q] = __byte_perm(ua, ub, 0x7632);
        plo[q] = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
      }
      l_part = l_part * factor + sum;
      // the previous P.V must be finished before P is overwritten or O rescaled
      if (!mbar_wait_warp(pempty, (n & 1) ^ 1)) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, rescale)) {
        uint32_t o[64];
        tmem_ld_32x32b_x32(tmem + lane_base + kColO + 64 * kh, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tmem_ld_32x32b_x32(tmem + lane_base + kColO + 64 * kh + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 64; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * factor);
        tmem_st_x32(tmem + lane_base + kColO + 64 * kh, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tmem_st_x32(tmem + lane_base + kColO + 64 * kh + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
      }
      tmem_st_x32(tmem + lane_base + kColP + 32 * kh, phi);
      tmem_st_x32(tmem + lane_base + kColP + 64 + 32 * kh, plo);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull);

      if (last) {
        if (!mbar_wait_warp(ofull, sg & 1)) {
          if (lane == 0) fail();
          break;
        }
        tc_fence_after();
        uint32_t o[64];
        tmem_ld_32x32b_x32(tmem + lane_base + kColO + 64 * kh, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tmem_ld_32x32b_x32(tmem + lane_base + kColO + 64 * kh + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(oempty);
        float l_other;
        if (!swap(l_part, l_other)) {
          if (lane == 0) fail();
          break;
        }
        const float l = l_part + l_other;
        const int t0 = t * p.TPT;
        const bool whole = (seg_start == t0) && (i == t0 + p.TPT - 1);
        if (whole) {
          float Lden = l;
          float a = 1.f;
          if (p.sink) {
            const float s2 = p.sink[h] * kLog2e;
            const float M = fmaxf(m_ref, s2);
            a = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - M);
            Lden = l * a + exp2f(s2 - M);
          }
          const float inv = Lden > 0.f ? a / Lden : 0.f;
          uint4 *dst = reinterpret_cast<uint4 *>(p.out + (static_cast<int64_t>(t) * kH + h) * kD + 64 * kh);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat16 lo = __float2bfloat16_rn(__uint_as_float(o[8 * q + 2 * e]) * inv);
              const __nv_bfloat16 hi = __float2bfloat16_rn(__uint_as_float(o[8 * q + 2 * e + 1]) * inv);
              pk[e] = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
                      (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
            }
            dst[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        } else {
          const int slot = (seg_start == begin) ? 0 : 1;
          float *rec = record(p, c, slot);
          if (kh == 0) {
            rec[h] = m_ref;
            rec[kH + h] = l;
          }
          float4 *od = reinterpret_cast<float4 *>(rec + 2 * kH + h * kD + 64 * kh);
#pragma unroll
          for (int q = 0; q < 16; ++q)
            od[q] = make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merges the records of every token split across CTAs, one block per
// (token, head): out = sum_r 2^(m_r - M) O_r / (sum_r 2^(m_r - M) l_r +
// 2^(sink - M)).
__global__ void __launch_bounds__(kD) attn_umma_combine_kernel(const AttnUmmaParams p, int G) {
  const int t = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const long long total = static_cast<long long>(p.T) * p.TPT;
  const long long first_tile = static_cast<long long>(t) * p.TPT, last_tile = first_tile + p.TPT - 1;
  auto cta_of = [&](long long i) {
    int cc = static_cast<int>(i * G / total);
    while (cc + 1 < G && tile_begin(total, cc + 1, G) <= i) ++cc;
    while (cc > 0 && tile_begin(total, cc, G) > i) --cc;
    return cc;
  };
  const int c0 = cta_of(first_tile), c1 = cta_of(last_tile);
  if (c0 == c1) return;  // finished inside one CTA
  auto slot_of = [&](int cc) { return (cc == c0 && tile_begin(total, cc, G) < first_tile) ? 1 : 0; };
  float M = p.sink ? p.sink[h] * kLog2e : -INFINITY;
  for (int cc = c0; cc <= c1; ++cc) M = fmaxf(M, record(p, cc, slot_of(cc))[h]);
  float o = 0.f;
  if (M != -INFINITY) {
    float Lden = p.sink ? exp2f(p.sink[h] * kLog2e - M) : 0.f, acc = 0.f;
    for (int cc = c0; cc <= c1; ++cc) {
      const float *rec = record(p, cc, slot_of(cc));
      const float a = exp2f(rec[h] - M);
      Lden = fmaf(a, rec[kH + h], Lden);
      acc = fmaf(a, rec[2 * kH + h * kD + d], acc);
    }
    o = Lden > 0.f ? acc / Lden : 0.f;
  }
  p.out[(static_cast<int64_t>(t) * kH + h) * kD + d] = __float2bfloat16_rn(o);
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

}  // namespace

bool attn_umma_supported(const sa_attn_args &aa) { return aa.H == kH && aa.D == kD; }

int attn_umma_grid(const sa_index_args &ia, const sa_attn_args &aa, int K) {
  const int WT = (aa.W + kTile - 1) / kTile, KT = (K + kTile - 1) / kTile;
  const long long total = static_cast<long long>(ia.T) * (WT + KT);
  const int sms = sm_count();
  return static_cast<int>(total < sms ? total : sms);
}

size_t attn_umma_scratch(const sa_index_args &ia, const sa_attn_args &aa, int K) {
  return static_cast<size_t>(attn_umma_grid(ia, aa, K)) * 2 * kRecFloats * sizeof(float);
}

cudaError_t launch_sparse_mqa_umma(const sa_index_args &ia, const sa_attn_args &aa, const int32_t *idx, int K,
                                   void *out, void *scratch, uint32_t *status, cudaStream_t stream) {
  if (ia.T == 0) return cudaSuccess;
  AttnUmmaParams p;
  p.B = ia.B;
  p.T = ia.T;
  p.N_c = ia.N_c;
  p.r = ia.r;
  p.W = aa.W;
  p.R = aa.R;
  p.K = K;
  p.WT = (aa.W + kTile - 1) / kTile;
  p.TPT = p.WT + (K + kTile - 1) / kTile;
  p.q_seq = ia.q_seq;
  p.q_pos = ia.q_pos;
  p.idx = idx;
  p.sink = aa.sink;
  p.qk_scale = aa.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.rec = static_cast<float *>(scratch);
  p.status = status;
  CUtensorMap qmap, kwmap, vwmap, kcmap, vcmap;
  if (!encode_rows(&qmap, aa.Q, static_cast<uint64_t>(ia.T) * kH, kH) ||
      !encode_rows(&kwmap, aa.Kw, static_cast<uint64_t>(ia.B) * aa.R, 1) ||
      !encode_rows(&vwmap, aa.Vw, static_cast<uint64_t>(ia.B) * aa.R, 1) ||
      !encode_rows(&kcmap, aa.Kc, static_cast<uint64_t>(ia.B) * ia.N_c, 1) ||
      !encode_rows(&vcmap, aa.Vc, static_cast<uint64_t>(ia.B) * ia.N_c, 1))
    return cudaErrorInvalidValue;
  const int G = attn_umma_grid(ia, aa, K);
  const size_t smem = AttnSmem::total + 1024;
  static bool attr_done[64] = {};
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(sparse_mqa_umma_kernel), smem, attr_done);
  if (e != cudaSuccess) return e;
  sparse_mqa_umma_kernel<<<G, kThreads, smem, stream>>>(qmap, kwmap, vwmap, kcmap, vcmap, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_umma_combine_kernel<<<dim3(ia.T, kH), kD, 0, stream>>>(p, G);
  return cudaGetLastError();
}

}  // namespace sa
