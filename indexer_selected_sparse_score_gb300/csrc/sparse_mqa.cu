// Sparse MQA over the raw window plus the selected compressed rows, with a
// split-KV combine ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
// Attention.forward: kv = cat(window_kv, compress_kv), topk_idxs =
// cat(window_idxs, compress_idxs + offset), sparse_attn(q, kv, attn_sink,
// topk_idxs, softmax_scale); one shared KV head serves every query head).
//
// Two kernels here: the CUDA-core kernel (head dim 128 with head counts other
// than 64; the tcgen05 kernel for 64 heads of dim 128 is in
// sparse_mqa_umma.cu) and, further down, the warp-level MMA kernel for head
// dim 512 (the released V4.1 shape).  Both run one CTA per (token, split).
// The token's key list is its window rows (oldest first) followed by its K
// index slots; a split takes a contiguous chunk of that list.  When K and V
// are one tensor (V4.1's single kv), each row is loaded once and serves as
// both tiles.  Rows are gathered 16 bytes per thread,
// logits and the online softmax run in fp32 in the log2 domain (logits are
// pre-multiplied by scale * log2(e)), and each split leaves (m, l, o) partials
// that the combine kernel merges.  A single split writes the output directly.
#include "common.cuh"
#include "internal.h"

namespace sa {
namespace {

constexpr int kKeyTile = 32;  // keys per tile

// Launch shape of the CUDA-core kernel per head dim: threads per CTA and keys
// per tile (a dim-512 form, 512 threads with 16-key tiles when K and V are
// separate, fits the shared memory; dim 512 is served by the MMA kernel).
template <int D, bool kSameKV>
struct AttnShape {
  static constexpr int kThreads = D == 512 ? 512 : 256;
  static constexpr int kTile = (D == 512 && !kSameKV) ? 16 : kKeyTile;
};

struct AttnParams {
  int B, T, N_c, r;
  const int32_t *q_seq, *q_pos;
  int W, R;
  int wseq, cseq;  // rows between consecutive sequences of the ring and of the compressed cache
  const uint16_t *Q, *Kw, *Vw, *Kc, *Vc;
  const float *sink;
  float qk_scale;  // scale * log2(e)
  const int32_t *idx;
  int K;
  int splits, split_keys;
  float *part_m, *part_l, *part_o;
  __nv_bfloat16 *out;
  uint32_t *status;
};

// Shared-memory rows of Q and K are D + 4 floats apart (16-byte aligned rows
// whose 16-byte chunks fall in distinct banks across 8 consecutive rows), P
// rows KT + 4.
template <int H, int D, bool kSameKV>
constexpr size_t attn_smem_bytes() {
  constexpr int KT = AttnShape<D, kSameKV>::kTile;
  return sizeof(float) * (static_cast<size_t>(H) * (D + 4) + KT * (D + 4) + (kSameKV ? 0 : KT * D) +
                          H * (KT + 4) + 3 * H) +
         sizeof(int) * 2 * KT;
}

template <int H, int D, bool kSameKV>
__global__ void __launch_bounds__(AttnShape<D, kSameKV>::kThreads) sparse_mqa_simt_kernel(AttnParams p) {
  constexpr int kAttnThreads = AttnShape<D, kSameKV>::kThreads;
  constexpr int kKeyTile = AttnShape<D, kSameKV>::kTile;
  constexpr int NPT = H * D / kAttnThreads;
  constexpr int DP = D + 4;
  constexpr int PP = kKeyTile + 4;
  constexpr int VS = kSameKV ? DP : D;  // row stride of the V tile
  // logits: thread = (key j, heads h0 + m * HSTEP); P.V: thread = (column d, heads d0 + e * DSTEP)
  constexpr int HSTEP = kAttnThreads / kKeyTile < H ? kAttnThreads / kKeyTile : H, HPT = H / HSTEP;
  constexpr int DSTEP = kAttnThreads / D;
  static_assert(NPT * kAttnThreads == H * D, "H*D must be a multiple of the CTA size");
  static_assert(HPT * HSTEP == H && kAttnThreads % kKeyTile == 0, "logit blocking");
  static_assert(kAttnThreads % D == 0 && kKeyTile % 4 == 0, "P.V blocking");
  extern __shared__ float4 smem4[];
  float *Qs = reinterpret_cast<float *>(smem4);     // [H][DP]
  float *Ks = Qs + H * DP;                          // [kKeyTile][DP]
  float *Vs = kSameKV ? Ks : Ks + kKeyTile * DP;    // [kKeyTile][VS]
  float *Ps = Ks + kKeyTile * DP + (kSameKV ? 0 : kKeyTile * D);  // [H][PP]
  float *m_s = Ps + H * PP;
  float *l_s = m_s + H;
  float *c_s = l_s + H;
  int *row_of = reinterpret_cast<int *>(c_s + H);  // [kKeyTile] row in its source, -1 = none
  int *src_of = row_of + kKeyTile;                 // [kKeyTile] 0 = window ring, 1 = compressed

  const int t = blockIdx.y, split = blockIdx.x, tid = threadIdx.x;
  Token tk;
  const bool ok = load_token(p.q_seq, p.q_pos, t, p.B, p.N_c, p.r, p.status, tk,
                             split == 0 && tid == 0);
  const int n_w = ok ? min(p.W, tk.pos + 1) : 0;
  const int n_keys = ok ? n_w + p.K : 0;
  const int k_begin = split * p.split_keys;
  const int k_end = min(k_begin + p.split_keys, n_keys);

  const int64_t qbase = static_cast<int64_t>(t) * H * D;
  for (int i = tid; i < H * D; i += kAttnThreads)
    Qs[(i / D) * DP + (i % D)] = bf16_bits_to_float(p.Q[qbase + i]) * p.qk_scale;
  for (int h = tid; h < H; h += kAttnThreads) {
    m_s[h] = -INFINITY;
    l_s[h] = 0.f;
  }
  float acc[NPT];
#pragma unroll
  for (int e = 0; e < NPT; ++e) acc[e] = 0.f;
  __syncthreads();

  for (int tile = k_begin; tile < k_end; tile += kKeyTile) {
    if (tid < kKeyTile) {
      const int kk = tile + tid;
      int row = -1, src = 0;
      if (kk < k_end) {
        if (kk < n_w) {
          const int pos = tk.pos - n_w + 1 + kk;
          row = tk.b * p.wseq + pos % p.R;
        } else {
          const int c = p.idx[static_cast<int64_t>(t) * p.K + (kk - n_w)];
          if (c >= 0 && c < tk.nv) {
            row = tk.b * p.cseq + c;
            src = 1;
          } else if (c != -1) {
            raise_flag(p.status, kFlagBadIndex);
          }
        }
      }
      row_of[tid] = row;
      src_of[tid] = src;
    }
    __syncthreads();
    constexpr int CH = D / 8;  // 16-byte chunks per row
    for (int i = tid; i < kKeyTile * CH; i += kAttnThreads) {
      const int j = i / CH, c = i % CH;
      const int row = row_of[j];
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (row >= 0) {
        const uint16_t *kb = src_of[j] ? p.Kc : p.Kw;
        kv = __ldg(reinterpret_cast<const uint4 *>(kb + static_cast<int64_t>(row) * D) + c);
        if constexpr (!kSameKV) {
          const uint16_t *vb = src_of[j] ? p.Vc : p.Vw;
          vv = __ldg(reinterpret_cast<const uint4 *>(vb + static_cast<int64_t>(row) * D) + c);
        }
      }
      const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
      const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        Ks[j * DP + 8 * c + 2 * e] = __uint_as_float(kw[e] << 16);
        Ks[j * DP + 8 * c + 2 * e + 1] = __uint_as_float(kw[e] & 0xFFFF0000u);
        if constexpr (!kSameKV) {
          Vs[j * D + 8 * c + 2 * e] = __uint_as_float(vw[e] << 16);
          Vs[j * D + 8 * c + 2 * e + 1] = __uint_as_float(vw[e] & 0xFFFF0000u);
        }
      }
    }
    __syncthreads();
    if (tid / kKeyTile < HSTEP) {
      // each 16-byte chunk of key j's row serves HPT heads (threads past HSTEP
      // rows of keys have no heads left and skip this)
      const int j = tid % kKeyTile, h0 = tid / kKeyTile;
      float dot[HPT];
#pragma unroll
      for (int m = 0; m < HPT; ++m) dot[m] = 0.f;
      const float *kj = Ks + j * DP;
#pragma unroll 4
      for (int d = 0; d < D; d += 4) {
        const float4 kv = *reinterpret_cast<const float4 *>(kj + d);
#pragma unroll
        for (int m = 0; m < HPT; ++m) {
          const float4 qv = *reinterpret_cast<const float4 *>(Qs + (h0 + m * HSTEP) * DP + d);
          float a = dot[m];
          a = fmaf(qv.x, kv.x, a);
          a = fmaf(qv.y, kv.y, a);
          a = fmaf(qv.z, kv.z, a);
          a = fmaf(qv.w, kv.w, a);
          dot[m] = a;
        }
      }
      const bool live = row_of[j] >= 0;
#pragma unroll
      for (int m = 0; m < HPT; ++m) Ps[(h0 + m * HSTEP) * PP + j] = live ? dot[m] : -INFINITY;
    }
    __syncthreads();
    for (int h = tid; h < H; h += kAttnThreads) {
      float mx = -INFINITY;
      for (int j = 0; j < kKeyTile; ++j) mx = fmaxf(mx, Ps[h * PP + j]);
      const float m_old = m_s[h];
      const float m_new = fmaxf(m_old, mx);
      float corr = 1.f, sum = 0.f;
      if (m_new != -INFINITY) {
        corr = exp2f(m_old - m_new);
        for (int j = 0; j < kKeyTile; ++j) {
          const float pj = exp2f(Ps[h * PP + j] - m_new);
          Ps[h * PP + j] = pj;
          sum += pj;
        }
      } else {
        for (int j = 0; j < kKeyTile; ++j) Ps[h * PP + j] = 0.f;
      }
      l_s[h] = l_s[h] * corr + sum;
      m_s[h] = m_new;
      c_s[h] = corr;
    }
    __syncthreads();
    {
      // each V element serves the thread's NPT heads; P comes four keys at a time
      const int d = tid % D, hb = tid / D;
#pragma unroll
      for (int e = 0; e < NPT; ++e) acc[e] *= c_s[hb + e * DSTEP];
#pragma unroll 1
      for (int j = 0; j < kKeyTile; j += 4) {
        const float v0 = Vs[j * VS + d], v1 = Vs[(j + 1) * VS + d];
        const float v2 = Vs[(j + 2) * VS + d], v3 = Vs[(j + 3) * VS + d];
#pragma unroll
        for (int e = 0; e < NPT; ++e) {
          const float4 pp = *reinterpret_cast<const float4 *>(Ps + (hb + e * DSTEP) * PP + j);
          float a = acc[e];
          a = fmaf(pp.x, v0, a);
          a = fmaf(pp.y, v1, a);
          a = fmaf(pp.z, v2, a);
          a = fmaf(pp.w, v3, a);
          acc[e] = a;
        }
      }
    }
    __syncthreads();
  }

  if (p.splits == 1) {
#pragma unroll
    for (int e = 0; e < NPT; ++e) {
      const int el = tid + e * kAttnThreads;
      const int h = el / D;
      const float m = m_s[h];
      const float s2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
      const float M = fmaxf(m, s2);
      float o = 0.f;
      if (M != -INFINITY) {
        const float a = exp2f(m - M);
        const float L = l_s[h] * a + (p.sink ? exp2f(s2 - M) : 0.f);
        o = acc[e] * a / L;
      }
      p.out[qbase + el] = __float2bfloat16_rn(o);
    }
  } else {
    for (int h = tid; h < H; h += kAttnThreads) {
      const int64_t pi = (static_cast<int64_t>(t) * H + h) * p.splits + split;
      p.part_m[pi] = m_s[h];
      p.part_l[pi] = l_s[h];
    }
#pragma unroll
    for (int e = 0; e < NPT; ++e) {
      const int el = tid + e * kAttnThreads;
      const int h = el / D, d = el % D;
      const int64_t pi = (static_cast<int64_t>(t) * H + h) * p.splits + split;
      p.part_o[pi * D + d] = acc[e];
    }
  }
}

// out[t,h,:] = sum_s 2^(m_s - M) o_s / (sum_s 2^(m_s - M) l_s + 2^(sink - M)),
// M the largest of the m_s and the sink (all in the log2 domain).
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(int H, int S, const float *__restrict__ part_m,
                                                    const float *__restrict__ part_l,
                                                    const float *__restrict__ part_o,
                                                    const float *__restrict__ sink,
                                                    __nv_bfloat16 *__restrict__ out) {
  const int th = blockIdx.x;  // t * H + h
  const int h = th % H, d = threadIdx.x;
  const float *pm = part_m + static_cast<int64_t>(th) * S;
  const float *pl = part_l + static_cast<int64_t>(th) * S;
  const float *po = part_o + static_cast<int64_t>(th) * S * D;
  const float s2 = sink ? sink[h] * kLog2e : -INFINITY;
  float M = s2;
  for (int s = 0; s < S; ++s) M = fmaxf(M, pm[s]);
  float o = 0.f;
  if (M != -INFINITY) {
    float L = sink ? exp2f(s2 - M) : 0.f, acc = 0.f;
    for (int s = 0; s < S; ++s) {
      const float a = exp2f(pm[s] - M);  // 0 for an empty split (m = -inf)
      L = fmaf(a, pl[s], L);
      acc = fmaf(a, po[static_cast<int64_t>(s) * D + d], acc);
    }
    o = acc / L;
  }
  out[static_cast<int64_t>(th) * D + d] = __float2bfloat16_rn(o);
}

template <int H, int D, bool kSameKV>
cudaError_t launch_attn(const AttnParams &p, cudaStream_t stream) {
  auto kern = sparse_mqa_simt_kernel<H, D, kSameKV>;
  constexpr size_t smem = attn_smem_bytes<H, D, kSameKV>();
  static_assert(smem <= 227 * 1024, "shared memory of one CTA");
  static bool attr_done[64] = {};
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), smem, attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, p.T);
  kern<<<grid, AttnShape<D, kSameKV>::kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  combine_kernel<D><<<p.T * H, D, 0, stream>>>(H, p.splits, p.part_m, p.part_l, p.part_o, p.sink,
                                               p.out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Head dim 512 (the released V4.1 shape) on the warp-level bf16 tensor-core MMA
// (mma.sync m16n8k16, fp32 accumulate).  One CTA of 16 warps per (token,
// split), 32 keys per tile:
//  - Q (bf16, unscaled) stays in shared memory; each tile's K rows (and V rows,
//    unless K and V are one tensor) are gathered into shared memory as bf16 by
//    cp.async, into one of two buffers while the other tile is computed;
//  - S = Q K^T: warp w owns the 16 x 8 block of heads 16 (w / 4).. and keys
//    8 (w % 4).. (fewer than 64 heads leave warps idle here), 32 MMAs over the
//    512 dims; the logits, scaled into the log2 domain, go to shared memory;
//  - the online softmax (one warp per head, a lane per key) writes P as two bf16 parts,
//    P = hi + lo with |P - hi - lo| < 2^-16 P, so P.V keeps fp32-level accuracy;
//  - O += P V: warp w owns the heads of one 16-row block and a run of 8-column
//    blocks of the 512 dims; its accumulators stay in registers across tiles,
//    rescaled by the softmax correction; V fragments come by ldmatrix.trans.
constexpr int kMmaThreads = 512;
constexpr int kMmaD = 512;
constexpr int kMmaKT = 32;
constexpr int kQS = kMmaD + 8;   // bf16 row stride of the Q, K and V tiles (1040 bytes)
constexpr int kSS = kMmaKT + 4;  // fp32 row stride of S
constexpr int kPS = kMmaKT + 8;  // bf16 row stride of P hi and lo (80 bytes)

template <int H, bool kSameKV>
struct Mma512Layout {
  static constexpr size_t tile = sizeof(uint16_t) * kMmaKT * kQS;  // one K (or V) tile
  static constexpr size_t q = 0;
  static constexpr size_t k = q + sizeof(uint16_t) * H * kQS;       // two K buffers
  static constexpr size_t v = k + 2 * tile;                         // two V buffers (separate V)
  static constexpr size_t s = v + (kSameKV ? 0 : 2 * tile);
  static constexpr size_t phi = s + sizeof(float) * H * kSS;
  static constexpr size_t plo = phi + sizeof(uint16_t) * H * kPS;
  static constexpr size_t ms = plo + sizeof(uint16_t) * H * kPS;
  static constexpr size_t rows = ms + sizeof(float) * 3 * H;
  static constexpr size_t total = rows + sizeof(int) * 4 * kMmaKT;  // row ids per buffer
};

// 16-byte global -> shared copy; with valid false it writes 16 zero bytes and
// reads nothing (src must still be a mapped address).
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t &r0, uint32_t &r1, const void *smem_row) {
  const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(smem_row));
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

template <int H, bool kSameKV>
__global__ void __launch_bounds__(kMmaThreads) sparse_mqa_mma512_kernel(AttnParams p) {
  using Lay = Mma512Layout<H, kSameKV>;
  constexpr int D = kMmaD, KT = kMmaKT;
  constexpr int MT = H / 16;          // 16-row blocks of heads
  constexpr int WPM = 16 / MT;        // warps per head block in P.V
  constexpr int NTW = (D / 8) / WPM;  // 8-column blocks per warp in P.V
  static_assert(MT * 16 == H && WPM * MT == 16 && NTW * WPM * 8 == D, "warp split");
  extern __shared__ float4 smem4[];
  char *sm = reinterpret_cast<char *>(smem4);
  uint16_t *Qb = reinterpret_cast<uint16_t *>(sm + Lay::q);
  uint16_t *Kbuf = reinterpret_cast<uint16_t *>(sm + Lay::k);                        // [2][KT][kQS]
  uint16_t *Vbuf = kSameKV ? Kbuf : reinterpret_cast<uint16_t *>(sm + Lay::v);     // [2][KT][kQS]
  float *Sf = reinterpret_cast<float *>(sm + Lay::s);
  uint16_t *Phi = reinterpret_cast<uint16_t *>(sm + Lay::phi);
  uint16_t *Plo = reinterpret_cast<uint16_t *>(sm + Lay::plo);
  float *m_s = reinterpret_cast<float *>(sm + Lay::ms);
  float *l_s = m_s + H;
  float *c_s = l_s + H;
  int *rows_buf = reinterpret_cast<int *>(sm + Lay::rows);  // [2][KT] row ids, then [2][KT] sources
  int *srcs_buf = rows_buf + 2 * KT;

  const int t = blockIdx.y, split = blockIdx.x, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, q4 = lane & 3;
  Token tk;
  const bool ok = load_token(p.q_seq, p.q_pos, t, p.B, p.N_c, p.r, p.status, tk, split == 0 && tid == 0);
  const int n_w = ok ? min(p.W, tk.pos + 1) : 0;
  const int n_keys = ok ? n_w + p.K : 0;
  const int k_begin = split * p.split_keys;
  const int k_end = min(k_begin + p.split_keys, n_keys);

  const int64_t qbase = static_cast<int64_t>(t) * H * D;
  for (int i = tid; i < H * (D / 8); i += kMmaThreads) {  // 16-byte chunks of Q
    const int h = i / (D / 8), c = i % (D / 8);
    *reinterpret_cast<uint4 *>(Qb + h * kQS + 8 * c) =
        __ldg(reinterpret_cast<const uint4 *>(p.Q + qbase + static_cast<int64_t>(h) * D) + c);
  }
  for (int h = tid; h < H; h += kMmaThreads) {
    m_s[h] = -INFINITY;
    l_s[h] = 0.f;
  }
  // P.V ownership: head block pm, column blocks pn0 .. pn0 + NTW - 1
  const int pm = warp / WPM, pn0 = (warp % WPM) * NTW;
  float acc[NTW][4];
#pragma unroll
  for (int i = 0; i < NTW; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
  __syncthreads();

  // row ids of a tile (threads below KT), then its rows copied into buffer b
  auto tile_rows = [&](int tile, int b) {
    const int kk = tile + tid;
    int row = -1, src = 0;
    if (kk < k_end) {
      if (kk < n_w) {
        const int pos = tk.pos - n_w + 1 + kk;
        row = tk.b * p.wseq + pos % p.R;
      } else {
        const int c = p.idx[static_cast<int64_t>(t) * p.K + (kk - n_w)];
        if (c >= 0 && c < tk.nv) {
          row = tk.b * p.cseq + c;
          src = 1;
        } else if (c != -1) {
          raise_flag(p.status, kFlagBadIndex);
        }
      }
    }
    rows_buf[b * KT + tid] = row;
    srcs_buf[b * KT + tid] = src;
  };
  auto tile_copy = [&](int b) {
    for (int i = tid; i < KT * (D / 8); i += kMmaThreads) {  // 16 bytes at a time; empty slots read as 0
      const int j = i / (D / 8), c = i % (D / 8);
      const int row = rows_buf[b * KT + j];
      const bool valid = row >= 0;
      const int64_t off = static_cast<int64_t>(valid ? row : 0) * D + 8 * c;
      const bool comp = srcs_buf[b * KT + j] != 0;
      cp_async16_zfill(Kbuf + (b * KT + j) * kQS + 8 * c, (comp ? p.Kc : p.Kw) + off, valid);
      if constexpr (!kSameKV) cp_async16_zfill(Vbuf + (b * KT + j) * kQS + 8 * c, (comp ? p.Vc : p.Vw) + off, valid);
    }
    cp_async_commit();
  };
  if (k_begin < k_end) {
    if (tid < KT) tile_rows(k_begin, 0);
    __syncthreads();
    tile_copy(0);
  }

  for (int tile = k_begin, it = 0; tile < k_end; tile += KT, ++it) {
    const int b = it & 1;
    if (tile + KT < k_end) {  // the next tile's copies go out before this one is computed
      if (tid < KT) tile_rows(tile + KT, b ^ 1);
      __syncthreads();
      tile_copy(b ^ 1);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_group<0>();
    }
    __syncthreads();  // every thread's copies of this tile are in
    const uint16_t *Kb = Kbuf + b * KT * kQS;
    const uint16_t *Vb = Vbuf + b * KT * kQS;
    const int *row_of = rows_buf + b * KT;
    if (warp < MT * (KT / 8)) {  // S block: heads 16 smt .., keys 8 snt ..
      const int smt = warp / (KT / 8), snt = warp % (KT / 8);
      // four accumulators over interleaved 16-dim steps: four short MMA chains, summed at the end
      float cc[4][4] = {};
      const uint16_t *qa = Qb + (16 * smt + g) * kQS + 2 * q4;
      const uint16_t *kbp = Kb + (8 * snt + g) * kQS + 2 * q4;
#pragma unroll 2
      for (int k0 = 0; k0 < D / 16; k0 += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ks = k0 + u;
          const uint32_t a[4] = {ld_u32(qa + 16 * ks), ld_u32(qa + 8 * kQS + 16 * ks), ld_u32(qa + 16 * ks + 8),
                                 ld_u32(qa + 8 * kQS + 16 * ks + 8)};
          mma_bf16_16816(cc[u], a, ld_u32(kbp + 16 * ks), ld_u32(kbp + 16 * ks + 8));
        }
      }
      float c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] = (cc[0][e] + cc[1][e]) + (cc[2][e] + cc[3][e]);
      const int h0 = 16 * smt + g, j0 = 8 * snt + 2 * q4;
      const bool v0 = row_of[j0] >= 0, v1 = row_of[j0 + 1] >= 0;
      Sf[h0 * kSS + j0] = v0 ? c[0] * p.qk_scale : -INFINITY;
      Sf[h0 * kSS + j0 + 1] = v1 ? c[1] * p.qk_scale : -INFINITY;
      Sf[(h0 + 8) * kSS + j0] = v0 ? c[2] * p.qk_scale : -INFINITY;
      Sf[(h0 + 8) * kSS + j0 + 1] = v1 ? c[3] * p.qk_scale : -INFINITY;
    }
    __syncthreads();
    for (int h = warp; h < H; h += kMmaThreads / 32) {  // online softmax: a warp per head, a lane per key
      const float sv = Sf[h * kSS + lane];
      float mx = sv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = m_s[h];
      const float m_new = fmaxf(m_old, mx);
      const float pj = m_new != -INFINITY ? exp2f(sv - m_new) : 0.f;
      float sum = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      const __nv_bfloat16 hi = __float2bfloat16_rn(pj);
      const __nv_bfloat16 lo = __float2bfloat16_rn(pj - __bfloat162float(hi));
      Phi[h * kPS + lane] = __bfloat16_as_ushort(hi);
      Plo[h * kPS + lane] = __bfloat16_as_ushort(lo);
      if (lane == 0) {
        const float corr = m_new != -INFINITY ? exp2f(m_old - m_new) : 1.f;
        l_s[h] = l_s[h] * corr + sum;
        m_s[h] = m_new;
        c_s[h] = corr;
      }
    }
    __syncthreads();
    {
      const int r0 = 16 * pm + g;
      const float cr0 = c_s[r0], cr1 = c_s[r0 + 8];
#pragma unroll
      for (int i = 0; i < NTW; ++i) {
        acc[i][0] *= cr0;
        acc[i][1] *= cr0;
        acc[i][2] *= cr1;
        acc[i][3] *= cr1;
      }
#pragma unroll
      for (int ks = 0; ks < KT / 16; ++ks) {
        const uint16_t *ph = Phi + r0 * kPS + 16 * ks + 2 * q4;
        const uint16_t *pl = Plo + r0 * kPS + 16 * ks + 2 * q4;
        const uint32_t ahi[4] = {ld_u32(ph), ld_u32(ph + 8 * kPS), ld_u32(ph + 8), ld_u32(ph + 8 * kPS + 8)};
        const uint32_t alo[4] = {ld_u32(pl), ld_u32(pl + 8 * kPS), ld_u32(pl + 8), ld_u32(pl + 8 * kPS + 8)};
        // lanes 0-15 address rows 16 ks + (lane & 15) of V (lanes 16-31 repeat them)
        const uint16_t *vrow = Vb + (16 * ks + (lane & 15)) * kQS;
#pragma unroll
        for (int i = 0; i < NTW; ++i) {
          uint32_t b0, b1;
          ldmatrix_x2_trans(b0, b1, vrow + 8 * (pn0 + i));
          mma_bf16_16816(acc[i], ahi, b0, b1);
          mma_bf16_16816(acc[i], alo, b0, b1);
        }
      }
    }
    __syncthreads();
  }

  const int r0 = 16 * pm + g;
  if (p.splits == 1) {
    float sc[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int h = r0 + 8 * half;
      const float m = m_s[h];
      const float s2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
      const float M = fmaxf(m, s2);
      sc[half] = 0.f;
      if (M != -INFINITY) {
        const float a = exp2f(m - M);
        const float L = l_s[h] * a + (p.sink ? exp2f(s2 - M) : 0.f);
        sc[half] = a / L;
      }
    }
#pragma unroll
    for (int i = 0; i < NTW; ++i) {
      const int d = 8 * (pn0 + i) + 2 * q4;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int64_t o = qbase + static_cast<int64_t>(r0 + 8 * half) * D + d;
        p.out[o] = __float2bfloat16_rn(acc[i][2 * half] * sc[half]);
        p.out[o + 1] = __float2bfloat16_rn(acc[i][2 * half + 1] * sc[half]);
      }
    }
  } else {
    for (int h = tid; h < H; h += kMmaThreads) {
      const int64_t pi = (static_cast<int64_t>(t) * H + h) * p.splits + split;
      p.part_m[pi] = m_s[h];
      p.part_l[pi] = l_s[h];
    }
#pragma unroll
    for (int i = 0; i < NTW; ++i) {
      const int d = 8 * (pn0 + i) + 2 * q4;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int64_t pi = (static_cast<int64_t>(t) * H + r0 + 8 * half) * p.splits + split;
        p.part_o[pi * D + d] = acc[i][2 * half];
        p.part_o[pi * D + d + 1] = acc[i][2 * half + 1];
      }
    }
  }
}

template <int H, bool kSameKV>
cudaError_t launch_attn_mma512(const AttnParams &p, cudaStream_t stream) {
  auto kern = sparse_mqa_mma512_kernel<H, kSameKV>;
  constexpr size_t smem = Mma512Layout<H, kSameKV>::total;
  static_assert(smem <= 227 * 1024, "shared memory of one CTA");
  static bool attr_done[64] = {};
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kern), smem, attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, p.T);
  kern<<<grid, kMmaThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.splits == 1) return e;
  combine_kernel<kMmaD><<<p.T * H, kMmaD, 0, stream>>>(H, p.splits, p.part_m, p.part_l, p.part_o, p.sink, p.out);
  return cudaGetLastError();
}

}  // namespace

bool attn_shape_supported(int H, int D) {
  return (D == 128 && (H == 16 || H == 32 || H == 64 || H == 128)) ||
         (D == 512 && (H == 16 || H == 32 || H == 64));
}

int fused_launch_count(const sa_index_args &ia, const sa_attn_args &aa, int K,
                       const SplitPlan &plan) {
  const int score = idx_score_umma_supported(ia) ? 2 : 1;  // (query packing +) scoring
  const int topk = K > 0 ? 1 : 0;
  const int attn = (attn_umma_supported(aa) || attn_umma512_supported(aa)) ? 1 : (plan.splits > 1 ? 2 : 1);
  return ia.T > 0 ? score + topk + attn : 0;
}

SplitPlan plan_splits(int T, int W, int K) {
  const int n_keys = W + K;
  const int max_splits = (n_keys + kKeyTile - 1) / kKeyTile;
  const int target_ctas = 2 * 152;
  int splits = T > 0 ? (target_ctas + T - 1) / T : 1;
  splits = splits < 1 ? 1 : (splits > max_splits ? max_splits : splits);
  int split_keys = (n_keys + splits - 1) / splits;
  split_keys = (split_keys + kKeyTile - 1) / kKeyTile * kKeyTile;
  splits = (n_keys + split_keys - 1) / split_keys;
  return SplitPlan{splits < 1 ? 1 : splits, split_keys < kKeyTile ? kKeyTile : split_keys};
}

cudaError_t launch_sparse_mqa(const sa_index_args &ia, const sa_attn_args &aa, const int32_t *idx,
                              int K, void *out, float *part_m, float *part_l, float *part_o,
                              void *attn_scratch, const SplitPlan &plan, bool inputs_ready, uint32_t *status,
                              cudaStream_t stream) {
  if (ia.T == 0) return cudaSuccess;
  if (attn_umma_supported(aa))
    return launch_sparse_mqa_umma(ia, aa, idx, K, out, attn_scratch, inputs_ready, status, stream);
  if (attn_umma512_supported(aa))
    return launch_sparse_mqa_umma512(ia, aa, idx, K, out, inputs_ready, status, stream);
  AttnParams p;
  p.B = ia.B;
  p.T = ia.T;
  p.N_c = ia.N_c;
  p.r = ia.r;
  p.q_seq = ia.q_seq;
  p.q_pos = ia.q_pos;
  p.W = aa.W;
  p.R = aa.R;
  p.wseq = static_cast<int>(w_rows_per_seq(aa));
  p.cseq = static_cast<int>(c_rows_per_seq(ia, aa));
  p.Q = static_cast<const uint16_t *>(aa.Q);
  p.Kw = static_cast<const uint16_t *>(aa.Kw);
  p.Vw = static_cast<const uint16_t *>(aa.Vw);
  p.Kc = static_cast<const uint16_t *>(aa.Kc);
  p.Vc = static_cast<const uint16_t *>(aa.Vc);
  p.sink = aa.sink;
  p.qk_scale = aa.scale * kLog2e;
  p.idx = idx;
  p.K = K;
  p.splits = plan.splits;
  p.split_keys = plan.split_keys;
  p.part_m = part_m;
  p.part_l = part_l;
  p.part_o = part_o;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.status = status;
  // one tensor for K and V (the window ring and the compressed cache alike)
  const bool same = aa.Kw == aa.Vw && aa.Kc == aa.Vc;
  if (aa.D == 512) {  // warp-level bf16 MMA
    switch (aa.H) {
      case 16: return same ? launch_attn_mma512<16, true>(p, stream) : launch_attn_mma512<16, false>(p, stream);
      case 32: return same ? launch_attn_mma512<32, true>(p, stream) : launch_attn_mma512<32, false>(p, stream);
      case 64: return same ? launch_attn_mma512<64, true>(p, stream) : launch_attn_mma512<64, false>(p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (aa.H) {
    case 16: return same ? launch_attn<16, 128, true>(p, stream) : launch_attn<16, 128, false>(p, stream);
    case 32: return same ? launch_attn<32, 128, true>(p, stream) : launch_attn<32, 128, false>(p, stream);
    case 64: return same ? launch_attn<64, 128, true>(p, stream) : launch_attn<64, 128, false>(p, stream);
    case 128: return same ? launch_attn<128, 128, true>(p, stream) : launch_attn<128, 128, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sa
