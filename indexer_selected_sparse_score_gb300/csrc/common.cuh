// Device helpers shared by the kernels of the sparse attention step.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sa {

// Sticky device status flags, OR-ed into the first word of the workspace.
enum : uint32_t {
  kFlagBadSeq = 1u,     // q_seq[t] outside [0, B)
  kFlagBadPos = 2u,     // q_pos[t] < 0 or n_vis(t) > N_c
  kFlagBadIndex = 4u,   // an index outside [-1, n_vis(t))
  kFlagTimeout = 8u,    // a bounded wait gave up
};

__device__ __forceinline__ void raise_flag(uint32_t *status, uint32_t f) {
  if (status) atomicOr(status, f);
}

// Programmatic dependent launch.  The kernels of one call run in a chain
// (query prep -> index scores -> top-k -> attention); each kernel after the
// first is launched so that it may start while its predecessor runs, does its
// set-up, and then pdl_wait()s: that returns once the predecessor has
// completed and its writes are visible (a no-op for an ordinary launch).
// pdl_trigger() lets the successor start; a successor only starts once every
// CTA of this kernel has triggered or exited, i.e. is already resident, so it
// can never hold resources this kernel still needs.  Every CTA of a waiting
// kernel waits, so completion is transitive along the chain.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Visible compressed entries of a token at absolute position p: compressed
// entry j covers tokens [j*r, (j+1)*r) and is visible once p >= (j+1)*r - 1.
__device__ __forceinline__ int n_vis_of(int pos, int r) { return (pos + 1) / r; }

// Validated (sequence, position, n_vis) of token t; returns false (and flags)
// when the token must be skipped.
struct Token {
  int b, pos, nv;
};

__device__ __forceinline__ bool load_token(const int32_t *q_seq, const int32_t *q_pos, int t,
                                           int B, int N_c, int r, uint32_t *status, Token &tk,
                                           bool report) {
  tk.b = q_seq[t];
  tk.pos = q_pos[t];
  if (tk.b < 0 || tk.b >= B) {
    if (report) raise_flag(status, kFlagBadSeq);
    return false;
  }
  if (tk.pos < 0) {
    if (report) raise_flag(status, kFlagBadPos);
    return false;
  }
  tk.nv = n_vis_of(tk.pos, r);
  if (tk.nv > N_c) {
    if (report) raise_flag(status, kFlagBadPos);
    tk.nv = N_c;
  }
  return true;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float e4m3_bits_to_float(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

// Order-preserving map of an fp32 score to uint32 (larger float -> larger
// key); -0 is folded onto +0 so that the two compare equal, as they do in
// floating point.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr float kLog2e = 1.4426950408889634f;

// Division by a runtime divisor d >= 1 with one 64-bit multiply: with
// l = ceil(log2 d) and m = ceil(2^(32+l) / d) (at most 2^33), floor(n / d) =
// (n m) >> (32 + l) for 0 <= n < 2^32 (the round-up multiplier of Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication", 1994:
// m d - 2^(32+l) < d <= 2^l bounds the error below one).  fast_div takes
// n < 2^31, where n m fits in 64 bits.
struct FastDiv {
  uint64_t m;
  int s;
  uint32_t d;  // the divisor
};

__host__ __device__ inline FastDiv make_fastdiv(uint32_t d) {
  int l = 0;
  while ((uint64_t{1} << l) < d) ++l;
  return FastDiv{((uint64_t{1} << (32 + l)) + d - 1) / d, 32 + l, d};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
  return static_cast<uint32_t>((static_cast<uint64_t>(n) * f.m) >> f.s);
}

}  // namespace sa
