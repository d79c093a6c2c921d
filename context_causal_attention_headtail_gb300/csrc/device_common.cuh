// Device helpers shared by the kernels: HeadTail geometry, accurate RoPE
// angles, and the bounded-wait clock.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

namespace cpattn {

// Natural chunk index kappa of the `half` (0 = head, 1 = tail) chunk of rank r.
__device__ __forceinline__ int chunk_of(int r, int half, int cp) {
  return half == 0 ? r : 2 * cp - 1 - r;
}
// (rank, half) owning natural chunk kappa.
__device__ __forceinline__ void owner_of(int kappa, int cp, int &r, int &half) {
  if (kappa < cp) { r = kappa; half = 0; } else { r = 2 * cp - 1 - kappa; half = 1; }
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded waits give up after this long and raise ERR_FLAG_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// cos/sin of pos * theta, theta = th_hi + th_lo, accurate to ~1e-6 rad for
// pos < 2^24. The product is formed as a float pair (exact FMA residual) and
// reduced modulo 2*pi with a three-part Cody-Waite split of 2*pi
// (6.28125 + 1.9353071693331003e-3 + 1.0253376273028358e-11): 6.28125 has
// 8 significant bits, so k * 6.28125 is exact for the k that occur here.
// The reduced angle |r| <= pi(1 + small) then goes to sincosf.
__device__ __forceinline__ void rope_sincos(int pos, float th_hi, float th_lo, float &s, float &c) {
  const float p = (float)pos;
  const float a_hi = p * th_hi;
  const float a_lo = fmaf(p, th_hi, -a_hi) + p * th_lo;
  const float k = rintf(a_hi * 0.159154943091895336f);
  float r = fmaf(-k, 6.28125f, a_hi);
  r = fmaf(-k, 1.9353071693331003e-3f, r);
  r = fmaf(-k, 1.0253376273028358e-11f, r);
  r += a_lo;
  sincosf(r, &s, &c);
}

// The same reduction with the reduced angle on the MUFU sin/cos units
// (absolute error ~2^-21 for |r| <= pi), for seeds that are recomputed often.
__device__ __forceinline__ void rope_sincos_fast(int pos, float th_hi, float th_lo, float &s, float &c) {
  const float p = (float)pos;
  const float a_hi = p * th_hi;
  const float a_lo = fmaf(p, th_hi, -a_hi) + p * th_lo;
  const float k = rintf(a_hi * 0.159154943091895336f);
  float r = fmaf(-k, 6.28125f, a_hi);
  r = fmaf(-k, 1.9353071693331003e-3f, r);
  r = fmaf(-k, 1.0253376273028358e-11f, r);
  r += a_lo;
  __sincosf(r, &s, &c);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
// Round two floats to bf16 (RNE) and pack: lo in bits 0..15, hi in 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace cpattn
