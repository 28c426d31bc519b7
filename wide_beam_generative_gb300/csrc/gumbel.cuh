// Gumbel noise for temperature > 0 (device side).
//
// "Deploying FlashRec" (serving parameters): temperature 0 is deterministic
// top-k; above 0 the selection is Gumbel top-k, the noise only orders the
// candidates and the returned sequence score leaves it out.  Ordering key of
// a candidate with score s: fl32(fl32(s * inv_tau) + g), g ~ Gumbel(0, 1)
// drawn for (request r, step t, beam b, token v):
//   word0 of Philox4x32-10 (Salmon, Moraes, Dror and Shaw, SC 2011) at
//   counter (v, b, r, t), key (seed low 32 bits, seed high 32 bits);
//   u = ((word0 >> 9) + 1/2) * 2^-23 (exact in float32, never 0 or 1),
//   g = -ln(-ln(u)).
// ln is computed here in float32 with every operation rounded to nearest and
// none fused, in a fixed order, so that any other implementation of the same
// steps takes identical ordering decisions: x = m * 2^e, m in
// [sqrt(1/2), sqrt(2)), ln m = 2 atanh(z) = 2 (z + z^3/3 + z^5/5 + z^7/7 +
// z^9/9) with z = (m - 1) / (m + 1) (Abramowitz and Stegun 4.1.27),
// ln x = e * ln 2 + ln m.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bd {

__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int rnd = 0; rnd < 10; ++rnd) {
    if (rnd) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

// ln of a positive normal float (see the notes above).
__device__ __forceinline__ float ln_f32(float x) {
  const uint32_t bits = __float_as_uint(x);
  int e = (int)((bits >> 23) & 0xFFu) - 127;
  float m = __uint_as_float((bits & 0x7FFFFFu) | (127u << 23));   // [1, 2)
  if (m > 1.41421353816986083984375f) {   // float32 nearest to sqrt(2)
    m = __fmul_rn(m, 0.5f);
    e += 1;
  }
  const float z = __fdiv_rn(__fsub_rn(m, 1.f), __fadd_rn(m, 1.f));
  const float z2 = __fmul_rn(z, z);
  float p = 0.111111111f;                                            // fl32(1/9)
  p = __fadd_rn(__fmul_rn(p, z2), 0.142857143f);                     // fl32(1/7)
  p = __fadd_rn(__fmul_rn(p, z2), 0.2f);                             // fl32(1/5)
  p = __fadd_rn(__fmul_rn(p, z2), 0.333333343f);                     // fl32(1/3)
  p = __fadd_rn(__fmul_rn(p, z2), 1.f);
  const float lnm = __fmul_rn(__fmul_rn(2.f, z), p);
  return __fadd_rn(__fmul_rn((float)e, 0.693147182f), lnm);          // fl32(ln 2)
}

__device__ __forceinline__ float gumbel_noise(uint32_t seed_lo, uint32_t seed_hi, int r, int t, int b,
                                              int v) {
  const uint32_t w = philox_word0((uint32_t)v, (uint32_t)b, (uint32_t)r, (uint32_t)t, seed_lo, seed_hi);
  const float u = __fmul_rn(__fadd_rn((float)(w >> 9), 0.5f), 1.1920928955078125e-7f);   // 2^-23
  return -ln_f32(-ln_f32(u));
}

}  // namespace bd
