// The symmetric quantization rule, shared by the row quantizer and the
// fused decode kernel (one definition, so both give the same codes).
//
// Rounding: q = clamp(rint(x / s), -qmax, qmax) with x / s one IEEE fp32
// division.  The kernel evaluates t = x * (1/s) with a correctly rounded
// reciprocal: |t - x/s| <= |x/s| (2^-23 + 2^-48) and the IEEE quotient is
// within |x/s| 2^-24 of x/s, so with |x/s| <= 127.01 the two differ by less
// than 2.3e-5.  When t is farther than 2^-14 from every half-integer, both
// lie strictly on the same side of the same half-integer and round to the
// same integer; only the rare t within 2^-14 of a half-integer takes the
// IEEE division itself.  The result is bit-identical to the plain rule.
//
// The clamp never acts: s = fl(a / qmax) for the group's absmax a, so every
// |x| <= a gives |x / s| <= qmax (1 + 2^-23) and |t| < qmax + 1/2, which
// rounds to at most qmax.  The codes are therefore computed without it.
#pragma once

#include <cuda_fp16.h>

namespace w8a8 {

__device__ __forceinline__ float absmax8(const uint4 &v) {
  const __half2 *h = reinterpret_cast<const __half2 *>(&v);
  __half2 m = __habs2(h[0]);
  m = __hmax2(m, __habs2(h[1]));
  m = __hmax2(m, __habs2(h[2]));
  m = __hmax2(m, __habs2(h[3]));
  return fmaxf(__low2float(m), __high2float(m));
}

// t within 2^-14 of a half-integer: t and x / s might round differently
__device__ __forceinline__ bool near_half(float t, float r) {
  return 0.5f - fabsf(t - r) <= 6.103515625e-05f;
}

// The eight codes of one 16-byte vector of fp16 x (scale s, rcp = 1 / s
// correctly rounded, 0 when s == 0), as integral floats in [-qmax, qmax].
__device__ __forceinline__ void quant_vec8(const uint4 &v, float s, float rcp, float (&r)[8]) {
  const __half2 *h = reinterpret_cast<const __half2 *>(&v);
  float x[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = __half22float2(h[j]);
    x[2 * j] = f.x;
    x[2 * j + 1] = f.y;
  }
  bool any_near = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float t = __fmul_rn(x[i], rcp);
    r[i] = rintf(t);
    any_near |= near_half(t, r[i]);
  }
  if (any_near) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float t = __fmul_rn(x[i], rcp);
      if (near_half(t, rintf(t))) r[i] = rintf(__fdiv_rn(x[i], s));
    }
  }
}

// eight integral float codes -> eight bytes (two's complement), low byte first
__device__ __forceinline__ uint2 pack_i8x8(const float (&r)[8]) {
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t b0 = static_cast<uint32_t>(__float2int_rn(r[4 * h])) & 0xffu;
    const uint32_t b1 = static_cast<uint32_t>(__float2int_rn(r[4 * h + 1])) & 0xffu;
    const uint32_t b2 = static_cast<uint32_t>(__float2int_rn(r[4 * h + 2])) & 0xffu;
    const uint32_t b3 = static_cast<uint32_t>(__float2int_rn(r[4 * h + 3])) & 0xffu;
    w[h] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
  }
  return make_uint2(w[0], w[1]);
}

}  // namespace w8a8
