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

// q = clamp(rint(x / s), -qmax, qmax), as described above; rcp = 1 / s
// correctly rounded (0 when s == 0).
__device__ __forceinline__ int quant1(float x, float s, float rcp, int qmax) {
  const float t = __fmul_rn(x, rcp);
  float r = rintf(t);
  const float to_half = 0.5f - fabsf(t - r);  // distance to the nearest half-integer
  if (to_half <= 6.103515625e-05f) r = rintf(__fdiv_rn(x, s));
  const int q = static_cast<int>(r);
  return max(-qmax, min(qmax, q));
}

}  // namespace w8a8
