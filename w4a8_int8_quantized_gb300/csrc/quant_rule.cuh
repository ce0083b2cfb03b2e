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

// Two IEEE fp32 products (or differences), rounded to nearest, with one
// paired instruction: the same results as two scalar operations.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 c;
  asm("{\n.reg .b64 a, b, c;\n"
      "mov.b64 a, {%2, %3};\n"
      "mov.b64 b, {%4, %5};\n"
      "mul.rn.f32x2 c, a, b;\n"
      "mov.b64 {%0, %1}, c;\n}\n"
      : "=f"(c.x), "=f"(c.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return c;
}

__device__ __forceinline__ float2 sub2_rn(float2 a, float2 b) {
  float2 c;
  asm("{\n.reg .b64 a, b, c;\n"
      "mov.b64 a, {%2, %3};\n"
      "mov.b64 b, {%4, %5};\n"
      "sub.rn.f32x2 c, a, b;\n"
      "mov.b64 {%0, %1}, c;\n}\n"
      : "=f"(c.x), "=f"(c.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return c;
}

// The eight codes of one 16-byte vector of fp16 x (scale s, rcp = 1 / s
// correctly rounded, 0 when s == 0), as integral floats in [-qmax, qmax].
// The products and the distances to the nearest integer go two at a time
// (paired fp32 instructions, each half an IEEE operation), and a code is
// near a tie when |t - rint(t)| >= 1/2 - 2^-14: the same test as
// near_half, since 1/2 - |d| is exact for |d| in [1/4, 1/2] and both tests
// fail below 1/4.
__device__ __forceinline__ void quant_vec8(const uint4 &v, float s, float rcp, float (&r)[8]) {
  const __half2 *h = reinterpret_cast<const __half2 *>(&v);
  const float2 rc = make_float2(rcp, rcp);
  float2 t[4];
  bool any_near = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    t[j] = mul2_rn(__half22float2(h[j]), rc);
    r[2 * j] = rintf(t[j].x);
    r[2 * j + 1] = rintf(t[j].y);
    const float2 d = sub2_rn(t[j], make_float2(r[2 * j], r[2 * j + 1]));
    any_near |= fabsf(d.x) >= 0.49993896484375f;  // 1/2 - 2^-14
    any_near |= fabsf(d.y) >= 0.49993896484375f;
  }
  if (any_near) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = __half22float2(h[j]);
      if (near_half(t[j].x, r[2 * j])) r[2 * j] = rintf(__fdiv_rn(x.x, s));
      if (near_half(t[j].y, r[2 * j + 1])) r[2 * j + 1] = rintf(__fdiv_rn(x.y, s));
    }
  }
}

// The eight codes as fp16 values (16 bytes): + 0 turns a -0 code into +0,
// the fp16 value of the integer 0 (two at a time), then two per convert.
__device__ __forceinline__ uint4 pack_h8(const float (&r)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float2 z;
    asm("{\n.reg .b64 a, b, c;\n"
        "mov.b64 a, {%2, %3};\n"
        "mov.b64 b, {%4, %4};\n"
        "add.rn.f32x2 c, a, b;\n"
        "mov.b64 {%0, %1}, c;\n}\n"
        : "=f"(z.x), "=f"(z.y)
        : "f"(r[2 * j]), "f"(r[2 * j + 1]), "f"(0.f));
    const __half2 hh = __floats2half2_rn(z.x, z.y);
    w[j] = *reinterpret_cast<const uint32_t *>(&hh);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

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
