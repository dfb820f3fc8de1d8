// NVFP4 helpers of the CUDA path: E4M3 scale encode/decode, E2M1 code
// selection, and the 16-element block quantiser shared by the activation
// quantiser and the NVFP4 SwiGLU epilogue of the grouped GEMM; the
// 32-element MX block quantiser of the MX SwiGLU epilogue.
//
// Format ("Driving vLLM WideEP and Large-Scale Serving Toward Maturity on
// Blackwell (Part I)", sections "NVFP4 GEMM for MoE and O-proj" and "NVFP4
// MoE dispatch"): packed E2M1 codes, one E4M3 scale per 16 elements, one fp32
// global scale g.  Recipe (IEEE fp32, round to nearest even):
//   s = E4M3_satfinite(amax16 / (6 g)),  q_i = E2M1_satfinite(x_i / (e4m3(s) g))
// with magnitude 0 when e4m3(s) == 0 and the code's sign bit = sign of x_i.
#pragma once

#include "common.cuh"

namespace moe {

// fp32 -> E4M3 byte: round to nearest even, saturate to the largest finite
// value (448).  Uses the hardware conversion.
DEVINL uint32_t e4m3_encode_satfinite(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v), "f"(v));
  return static_cast<uint32_t>(r) & 0xFFu;
}

// E4M3 byte -> fp32 (exact).  code (e<<3)|m: e == 0 -> m * 2^-9, else
// (8 + m) * 2^(e - 10); bit 7 is the sign.
DEVINL float e4m3_decode(uint32_t b) {
  uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
  return (b & 0x80u) ? -v : v;
}

// Magnitude code of a non-negative ratio: nearest of {0,.5,1,1.5,2,3,4,6},
// ties to the even code, saturating at 6.  The decision points are the
// midpoints between neighbours; at a midpoint the even code wins, which makes
// the comparison strict (>) where the lower neighbour's code is even and
// inclusive (>=) where it is odd.
DEVINL uint32_t e2m1_magnitude(float a) {
  return static_cast<uint32_t>(a > 0.25f) + static_cast<uint32_t>(a >= 0.75f) +
         static_cast<uint32_t>(a > 1.25f) + static_cast<uint32_t>(a >= 1.75f) +
         static_cast<uint32_t>(a > 2.5f) + static_cast<uint32_t>(a >= 3.5f) + static_cast<uint32_t>(a > 5.0f);
}

// A quotient q with the same E2M1 code as the correctly rounded RN(x / d)
// (d > 0), with one multiply in the common case, given r = RN(1 / d).  The
// product q = RN(x * r) carries two roundings of at most 2^-24 relative
// each and RN(x / d) one, so they lie within 4 ulp of q of each other; they
// can then round to different E2M1 codes only if a decision point of the
// E2M1 grid (a midpoint between neighbouring magnitudes: 0.25, 0.75, 1.25,
// 1.75, 2.5, 3.5, 5) lies within those 4 ulp.  Each decision point has at
// most three significant bits, so its low 21 mantissa bits are zero: when
// the low 21 mantissa bits of q are more than 8 away from a multiple of
// 2^21, no decision point is that close and q is returned.  Otherwise (and
// when q is not finite: d so small that r overflows) the quotient is formed
// by an IEEE division.
DEVINL float e2m1_quotient(float x, float d, float r) {
  const float q = __fmul_rn(x, r);
  if (((__float_as_uint(q) + 8u) & 0x1FFFFFu) <= 16u || !(fabsf(q) < INFINITY)) return __fdiv_rn(x, d);
  return q;
}

// Eight fp32 values -> eight E2M1 codes (element i in nibble i), round to
// nearest with ties to the even code, saturating to +-6, sign kept (the
// hardware conversion).
DEVINL uint32_t e2m1x8_rn_satfinite(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Quantise 16 fp32 values with global scale g.  Returns the E4M3 scale byte;
// codes[0] holds elements 0..7 (element 2j in the low nibble of byte j),
// codes[1] elements 8..15.  Bit for bit the recipe above with an IEEE
// division per element (see e2m1_quotient).
DEVINL uint32_t nvfp4_quantize16(const float (&v)[16], float g, uint32_t (&codes)[2]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t s = e4m3_encode_satfinite(__fdiv_rn(amax, __fmul_rn(6.0f, g)));
  const float denom = __fmul_rn(e4m3_decode(s), g);
  const float r = denom != 0.0f ? __frcp_rn(denom) : 0.0f;
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    q[i] = denom != 0.0f ? e2m1_quotient(v[i], denom, r) : copysignf(0.0f, v[i]);  // magnitude 0 if denom == 0
  codes[0] = e2m1x8_rn_satfinite(q);
  codes[1] = e2m1x8_rn_satfinite(q + 8);
  return s;
}

// One MX block of 32 fp32 values (moe_quant_mx's recipe): E8M0 scale
// exponent e = floor(log2 amax) - emax (emax 2 for E2M1, 8 for E4M3),
// clamped to [-127, 127], read from the abs-max's exponent field (a zero or
// subnormal abs-max gives -127); elements RNE_satfinite(v * 2^-e) with the
// sign kept.  2^-e is a normal fp32 because a finite amax has exponent
// field <= 254, so the scaling is exact unless the product underflows.
// Returns the E8M0 byte; codes: FP4 -> 4 words of packed E2M1 (element 2j
// in the low nibble of byte j), FP8 -> 8 words of E4M3 bytes.
template <bool FP4>
DEVINL uint32_t mx_quantize32(const float (&v)[32], uint32_t (&codes)[FP4 ? 4 : 8]) {
  constexpr int EMAX = FP4 ? 2 : 8;
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = max(-127, min(127, static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - EMAX));
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
  for (int w = 0; w < (FP4 ? 4 : 8); ++w) codes[w] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float x = v[i] * inv;
    if (FP4) {
      const uint32_t code = e2m1_magnitude(fabsf(x)) | ((__float_as_uint(v[i]) >> 31) << 3);
      codes[i >> 3] |= code << (4 * (i & 7));
    } else {
      codes[i >> 2] |= e4m3_encode_satfinite(x) << (8 * (i & 3));
    }
  }
  return static_cast<uint32_t>(e + 127);
}

// bf16 bit pattern of each E2M1 code (sign in bit 3).
DEVINL uint32_t e2m1_to_bf16_bits(uint32_t code) {
  // magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
  const uint32_t mag = code & 7u;
  uint32_t bits = 0u;
  switch (mag) {
    case 0: bits = 0x0000u; break;
    case 1: bits = 0x3F00u; break;
    case 2: bits = 0x3F80u; break;
    case 3: bits = 0x3FC0u; break;
    case 4: bits = 0x4000u; break;
    case 5: bits = 0x4040u; break;
    case 6: bits = 0x4080u; break;
    default: bits = 0x40C0u; break;
  }
  return bits | ((code & 8u) << 12);
}

}  // namespace moe
