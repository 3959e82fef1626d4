// E2M1 / E4M3 element codecs of the CUDA path (device side).
//
// Formats: OCP 8-bit floating point E4M3 "FN" (bias 7, largest finite 448,
// S.1111.111 = NaN) and the OCP microscaling E2M1 element (bias 1, magnitudes
// 0, .5, 1, 1.5, 2, 3, 4, 6), as used for the FP4 main-KV cache of the
// "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression" knowledge
// note (section "FP4 main KV: trade precision for bytes, not for a new GEMM").
// Encoders round to nearest with ties to the even code and saturate at the
// largest finite magnitude; the sign bit is copied from the input.
#pragma once

#include <stdint.h>

namespace csa2 {

// |a| (finite, >= 0) -> 7-bit E4M3 magnitude code.
__device__ __forceinline__ uint32_t e4m3_encode_mag(float a) {
  if (a >= 448.0f) return 0x7Eu;
  if (a < 0.015625f) {                       // below 2^-6: subnormal step 2^-9
    return (uint32_t)__float2int_rn(a * 512.0f);   // exact scaling, RNE; 8 -> 2^-6
  }
  const uint32_t u = __float_as_uint(a);
  const int e = (int)((u >> 23) & 0xFFu) - 127;    // -6 .. 8
  const uint32_t mant = u & 0x7FFFFFu;
  uint32_t m3 = mant >> 20;
  const uint32_t rest = mant & 0xFFFFFu;
  if (rest > 0x80000u || (rest == 0x80000u && (m3 & 1u))) m3 += 1u;
  const uint32_t code = ((uint32_t)(e + 7) << 3) + m3;   // a carry moves into the exponent
  return code > 0x7Eu ? 0x7Eu : code;
}

__device__ __forceinline__ uint32_t e4m3_encode(float x) {
  return e4m3_encode_mag(fabsf(x)) | ((__float_as_uint(x) >> 24) & 0x80u);
}

// E4M3 code -> exact fp32 value (NaN codes are never produced by the encoder).
__device__ __forceinline__ float e4m3_decode(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
  return (c & 0x80u) ? -v : v;
}

// Two fp32 values -> one byte of E2M1 codes (lo in bits 0-3, hi in bits
// 4-7): the hardware conversion, round to nearest with ties to the even code
// (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; midpoints 0.25 and 1.25 and 2.5 and
// 5 go down, 0.75 and 1.75 and 3.5 go up), saturating at +-6, sign kept (also
// for values that round to zero).
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint32_t out;
  asm("{\n.reg .b8 t;\ncvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\ncvt.u32.u8 %0, t;\n}"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  return out;
}

// Two fp32 values -> two E4M3 bytes (lo in bits 0-7, hi in bits 8-15): the
// hardware conversion, round to nearest even, saturating at +-448 -- the
// same bytes as e4m3_encode.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint32_t out;
  asm("{\n.reg .b16 t;\ncvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\ncvt.u32.u16 %0, t;\n}"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  return out;
}

// Two E2M1 codes packed in one byte (low nibble first) -> f16x2 (low half
// first).  Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n.reg .b8 t;\ncvt.u8.u32 t, %1;\ncvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(out) : "r"(byte));
  return out;
}

// Two E4M3 bytes (low byte first) -> f16x2 (low half first).  Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n.reg .b16 t;\ncvt.u16.u32 t, %1;\ncvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(out) : "r"(two_bytes));
  return out;
}

}  // namespace csa2
