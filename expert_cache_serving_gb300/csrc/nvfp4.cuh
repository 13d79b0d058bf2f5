// NVFP4-style quantisation of activations for the FP4 x FP4 prefill GEMMs:
// e2m1 codes with one e4m3 scale per block of 16 consecutive elements along
// the contraction dimension, the format of the FP4 expert weights (FreeToken
// write-up, experimental setup: MXFP4 / NVFP4 experts).
//
// Rule (the same one the weights were produced with): scale = e4m3(amax / 6)
// and code = e2m1(v / scale), each rounded to nearest with ties to the even
// code and saturated to the largest finite value; both divisions are IEEE
// float32 divisions.  A block whose scale rounds to 0 gets codes 0, and a
// value that rounds to magnitude 0 gets code 0 (never 0x8).
#pragma once
#include <cstdint>

namespace moe {

// e4m3 byte of a non-negative float (round to nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3_rn_sat(float v) {
  unsigned short pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(v));  // second operand -> low byte
  return pair & 0xFFu;
}

// Value of an e4m3 byte as a float (exact).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)byte));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Two floats -> one byte of e2m1 codes (lo in the low nibble), round to
// nearest even, saturating at 6; a nibble of magnitude 0 is made +0.
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float lo, float hi) {
  uint32_t b;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(b) : "f"(hi), "f"(lo));
  if ((b & 0x7u) == 0) b &= 0xF0u;
  if ((b & 0x70u) == 0) b &= 0x0Fu;
  return b;
}

// One block of 16 values -> 8 code bytes (element 2i in the low nibble of
// byte i, returned as two little-endian words) and the scale byte.
__device__ __forceinline__ uint32_t quant16(const float* v, uint32_t* c01) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sb = e4m3_rn_sat(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_to_float(sb);
  uint32_t w[2] = {0u, 0u};
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = e2m1x2_rn_sat(__fdiv_rn(v[2 * i], s), __fdiv_rn(v[2 * i + 1], s));
      w[i >> 2] |= b << (8 * (i & 3));
    }
  }
  c01[0] = w[0];
  c01[1] = w[1];
  return sb;
}

}  // namespace moe
