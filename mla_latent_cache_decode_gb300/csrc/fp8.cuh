// FP8 (OCP E4M3) and f16 conversions used by the FP8-cache path, each one
// hardware cvt instruction:
//  - e4m3 -> f16 is exact (every E4M3 value, subnormals and NaN included, is
//    an f16 value), two elements per instruction;
//  - f32 -> e4m3 rounds to nearest, ties to even, and saturates to +-448
//    (.satfinite), the stored form of a new latent row;
//  - bf16 -> f16 (through f32) is exact for |x| in [2^-14, 65504] and rounds
//    below; magnitudes above 65504 saturate (the f16 operand form of q).
#pragma once

#include <stdint.h>

namespace mla {

// two E4M3 codes (low byte = first element) -> f16x2 (low half = first)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t d;
  const uint16_t h = (uint16_t)two;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(h));
  return d;
}

// (first, second) f32 -> two E4M3 codes, first in the low byte
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float first, float second) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(second), "f"(first));
  return d;
}

// bf16x2 (low half = first) -> f16x2 (low half = first)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float first = __uint_as_float(w << 16), second = __uint_as_float(w & 0xffff0000u);
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(second), "f"(first));
  return d;
}

// Eight bf16 values (one 16-byte word) -> eight E4M3 codes (8 bytes): each
// x becomes the code nearest to fp32(x) * inv_scale (one fp32 rounding).
__device__ __forceinline__ uint2 quantize_bf16x8(uint4 w, float inv_scale) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t code[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    code[i] = f32x2_to_e4m3x2(__fmul_rn(__uint_as_float(in[i] << 16), inv_scale),
                              __fmul_rn(__uint_as_float(in[i] & 0xffff0000u), inv_scale));
  return make_uint2(code[0] | (code[1] << 16), code[2] | (code[3] << 16));
}

}  // namespace mla
