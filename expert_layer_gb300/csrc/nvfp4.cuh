// NVFP4 element and scale decoding for the weight-streaming kernel: the
// hardware conversions of PTX (cvt.rn.f16x2.e2m1x2, cvt.rn.f16x2.e4m3x2),
// which are exact -- every e2m1 and every finite e4m3 value is an f16 value
// -- and the f16 product of code and scale, also exact (at most 6
// significant bits, magnitudes 2^-10 .. 2688).  Byte order as the formats
// are packed here: the low nibble (even k) and the low byte map to the low
// f16 half.
#pragma once

#include "common.cuh"

namespace moe {
namespace nvfp4 {
namespace {  // internal linkage: each translation unit gets its own copy

// Two e4m3 bytes (low byte -> low half) to f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t v) {
  uint32_t d;
  asm("{\n .reg .b16 h;\n mov.b32 {h, _}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}" : "=r"(d) : "r"(v));
  return d;
}
// The four e2m1 codes in the low 16 bits of v (byte 0 -> d0, byte 1 -> d1;
// low nibble -> low half) to f16x2, exact.
__device__ __forceinline__ void e2m1x4_f16x2(uint32_t v, uint32_t& d0, uint32_t& d1) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %2;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n}"
      : "=r"(d0), "=r"(d1)
      : "r"(v));
}
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

}  // namespace
}  // namespace nvfp4
}  // namespace moe
