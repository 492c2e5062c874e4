// NVFP4 element and scale formats, decoded from their definitions (shared
// by the weight-streaming and tensor-core NVFP4 kernels).
#pragma once

#include "common.cuh"

namespace moe {
namespace nvfp4 {
namespace {  // internal linkage: each translation unit gets its own copy

// e2m1 code -> value, from the format: sign, 2-bit exponent (bias 1), 1-bit
// mantissa; exponent 0 is subnormal (m * 0.5).
__device__ float e2m1_value(int code) {
  const int e = (code >> 1) & 3, m = code & 1;
  const float mag = e == 0 ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
  return (code & 8) ? -mag : mag;
}

// e4m3 byte -> value: sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0
// is subnormal (m/8 * 2^-6); S.1111.111 is NaN.
__device__ float e4m3_value(int b) {
  const int e = (b >> 3) & 15, m = b & 7;
  float mag;
  if (e == 15 && m == 7) mag = __int_as_float(0x7fc00000);
  else if (e == 0) mag = ldexpf((float)m / 8.0f, -6);
  else mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return (b & 0x80) ? -mag : mag;
}

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

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Fill the decode tables: lut2[b*32 + lane] = the two bf16 values of code
// byte b (low nibble = even element in the low half), one copy per lane so
// that 32 lanes looking up different bytes hit 32 different banks; lut8[b] =
// bf16 of the e4m3 scale byte b.  Called by all `nthreads` threads of a block.
__device__ void fill_tables(uint32_t* lut2, uint16_t* lut8, int tid, int nthreads) {
  for (int i = tid; i < 256 * 32; i += nthreads) {
    const int b = i >> 5;
    lut2[i] = pack_bf16x2(e2m1_value(b & 15), e2m1_value(b >> 4));
    if ((i & 31) == 0) lut8[b] = f2bf(e4m3_value(b));
  }
}

}  // namespace
}  // namespace nvfp4
}  // namespace moe
