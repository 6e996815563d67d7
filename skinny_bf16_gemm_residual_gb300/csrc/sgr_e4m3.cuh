// sgr_e4m3.cuh -- exact widening of low-bit weight codes (FP8 E4M3, and
// NVFP4: FP4 E2M1 with E4M3 block scales) for the tensor-core and CUDA-core
// low-bit kernels.
//
// E4M3 (OCP 8-bit floating point): sign, exponent e (4 bits, bias 7),
// fraction f (3 bits); e > 0: (1 + f/8) 2^(e-7), e = 0: f 2^-9; S.1111.111
// is NaN (outside the kernels' domain).  Placing the seven magnitude bits
// eeee.fff at bits 10-4 of a BF16 pattern (sign at bit 15) gives a BF16 whose
// exponent field is the code's unbiased one, the code's value times 2^-120
// (zero and subnormal codes land on BF16 zero and subnormals); one BF16x2
// multiply by 2^112 then gives the code's value times 2^-8 exactly (a
// power-of-two product whose result is normal or zero; BF16 arithmetic keeps
// subnormal inputs).  The kernels multiply their FP32 sums by scale * 2^8.
#pragma once

#include <cstdint>

namespace sgr {

constexpr float kE4m3Unscale = 256.0f;  // 2^8: undoes the widening's 2^-8

// Two E4M3 codes (bytes SEL of x) -> two BF16 values code * 2^-8.  SEL =
// 0x9180: bytes 0, 1 (low, high half); 0xB3A2: bytes 2, 3.  The permute puts
// each code in the low byte of its 16-bit half with its sign replicated in
// the high byte; shift and mask leave s | eeee.fff << 4.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_scaled(uint32_t x) {
  uint32_t t, d;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(x), "n"(SEL));
  t = (t << 4) & 0x87F087F0u;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(0x77807780u));  // 0x7780 = 2^112
  return d;
}

// Eight E2M1 codes (the nibbles of x, element 0 in the lowest) to four FP16
// pairs, two codes per hardware conversion (the byte's low nibble to the low
// half).  E2M1 (OCP MX FP4): sign, exponent (2 bits, bias 1), one fraction
// bit; every value is an FP16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t x, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b32 {c0, c1, c2, c3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(x));
}

// Two E4M3 block scales (the low byte of sc2 first) as the FP16 pairs
// {scale 0, scale 0} and {scale 1, scale 1} (every E4M3 value is an FP16 value).
__device__ __forceinline__ void e4m3x2_block_scales_f16(uint16_t sc2, uint32_t& s0, uint32_t& s1) {
  uint32_t s16;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(sc2));
  asm("prmt.b32 %0, %1, %1, 0x1010;" : "=r"(s0) : "r"(s16));
  asm("prmt.b32 %0, %1, %1, 0x3232;" : "=r"(s1) : "r"(s16));
}

// 32 NVFP4 codes (16 bytes, element 0 in the lowest nibble) times their two
// block scales (codes 0-15: s0, 16-31: s1, as FP16 pairs) -> 16 words of BF16
// pairs (word c holds codes 2c, 2c+1, the lower in the low half).  Exact: a
// code (2 significant bits) times a scale (4) has at most 6 significant bits
// and lies in [2^-10, 2688], so the FP16 product, its FP32 widening and the
// BF16 rounding are all exact.
__device__ __forceinline__ void w4_widen32(const uint4& v, uint32_t s0, uint32_t s1, uint32_t (&o)[16]) {
  const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t hx[4];
    e2m1x8_to_f16x2(x[i], hx);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t h = hx[b];
      asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h) : "r"(i < 2 ? s0 : s1));
      asm("{\n\t.reg .b16 l, u;\n\t.reg .f32 fl, fu;\n\tmov.b32 {l, u}, %1;\n\t"
          "cvt.f32.f16 fl, l;\n\tcvt.f32.f16 fu, u;\n\t"
          "cvt.rn.bf16x2.f32 %0, fu, fl;\n\t}"
          : "=r"(o[4 * i + b]) : "r"(h));
    }
  }
}

}  // namespace sgr
