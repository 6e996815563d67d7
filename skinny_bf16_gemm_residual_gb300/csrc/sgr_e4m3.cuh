// sgr_e4m3.cuh -- exact widening of FP8 E4M3 weight codes to BF16, shared by
// the tensor-core and CUDA-core low-bit kernels.
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

}  // namespace sgr
