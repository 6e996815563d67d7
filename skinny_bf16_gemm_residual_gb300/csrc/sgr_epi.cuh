// sgr_epi.cuh -- small pieces shared by the decode epilogues of the row-slab
// (sgr_rows.cuh) and FP8 split-activation (sgr_w8s.cuh) kernels: the sum of
// two MMA issuers' accumulators and a store that a warm-up pass can run with
// no effect.
#pragma once

#include <cuda_bf16.h>

#include "sgr_tc.cuh"

namespace sgr {

// 16 accumulator columns at taddr, plus the same columns of the second
// accumulator (C columns further) when there are two issuers, added in that
// order.  Warp-collective.
__device__ __forceinline__ void tmem_ld16_sum(uint32_t taddr, uint32_t C, bool two, float (&v)[16]) {
  tmem_ld16(taddr, v);
  if (two) {
    float w[16];
    tmem_ld16(taddr + C, w);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += w[i];
  }
}

// Store one BF16 value if `pred`; the store instruction is executed either
// way (predicated off, it touches no memory), so a warm-up pass fetches it.
__device__ __forceinline__ void st_global_bf16_if(__nv_bfloat16* ptr, __nv_bfloat16 x, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.global.b16 [%0], %1;\n\t}" ::"l"(ptr),
      "h"(__bfloat16_as_ushort(x)), "r"((int)pred)
      : "memory");
}

}  // namespace sgr
