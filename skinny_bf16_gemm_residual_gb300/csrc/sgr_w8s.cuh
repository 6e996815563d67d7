// sgr_w8s.cuh -- FP8-weight decode kernel on the FP8 tensor-core path
// (tcgen05.mma kind::f8f6f4) for up to 16 tokens.
//
//     Y[m,n] = bf16_rn( scale[n] * sum_k A[m,k] * e4m3(Wq[n,k])  +  R[m,n] )
//
// The low-bit weight direction of the bitsandbytes "QLORA-2" page (quantized
// weights streamed for decode-sized batches, 16-bit activations, the scale
// applied to the dot product; "Three-Kernel Strategy").  The other FP8 kernel
// (sgr_w8.cuh) widens every weight code to BF16 on chip and runs BF16 MMAs;
// here the codes go from TMA straight into the tensor core, and the small
// operand -- the activations -- is brought into E4M3 instead, exactly enough
// for the result:
//
//   per token row m, a power-of-two scale 2^k_m puts max_k |A[m,k]| in
//   [128, 256); each scaled value b = A[m,k] 2^k_m is written as
//       hi = e4m3_rn(b),   lo = e4m3_rn(16 (b - hi)),   b = hi + lo / 16,
//   which is exact for every value within 2^13 of its row's maximum (both
//   parts then keep 4 significant bits inside the E4M3 exponent range; a BF16
//   value has 8), and off by less than 2^-21 max_k |A[m,k]| below that.
//   Products of two E4M3 values are exact, so the tensor core accumulates
//   (in FP32) exactly the products of the definition; the epilogue forms
//   (D_hi + D_lo / 16) 2^-k_m, multiplies by scale[n], adds R and rounds once.
//
// Decomposition as the BF16 row-slab kernel: each CTA owns a slab of RB whole
// W rows; G consecutive 128-code K blocks are packed along the diagonal of one
// M = 128 MMA window (block j+g's W rows in TMEM lanes [g RB, g RB + RB), its
// activations -- NT hi rows then NT lo rows -- in columns [2 NT g, 2 NT (g+1))).
// With K = 32 codes per instruction this is a quarter of the MMAs per weight
// byte of the BF16 kernel.
//
// Roles (352 threads).  Warp 0 lane 0 streams the weight codes with TMA into
// a ring (they do not depend on the preceding kernel, so they stream from the
// CTA's start).  Warps 2-9 zero the operand, wait for the preceding kernel,
// read A once (the threads of a token split its K range), find each token's
// scale, then write the split activation operand into shared memory in K
// order, announcing each stage on its own barrier (with A held in registers:
// stage 0 first, then all others at once).  Warp 1 owns tensor memory; its
// lane 0 issues the MMAs of a stage once its codes have landed and its
// activations are written -- with two issuers, the even windows, while lane
// 0 of warp 10 issues the odd ones into a second accumulator (a small-N MMA
// occupies its issuing thread for ~75 cycles); the epilogue adds the two in
// a fixed order.  Warps 2-5 then run the epilogue.  With A held in
// registers the epilogue runs a warm-up pass over its instructions while the
// MMAs finish (see the epilogue).
//
// The conversion runs on every CTA (each needs all of A), on the conversion
// pipe: per value one packed FP32 -> FP16 conversion share and three packed
// E4M3 conversions (FP16 pairs), with the remainder formed in FP16 (exact).
#pragma once

#include <cstring>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sgr_ptx.cuh"
#include "sgr_epi.cuh"
#include "sgr_tc.cuh"
#include "sgr_w8.cuh"
#include "skinny_gemm_residual.h"

namespace sgr {

constexpr int kW8sThreads = 352;      // warp 0 codes, warps 1 and 10 MMA, warps 2-9 activations (2-5 epilogue)
constexpr int kW8sConvThreads = 256;  // activation converters
constexpr int kW8sKBlock = 128;       // codes per 128-byte swizzled row
constexpr int kW8sMaxStages = 8;
constexpr int kW8sStageVec = 8;       // 16-byte activation vectors per converter thread per stage (at most)
constexpr int kW8sMaxTokens = 16;

struct W8sParams {
  const __nv_bfloat16* A;
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  const float* scale;
  long long lda, ldr, ldy;
  unsigned* err;
  int M, N, K;
  int RB;        // W rows per CTA (multiple of 8)
  int NT;        // token rows per part of the activation operand (8 or 16)
  int kb;        // 128-code K blocks: ceil(K / 128)
  int kbp;       // K blocks in the activation operand: kb rounded up to whole MMA windows
  int kbps;      // K blocks per weight stage (a multiple of groups)
  int k_stages;  // ceil(kb / kbps)
  int stages;    // weight ring depth
  int groups;    // K blocks per MMA window (1, 2 or 4)
  int issuers;   // MMA-issuing threads (1 or 2), each into its own accumulator
  int tmem_cols;
};

__host__ __device__ inline uint32_t w8s_wstage_bytes(int kbps, int rb) { return (uint32_t)kbps * rb * 128u; }
__host__ __device__ inline uint32_t w8s_bblock_bytes(int nt) { return 2u * nt * 128u; }

// Bytes after the weight ring that the kernel's MMAs may read: the
// activation operand, or the last MMA window's over-read past the ring when
// that is longer.
__host__ __device__ inline uint32_t w8s_operand_span(int kbp, int nt, int rb) {
  const uint32_t act = (uint32_t)kbp * w8s_bblock_bytes(nt);
  const uint32_t over = (uint32_t)(kTcTileRows - rb) * 128u;
  return act > over ? act : over;
}

constexpr uint32_t kW8sScratchBytes = 256;  // epilogue warm-up pass, after the operand span

// Whether each converter thread's share of its token row fits the registers
// (kW8sStageVec 16-byte vectors; all 256 threads over the next power of two
// >= M tokens): then A is read once into registers, the conversion ends well
// before the MMAs, and the kernel instance with the epilogue warm-up runs.
__host__ __device__ inline bool w8s_in_regs(int M, int K) {
  const int mp = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : (M <= 8 ? 8 : 16)));
  const int tpt = kW8sConvThreads / mp;
  return (K / 8 + tpt - 1) / tpt <= kW8sStageVec;
}

// Shared memory: alignment slack, barrier region, weight ring, operand span,
// scratch.
__host__ __device__ inline size_t w8s_smem_bytes(int stages, int kbps, int rb, int nt, int kbp) {
  const size_t ring = (size_t)stages * w8s_wstage_bytes(kbps, rb);
  return 1024 + 1024 + ring + w8s_operand_span(kbp, nt, rb) + kW8sScratchBytes;
}

// Four floats -> four E4M3 codes (round to nearest even, saturating), byte i
// = value i.
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float a0, float a1, float a2, float a3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

// Four E4M3 codes (byte i) -> their values (exact, through FP16).
__device__ __forceinline__ void e4m3x4_to_f32x4(uint32_t v, float& a0, float& a1, float& a2, float& a3) {
  asm("{\n\t.reg .b16 lo, hi, x0, x1, x2, x3;\n\t.reg .b32 h01, h23;\n\t"
      "mov.b32 {lo, hi}, %4;\n\t"
      "cvt.rn.f16x2.e4m3x2 h01, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 h23, hi;\n\t"
      "mov.b32 {x0, x1}, h01;\n\t"
      "mov.b32 {x2, x3}, h23;\n\t"
      "cvt.f32.f16 %0, x0;\n\tcvt.f32.f16 %1, x1;\n\tcvt.f32.f16 %2, x2;\n\tcvt.f32.f16 %3, x3;\n\t}"
      : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
      : "r"(v));
}

// Eight scaled activations -> eight hi codes and eight lo codes (b = hi + lo/16).
__device__ __forceinline__ void split8(const float (&b)[8], uint2& hi, uint2& lo) {
  hi.x = f32x4_to_e4m3x4(b[0], b[1], b[2], b[3]);
  hi.y = f32x4_to_e4m3x4(b[4], b[5], b[6], b[7]);
  float h[8];
  e4m3x4_to_f32x4(hi.x, h[0], h[1], h[2], h[3]);
  e4m3x4_to_f32x4(hi.y, h[4], h[5], h[6], h[7]);
  float r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = (b[i] - h[i]) * 16.0f;  // both steps exact
  lo.x = f32x4_to_e4m3x4(r[0], r[1], r[2], r[3]);
  lo.y = f32x4_to_e4m3x4(r[4], r[5], r[6], r[7]);
}

// Two E4M3 codes (a 16-bit pair, the lower in the low byte) -> their values
// as an FP16 pair, exactly: each code's seven magnitude bits eeee.mmm go to
// FP16 bits 13..7 (sign replicated above), which reads as the code's value
// times 2^-8 in FP16 (exponent bias 15 against 7; zero and subnormal codes
// land on FP16 zero and subnormals), and one FP16x2 multiply by 2^8 restores
// it.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t c) {
  uint32_t t;
  asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(t) : "r"((uint32_t)c));
  t = (t << 7) & 0xBF80BF80u;
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(0x5C005C00u));  // 0x5C00 = 256
  return d;
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// D (+)= A[smem] . B[smem]^T with E4M3 A and B, FP32 D, issued by one thread.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format 0), FP32
// D (bits 4-5 = 1), both K-major: N >> 3 at bits 17-22, M >> 4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// kInRegs = w8s_in_regs(M, K): the instance with the register form of the
// converters and the epilogue's warm-up pass; the other instance has the
// per-stage form and no warm-up.  Each carries only its own code (the first
// run of a code path in a CTA is paid in instruction fetches).
template <bool kInRegs>
__global__ void __launch_bounds__(kW8sThreads, 1)
    w8s_kernel(const __grid_constant__ CUtensorMap tmW, const W8sParams p) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  const int S = p.stages;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(sb);  // [S]  codes landed
  uint64_t* wempty = wfull + S;                        // [S]  MMAs done with the slot
  uint64_t* acc_full = wempty + S;                     // [1]
  uint64_t* drain = acc_full + 1;                      // [1]
  uint64_t* bready = drain + 1;                        // [KS] activations of stage s written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bready + p.k_stages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* tok_k = reinterpret_cast<int*>(sb + 896);             // [16] per-token scale exponents
  unsigned* tok_mag = reinterpret_cast<unsigned*>(sb + 960);  // [16] per-token largest |A| (BF16 bits)
  const uint32_t wbox = (uint32_t)p.RB * 128u;
  const uint32_t w_stage = w8s_wstage_bytes(p.kbps, p.RB);
  const uint32_t bblk = w8s_bblock_bytes(p.NT);
  const uint32_t w_ring = base + 1024;
  const uint32_t b_buf = w_ring + (uint32_t)S * w_stage;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KS = p.k_stages;
  const int G = p.groups;
  const int n0 = (int)blockIdx.x * p.RB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&wfull[s]), 1);
      mbar_init(smem_u32(&wempty[s]), (uint32_t)p.issuers);  // one commit per issuer and stage
    }
    for (int k = 0; k < p.k_stages; ++k) mbar_init(smem_u32(&bready[k]), 1);
    mbar_init(smem_u32(acc_full), (uint32_t)p.issuers);
    mbar_init(smem_u32(drain), (uint32_t)p.issuers);
    for (int t = 0; t < kW8sMaxTokens; ++t) tok_mag[t] = 0u;
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) prefetch_tmap(&tmW);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();  // the dependent grid still waits for our completion before reading

  if (warp == 0) {
    // ---------------------------------------------------- weight-code producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      int slot = 0, issued = 0;
      uint32_t par = 0;
      for (int s = 0; s < KS; ++s) {
        if (s >= S && !mbar_wait_or_abort(smem_u32(&wempty[slot]), par ^ 1u, abort_flag)) {
          if (!*abort_flag) report_error(p.err, kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        // Blocks of this stage up to the last MMA window's end: a box past K
        // is filled with zeros by the copy, so that no stale ring byte meets
        // the zero padding of the activation operand.
        const int j0 = s * p.kbps;
        const int nb = p.kbp - j0 < p.kbps ? p.kbp - j0 : p.kbps;
        const uint32_t fb = smem_u32(&wfull[slot]);
        mbar_arrive_expect_tx(fb, (uint32_t)nb * wbox);
        for (int j = 0; j < nb; ++j)
          tma_load_2d(w_ring + (uint32_t)slot * w_stage + (uint32_t)j * wbox, &tmW, (j0 + j) * kW8sKBlock, n0, fb,
                      pol_w);
        issued = s + 1;
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
        }
      }
      bool ok = true;  // every copy this thread issued lands before the CTA may exit
      for (int t = issued > S ? issued - S : 0; t < issued && ok; ++t)
        ok = mbar_wait(smem_u32(&wfull[t % S]), (t / S) & 1);
      if (!ok) report_error(p.err, kErrDrain);
    }
  } else if (warp == 1 || warp == 10) {
    // ----------------------------------------------------------- MMA issuers
    // Issuer i takes MMA windows i, i + issuers, ... of every stage into
    // accumulator i (G * 2 NT columns each).
    const int iss = warp == 10 ? 1 : 0;
    if (lane == 0 && iss < p.issuers) {
      const uint32_t dacc = tmem + (uint32_t)(iss * G * 2 * p.NT);
      const uint32_t idesc = idesc_e4m3_f32(kTcTileRows, G * 2 * p.NT);
      const uint64_t wdesc0 = smem_desc_sw128(w_ring);
      const uint64_t bdesc0 = smem_desc_sw128(b_buf);
      // No index arithmetic per MMA: descriptors advance by fixed steps and
      // the accumulate flag is a register the first MMA clears.
      const int w0 = iss * G, wstep = p.issuers * G;
      const uint64_t w_win = (uint64_t)((uint32_t)wstep * wbox >> 4), b_win = (uint64_t)((uint32_t)wstep * bblk >> 4);
      const uint64_t w_first = (uint64_t)((uint32_t)w0 * wbox >> 4);
      bool ok = true;
      int slot = 0;
      uint32_t par = 0;
      uint32_t accum = 0;
      uint64_t wstage = wdesc0;                                        // this slot's first code box
      uint64_t bstage = bdesc0 + (uint64_t)((uint32_t)w0 * bblk >> 4);  // this issuer's first window in stage s
      const uint64_t b_stage = (uint64_t)((uint32_t)p.kbps * bblk >> 4);
      for (int s = 0; s < KS && ok; ++s) {
        if (!mbar_wait_or_abort(smem_u32(&wfull[slot]), par, abort_flag) ||
            !mbar_wait_or_abort(smem_u32(&bready[s]), 0, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int wend = p.kb - s * p.kbps < p.kbps ? p.kb - s * p.kbps : p.kbps;  // windows starting inside K
        uint64_t wd = wstage + w_first, bd = bstage;
        for (int w = w0; w < wend; w += wstep) {
#pragma unroll
          for (int kk = 0; kk < kW8sKBlock / 32; ++kk) {
            mma_e4m3(dacc, wd + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, accum);  // K step: 32 bytes
            accum = 1u;
          }
          wd += w_win;
          bd += b_win;
        }
        mma_commit(smem_u32(&wempty[slot]));
        bstage += b_stage;
        wstage += w_stage >> 4;
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
          wstage = wdesc0;
        }
      }
      if (ok) {
        mma_commit(smem_u32(acc_full));
      } else {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      mma_commit(smem_u32(drain));
      if (!mbar_wait(smem_u32(drain), 0)) report_error(p.err, kErrDrain);
    }
  } else {
    // ------------------------------------------------ activation converters
    const int ct = threadIdx.x - 64;  // 0 .. 255
    // The operand starts as zeros everywhere (rows of tokens M .. NT-1, the
    // tail of a ragged last block, the padding block of the last MMA
    // window): this CTA's own shared memory, so before the dependency wait.
    {
      const uint32_t z1 = b_buf + (uint32_t)p.kbp * bblk;
      for (uint32_t a = b_buf + (uint32_t)ct * 16u; a < z1; a += (uint32_t)kW8sConvThreads * 16u)
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
    }
    // Threads per token: all 256 over the next power of two >= M tokens.
    const int mp = p.M <= 1 ? 1 : (p.M <= 2 ? 2 : (p.M <= 4 ? 4 : (p.M <= 8 ? 8 : 16)));
    const int tpt = kW8sConvThreads / mp;
    const int t = ct / tpt, part = ct % tpt;
    const int nvec = p.K / 8;  // 16-byte vectors per token row
    const bool row_ok = t < p.M;
    const __nv_bfloat16* arow = p.A + (size_t)(row_ok ? t : 0) * p.lda;
    // When a thread's share of its token row is at most kW8sStageVec vectors
    // (M <= 4 at K = 3584), the max pass keeps them in registers (cur[i] =
    // vector part + i tpt) and converts them from there; otherwise the stage
    // loop reads each stage's vectors again, one stage ahead.  (Reading them
    // again puts one memory round trip per stage on the converters' path,
    // which then paces the MMAs and the weight ring.)
    constexpr bool in_regs = kInRegs;  // the host launched the instance for w8s_in_regs(M, K)
    const int vps = p.kbps * (kW8sKBlock / 8);  // vectors per stage (kbps blocks of 128 codes)
    const int voff = ((part % tpt) + tpt) % tpt;
    uint4 cur[kW8sStageVec], nxt[kW8sStageVec];
    float sc = 1.f;
    // The token's largest |A[t,k]| (a BF16 magnitude pattern, this thread's
    // share in `mag`) over its threads -- a lane group of one warp (tpt <=
    // 32) or whole warps -- and from it the scale exponent: max |b| in
    // [2^7, 2^8) (for a zero or subnormal maximum the largest scale keeps
    // everything representable), published in tok_k for the epilogue.
    auto token_scale = [&](uint32_t mag) {
      for (int o = (tpt < 32 ? tpt : 32) / 2; o > 0; o >>= 1) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, mag, o);
        mag = other > mag ? other : mag;
      }
      if ((lane & ((tpt < 32 ? tpt : 32) - 1)) == 0) atomicMax(&tok_mag[t], mag);
      named_bar_sync(2, kW8sConvThreads);
      mag = tok_mag[t];
      const int ex = (int)(mag >> 7);  // biased exponent of the maximum
      int k = ex == 0 ? 126 : 134 - ex;
      k = k < -120 ? -120 : (k > 126 ? 126 : k);
      if (part == 0) tok_k[t] = k;
      sc = exp2i(k);
    };
    auto max_mag = [](const uint4& a, uint32_t mag) {
      const uint32_t w4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t lo = w4[h] & 0x7FFFu, hi = (w4[h] >> 16) & 0x7FFFu;
        mag = lo > mag ? lo : mag;
        mag = hi > mag ? hi : mag;
      }
      return mag;
    };
    // Split one 16-byte vector (8 activations of token t at K = 8 v) into its
    // hi and lo E4M3 parts and store both into the operand's block.
    auto convert_store = [&](const uint4& a, int v) {
      const uint32_t w4[4] = {a.x, a.y, a.z, a.w};
      uint32_t hiw[2], low[2];
#pragma unroll
      for (int h = 0; h < 4; h += 2) {
        uint32_t b16[2], hi16[2], r16[2];
        uint16_t hi8[2], lo8[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(b16[u]) : "f"(bf16hi(w4[h + u]) * sc), "f"(bf16lo(w4[h + u]) * sc));
          asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(hi8[u]) : "r"(b16[u]));
          hi16[u] = e4m3x2_to_f16x2(hi8[u]);
          asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r16[u]) : "r"(b16[u]), "r"(hi16[u]));      // exact
          asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r16[u]) : "r"(r16[u]), "r"(0x4C004C00u));  // x 16, exact
          asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(lo8[u]) : "r"(r16[u]));
        }
        hiw[h >> 1] = (uint32_t)hi8[0] | ((uint32_t)hi8[1] << 16);
        low[h >> 1] = (uint32_t)lo8[0] | ((uint32_t)lo8[1] << 16);
      }
      const int j = v >> 4;               // K block
      const int cc = (v & 15) >> 1;       // 16-byte chunk of the 128-byte row
      const uint32_t half = (uint32_t)(v & 1) * 8u;
      const int rh = t, rl = p.NT + t;    // hi row, lo row of the block
      const uint32_t blk = b_buf + (uint32_t)j * bblk;
      const uint32_t ah = blk + (uint32_t)rh * 128u + (uint32_t)((cc ^ (rh & 7)) * 16) + half;
      const uint32_t al = blk + (uint32_t)rl * 128u + (uint32_t)((cc ^ (rl & 7)) * 16) + half;
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(ah), "r"(hiw[0]), "r"(hiw[1]) : "memory");
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(al), "r"(low[0]), "r"(low[1]) : "memory");
    };
    auto load_stage = [&](int st, uint4 (&buf)[kW8sStageVec]) {
      const int v0 = st * vps;
      const int v1 = v0 + vps < nvec ? v0 + vps : nvec;
      const int vfirst = v0 + ((voff - v0) % tpt + tpt) % tpt;
#pragma unroll
      for (int i = 0; i < kW8sStageVec; ++i) {
        const int v = vfirst + i * tpt;
        buf[i] = (row_ok && st < KS && v < v1) ? *reinterpret_cast<const uint4*>(arow + (size_t)v * 8)
                                              : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    if constexpr (in_regs) {
      pdl_wait();  // A and R may come from the preceding kernel; Y may be read by it
      uint32_t mag = 0;
#pragma unroll
      for (int i = 0; i < kW8sStageVec; ++i) {
        const int v = part + i * tpt;
        cur[i] = (row_ok && v < nvec) ? *reinterpret_cast<const uint4*>(arow + (size_t)v * 8)
                                      : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kW8sStageVec; ++i) mag = max_mag(cur[i], mag);
      token_scale(mag);
      // Stage 0 first (the first MMAs wait for it), then all the others
      // (one barrier each: the conversion of a whole stage is short here).
      for (int ph = 0; ph < 2; ++ph) {
        const int v0 = ph == 0 ? 0 : vps;
        const int v1 = ph == 0 ? (vps < nvec ? vps : nvec) : nvec;
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < kW8sStageVec; ++i) {
            const int v = part + i * tpt;
            if (v >= v0 && v < v1) convert_store(cur[i], v);
          }
        }
        fence_proxy_async_smem();  // the generic-proxy writes become visible to the tensor core
        named_bar_sync(2, kW8sConvThreads);
        if (ct == 0) {
          if (ph == 0) {
            mbar_arrive(smem_u32(&bready[0]));
          } else {
            for (int st = 1; st < KS; ++st) mbar_arrive(smem_u32(&bready[st]));
          }
        }
      }
    } else {
      pdl_wait();  // A and R may come from the preceding kernel; Y may be read by it
      uint32_t mag = 0;
      if (row_ok) {
#pragma unroll 4
        for (int v = part; v < nvec; v += tpt) mag = max_mag(*reinterpret_cast<const uint4*>(arow + (size_t)v * 8), mag);
      }
      token_scale(mag);
      // Stage by stage in K order, each stage's vectors read again (from L2)
      // with the next stage's requested while this one is converted.
      load_stage(0, cur);
      for (int st = 0; st < KS; ++st) {
        load_stage(st + 1, nxt);
        const int v0 = st * vps;
        const int v1 = v0 + vps < nvec ? v0 + vps : nvec;
        const int vfirst = v0 + ((voff - v0) % tpt + tpt) % tpt;
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < kW8sStageVec; ++i) {
            const int v = vfirst + i * tpt;
            if (v >= v1) break;
            convert_store(cur[i], v);
          }
        }
#pragma unroll
        for (int i = 0; i < kW8sStageVec; ++i) cur[i] = nxt[i];
        fence_proxy_async_smem();  // the generic-proxy writes become visible to the tensor core
        named_bar_sync(2, kW8sConvThreads);
        if (ct == 0) mbar_arrive(smem_u32(&bready[st]));
      }
    }

    if (warp < 6) {
      // ---------------------------------------------------------- epilogue
      // Thread on TMEM lane L = g RB + r (g < G) holds window group g's sums
      // for W row n0 + r; groups 1 .. G-1 hand theirs to group 0's thread
      // through the drained weight ring, which adds them in group order.
      // With A held in registers the conversion ends microseconds before the
      // accumulator is ready, and the epilogue first runs a warm-up pass over
      // its own instructions in that time (tensor-memory columns no MMA
      // writes, a scratch area past the operand, stores predicated off): the
      // first run of a code path in a CTA costs ~0.7 us more than the next
      // while the weight stream saturates L2.  Otherwise (the conversion
      // ends close to the MMAs) it runs once.
      const int q = warp & 3;
      const int L = q * 32 + lane;
      const int g = L / p.RB;
      const int r = L - g * p.RB;
      const bool owner = g == 0 && n0 + r < p.N;
      const bool helper = g >= 1 && g < G;
      const int NT = p.NT;
      float res[kW8sMaxTokens];
#pragma unroll
      for (int m = 0; m < kW8sMaxTokens; ++m)
        res[m] = (owner && m < p.M) ? __bfloat162float(p.R[(size_t)m * p.ldr + n0 + r]) : 0.f;
      const float wscale = owner ? p.scale[n0 + r] : 0.f;
      const uint32_t xch0 = w_ring + (uint32_t)(helper || owner ? r : 0) * 80u;  // 16 floats + pad per row
      const uint32_t xstep = (uint32_t)p.RB * 80u;
      const uint32_t scratch = b_buf + (uint32_t)w8s_operand_span(p.kbp, p.NT, p.RB);
#pragma unroll 1
      for (int pass = kInRegs ? 0 : 1; pass < 2; ++pass) {
        int passv;  // opaque to the compiler: one copy of the loop body serves both passes
        asm volatile("mov.b32 %0, %1;" : "=r"(passv) : "r"(pass));
        const bool real = passv != 0;
        bool ok = true;
        if (real) {
          ok = mbar_wait_sleepy_or_abort(smem_u32(acc_full), 0, abort_flag);
          if (!ok) {
            if (!*abort_flag) report_error(p.err, kErrWaitMma);
            *abort_flag = 1;
          }
          ok = __all_sync(0xffffffffu, ok);
        }
        tc_fence_after();
        float v[kW8sMaxTokens];
#pragma unroll
        for (int m = 0; m < kW8sMaxTokens; ++m) v[m] = 0.f;
        if (ok && q * 32 < G * p.RB) {  // warp-uniform: this warp holds rows of the MMA window in use
          // Accumulator i (one per MMA issuer) at columns [i C, (i + 1) C).
          const uint32_t C = (uint32_t)(G * 2 * NT);
          const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (real ? 0u : (uint32_t)p.issuers * C);
          const bool two = p.issuers == 2;
          const int glo = (q * 32) / p.RB;
          const int ghi = min(G - 1, (q * 32 + 31) / p.RB);
          for (int gg = glo; gg <= ghi; ++gg) {
            // columns [2 NT gg, 2 NT gg + NT): hi part, then NT columns of the lo part
            float hi16[16], lo16[16];
            if (NT == 16) {
              tmem_ld16_sum(taddr + (uint32_t)(gg * 32), C, two, hi16);  // warp-collective
              tmem_ld16_sum(taddr + (uint32_t)(gg * 32 + 16), C, two, lo16);
            } else {
              tmem_ld16_sum(taddr + (uint32_t)(gg * 16), C, two, hi16);  // 8 hi then 8 lo columns
#pragma unroll
              for (int m = 0; m < 8; ++m) lo16[m] = hi16[8 + m];
            }
            if (gg == g) {
#pragma unroll
              for (int m = 0; m < kW8sMaxTokens; ++m)
                if (m < NT) v[m] = hi16[m] + lo16[m] * 0.0625f;
            }
          }
        }
        const uint32_t x0 = real ? xch0 : scratch;
        const uint32_t xs = real ? xstep : 0u;
        if (ok && helper) {
          const uint32_t dst = x0 + (uint32_t)(g - 1) * xs;
#pragma unroll
          for (int m = 0; m < kW8sMaxTokens; m += 4)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + (uint32_t)m * 4u), "f"(v[m]),
                         "f"(v[m + 1]), "f"(v[m + 2]), "f"(v[m + 3])
                         : "memory");
        }
        named_bar_sync(1, 128);
        if (ok && owner) {
          for (int gg = 1; gg < G; ++gg) {
            const uint32_t src = x0 + (uint32_t)(gg - 1) * xs;
#pragma unroll
            for (int m = 0; m < kW8sMaxTokens; m += 4) {
              float a0, a1, a2, a3;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                           : "r"(src + (uint32_t)m * 4u)
                           : "memory");
              v[m] += a0;
              v[m + 1] += a1;
              v[m + 2] += a2;
              v[m + 3] += a3;
            }
          }
          __nv_bfloat16* yp = p.Y + n0 + r;
#pragma unroll
          for (int m = 0; m < kW8sMaxTokens; ++m)
            st_global_bf16_if(yp + (size_t)m * p.ldy,
                              __float2bfloat16_rn(fmaf(v[m] * exp2i(-tok_k[m]), wscale, res[m])), real && m < p.M);
        }
      }
    }
  }

  __syncwarp();  // lane-0 roles rejoin their warp before the CTA-wide barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

// ------------------------------------------------------------------ host side
// Up to 16 tokens; the split operand of all of K in shared memory next to a
// weight ring of at least two stages.
inline bool w8s_supported(int sms, int M, int N, int K, long long ldw) {
  if (M < 1 || M > kW8sMaxTokens || N < 8 || K < 8 || N % 8 || K % 8) return false;
  (void)ldw;
  const int nt = M <= 8 ? 8 : 16;
  const int rb = w8_rows_per_cta(sms, N);
  if (rb > kTcTileRows) return false;
  const int kb = (K + kW8sKBlock - 1) / kW8sKBlock;
  return w8s_smem_bytes(2, 2, rb, nt, kb + 1) <= 232448;
}

inline void w8s_default_config(int sms, int M, int N, int K, sgr_config* c) {
  std::memset(c, 0, sizeof *c);
  c->path = SGR_PATH_W8S;
  c->ctas_per_sm = 1;
  c->token_tile = M <= 8 ? 8 : 16;
  const int rb = w8_rows_per_cta(sms, N);
  const int kb = (K + kW8sKBlock - 1) / kW8sKBlock;
  // Measured at N = 7168, K = 3584 (graph of calls over distinct code
  // copies): with A in registers (up to 4 tokens) four stages of four
  // 128-code blocks (8.2-8.7 us, ahead of 3 or 5-7 stages and of 2 x 8);
  // above, where each stage's activations are read again, two stages of
  // eight (9.8-10.0 us at 5-8 tokens, ahead of 3-4 x 4).  Shallower rings
  // where shared memory is short.
  const bool regs = w8s_in_regs(M, K);
  const int want_kbps = regs ? 4 : 8, want_stages = regs ? 4 : 2;
  c->k_blocks_per_stage = 2;
  c->stages = 2;
  for (int kbps = want_kbps; kbps >= 2; kbps /= 2)
    for (int st = want_stages; st >= 2; --st)
      if (w8s_smem_bytes(st, kbps, rb, c->token_tile, kb + 4) <= 232448) {
        c->k_blocks_per_stage = kbps;
        c->stages = st;
        return;
      }
}

inline int w8s_plan(const sgr_config& c, int sms, int M, int N, int K, long long ldw, W8sParams* p, int* grid,
                    size_t* smem) {
  if (!w8s_supported(sms, M, N, K, ldw)) return SGR_ERR_UNSUPPORTED;
  const int nt = c.token_tile;
  if ((nt != 8 && nt != 16) || nt < M) return SGR_ERR_UNSUPPORTED;
  if (c.ctas_per_sm != 1) return SGR_ERR_UNSUPPORTED;
  if (c.stages < 2 || c.stages > kW8sMaxStages) return SGR_ERR_UNSUPPORTED;
  const int kbps = c.k_blocks_per_stage;
  if (kbps < 1 || kbps > 8) return SGR_ERR_UNSUPPORTED;
  const int rb = c.rows_per_stage > 0 ? c.rows_per_stage : w8_rows_per_cta(sms, N);
  if (rb % 8 != 0 || rb > kTcTileRows) return SGR_ERR_UNSUPPORTED;
  int groups = 1;
  for (int gcount = 4; gcount >= 2; gcount /= 2)
    if (gcount * rb <= kTcTileRows && gcount * 2 * nt <= 256 && kbps % gcount == 0) {
      groups = gcount;
      break;
    }
  const int kb = (K + kW8sKBlock - 1) / kW8sKBlock;
  const int kbp = (kb + groups - 1) / groups * groups;
  // Each converter thread holds one stage's share of activation vectors: at
  // least 16 threads per token, kbps x 16 vectors per stage.
  if (kbps * (kW8sKBlock / 8) / (kW8sConvThreads / 16) > kW8sStageVec) return SGR_ERR_UNSUPPORTED;
  // Barrier region: 2 x stages + k_stages + 2 barriers, TMEM address and abort
  // flag below the per-token words at byte 896.
  if ((2 * c.stages + (kb + kbps - 1) / kbps + 2) * 8 + 8 > 896) return SGR_ERR_UNSUPPORTED;
  // The epilogue hands over [groups - 1][RB] rows of 80 bytes in the drained ring.
  if ((size_t)(groups - 1) * rb * 80 > (size_t)c.stages * w8s_wstage_bytes(kbps, rb)) return SGR_ERR_UNSUPPORTED;
  const size_t sm = w8s_smem_bytes(c.stages, kbps, rb, nt, kbp);
  if (sm > 232448) return SGR_ERR_UNSUPPORTED;
  p->M = M;
  p->N = N;
  p->K = K;
  p->RB = rb;
  p->NT = nt;
  p->kb = kb;
  p->kbp = kbp;
  p->kbps = kbps;
  p->k_stages = (kb + kbps - 1) / kbps;
  p->stages = c.stages;
  p->groups = groups;
  // Two MMA issuers when every stage has two or more windows and the second
  // issuer has one in the first stage (otherwise its accumulator would stay
  // unwritten); the epilogue's warm-up pass reads as many columns again.
  p->issuers = kbps >= 2 * groups && kb > groups ? 2 : 1;
  p->tmem_cols = detail::pow2_at_least(2 * p->issuers * groups * 2 * nt);
  *grid = (N + rb - 1) / rb;
  *smem = sm;
  return SGR_OK;
}

inline cudaError_t w8s_init_device() {
  cudaError_t e = set_kernel_smem_attrs(reinterpret_cast<const void*>(w8s_kernel<true>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(w8s_kernel<false>));
  return e;
}

inline int w8s_launch(const sgr_config& c, int sms, unsigned* err, const void* A, long long lda, const void* Wq,
                      long long ldw, const float* scale, const void* R, long long ldr, void* Y, long long ldy, int M,
                      int N, int K, bool pdl, cudaStream_t stream) {
  W8sParams p;
  int grid = 0;
  size_t smem = 0;
  int rc = w8s_plan(c, sms, M, N, K, ldw, &p, &grid, &smem);
  if (rc != SGR_OK) return rc;
  CUtensorMap tmW;
  if (!detail::make_tmap_u8(&tmW, Wq, N, K, ldw, p.RB, kW8sKBlock)) return SGR_ERR_LAUNCH;
  p.A = static_cast<const __nv_bfloat16*>(A);
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.scale = scale;
  p.lda = lda;
  p.ldr = ldr;
  p.ldy = ldy;
  p.err = err;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kW8sThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&lc, w8s_in_regs(M, K) ? w8s_kernel<true> : w8s_kernel<false>, tmW, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

}  // namespace sgr
