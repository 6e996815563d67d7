// sgr_w8.cuh -- low-bit weight variant of the row-slab tensor-core kernel:
// FP8 E4M3 weights with one FP32 scale per output column, BF16 activations,
//
//     Y[m,n] = bf16_rn( scale[n] * sum_k A[m,k] * e4m3(Wq[n,k])  +  R[m,n] )
//
// with FP32 accumulation and one rounding.  The direction is the one of the
// bitsandbytes "QLORA-2" page (quantized weights streamed for decode-sized
// batches with 16-bit activations, the scale applied to the dot product,
// "Three-Kernel Strategy"); the FP8 encoding is OCP E4M3 (bias 7, subnormals,
// no infinities).  Weight bytes per call halve against the BF16 kernel.
//
// Decomposition as in the BF16 row-slab kernel: each CTA owns a slab of RB
// whole W rows (no output element is split across CTAs) and packs G
// consecutive 64-wide K blocks along the diagonal of one M = 128 MMA window.
//
// The tensor core has no FP8 x BF16 form (kind::f16 wants two 16-bit
// operands, kind::f8f6f4 two narrow ones), so the codes are widened on chip:
// TMA brings boxes of RB rows x 128 codes into a shared-memory ring; the
// converter warps read each W row's codes, widen them in registers and write
// them into tensor memory (tcgen05.st); the MMA takes its weight operand
// straight from tensor memory and the activations from shared memory.  The
// widened weights never go back through shared memory: per weight byte there
// is one TMA write and one shared-memory read.
//
// Widening (sgr_e4m3.cuh): exact for every code, one byte permute, a shift,
// a mask and a BF16x2 multiply per two codes, giving code * 2^-8; the
// epilogue multiplies the FP32 sum by scale * 2^8 (exact).  The NaN codes
// (0x7F, 0xFF) are outside the supported domain: a saturating quantiser never
// writes them, and the kernel reads them as +-480.
//
// The NVFP4 instantiation (FP4 = true) runs the same pipeline on 4-bit E2M1
// codes (two per byte, element 2i in the low nibble) with one E4M3 scale per
// 16 elements and one FP32 tensor scale: a 128-byte box row holds 256 codes
// (four 64-wide K blocks); each stage also brings the RB rows' block scales of
// its K range (a small unswizzled box, counted on the same barrier); a
// converter lane widens its 32 codes with the hardware E2M1 -> FP16
// conversion, multiplies each pair by its block scale in FP16 and rounds to
// BF16, all exact (sgr_e4m3.cuh); the epilogue multiplies by the tensor scale.
//
// Warp roles (352 threads): warp 0 lane 0 streams the weight codes with TMA
// into their own ring, released by the converters (the codes do not depend on
// the preceding kernel, so they stream from the start); warp 10 lane 0 loads
// the activations (a ring released by the MMAs) and the residual tile after
// griddepcontrol.wait; warp 1 owns tensor memory and lane 0 issues the MMAs;
// warps 2-9 convert (two warps per tensor-memory lane quarter, one per half
// of a 64-code block); warps 2-5 then run the epilogue.
#pragma once

#include <cstring>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sgr_e4m3.cuh"
#include "sgr_ptx.cuh"
#include "sgr_tc.cuh"
#include "skinny_gemm_residual.h"

namespace sgr {

constexpr int kW8ConvWarps = 8;
constexpr int kW8Threads = 64 + 32 * kW8ConvWarps + 32;  // + one activation-producer warp
constexpr int kW8AWarp = 2 + kW8ConvWarps;               // warp index of the activation producer
constexpr int kW8MaxTokens = 256;
constexpr int kW8SlotCols = 32;   // TMEM columns of one widened 64-code block row (64 BF16)
constexpr int kW8MaxStages = 16;
constexpr int kW8MaxAStages = 8;
constexpr int kW8MaxSlots = 8;
constexpr int kW8MaxWins = 8;     // MMA windows per stage (kbps / groups)

struct W8Params {
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  const float* scale;  // E4M3: per-column scales (NVFP4: unused)
  float gs;            // NVFP4: tensor scale
  long long ldr, ldy;
  unsigned* err;
  int M, N, K;
  int RB;          // W rows per CTA (multiple of 8, <= 128)
  int NT;          // token tile = MMA N per group (multiple of 16, >= M)
  int k_stages;    // ceil(K / (64 * kbps))
  int kbps;        // 64-wide K blocks per stage (even; NVFP4: 4 or 8)
  int stages;      // depth of the weight-code ring
  int a_stages;    // depth of the activation ring
  int groups;      // K blocks packed into one MMA window (1, 2 or 4)
  int slots;       // stages of widened weights held in tensor memory
  int acc_cols;    // accumulator columns; the weight slots follow
  int tmem_cols;
  int conv_warps;  // converter warps whose lane quarter holds rows of the window
};

__host__ __device__ inline uint32_t w8_wstage_bytes(int kbps, int rb) { return (uint32_t)(kbps / 2) * rb * 128u; }
// NVFP4 stage: kbps/4 code boxes (RB rows x 256 codes), then the RB rows'
// block scales (kbps * 4 bytes each), rounded up to keep the next stage's
// swizzled boxes 1024-byte aligned.
__host__ __device__ inline uint32_t w4_scale_off(int kbps, int rb) { return (uint32_t)(kbps / 4) * rb * 128u; }
__host__ __device__ inline uint32_t w4_wstage_bytes(int kbps, int rb) {
  return (w4_scale_off(kbps, rb) + (uint32_t)rb * kbps * 4u + 1023u) & ~1023u;
}
__host__ __device__ inline uint32_t wring_stage_bytes(bool fp4, int kbps, int rb) {
  return fp4 ? w4_wstage_bytes(kbps, rb) : w8_wstage_bytes(kbps, rb);
}
__host__ __device__ inline uint32_t w8_astage_bytes(int kbps, int nt) { return (uint32_t)kbps * nt * 128u; }
__host__ __device__ inline uint32_t w8_rtile_bytes(int rb, int nt) { return ((uint32_t)rb * nt * 2u + 1023u) & ~1023u; }

__host__ __device__ inline size_t w8_smem_bytes(int stages, int a_stages, int kbps, int rb, int nt, bool fp4 = false) {
  return 1024 /* alignment slack */ + 1024 /* barriers */ + (size_t)stages * wring_stage_bytes(fp4, kbps, rb) +
         (size_t)a_stages * w8_astage_bytes(kbps, nt) + w8_rtile_bytes(rb, nt);
}

// 32 codes (8 words, code i in byte i%4 of word i/4) -> 16 words of BF16
// pairs (column c holds codes 2c, 2c+1, the lower in the low half).
__device__ __forceinline__ void w8_widen32(const uint32_t (&x)[8], uint32_t (&o)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    o[2 * i] = e4m3x2_to_bf16x2_scaled<0x9180u>(x[i]);
    o[2 * i + 1] = e4m3x2_to_bf16x2_scaled<0xB3A2u>(x[i]);
  }
}

// The 16-token epilogue form serves the plan.
__host__ __device__ inline bool w8_decode_epi(const W8Params& p) { return p.NT == 16 && p.groups <= 2; }

// tmS: the NVFP4 block scales (unused, any map, for E4M3).  kDecode: the
// 16-token epilogue with at most two packed groups (w8_decode_epi), else the
// general one; each instance carries only its own epilogue code (the first
// run of a code path in a CTA is paid in instruction fetches).
template <bool FP4, bool kDecode>
__global__ void __launch_bounds__(kW8Threads, 2)
    w8_rows_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmS,
                   const W8Params p) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  const int S = p.stages, SA = p.a_stages, TS = p.slots;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(sb);  // [S]  weight codes landed
  uint64_t* wempty = wfull + S;                        // [S]  codes read by the converters
  uint64_t* afull = wempty + S;                        // [SA] activations landed
  uint64_t* aempty = afull + SA;                       // [SA] activations read by the MMAs
  uint64_t* tfull = aempty + SA;                       // [TS] a stage of widened weights in tensor memory
  uint64_t* tfree = tfull + TS;                        // [TS] MMAs done with a tensor-memory stage
  uint64_t* acc_full = tfree + TS;
  uint64_t* drain = acc_full + 1;
  uint64_t* rfull = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t wbox = (uint32_t)p.RB * 128u;  // one weight box: RB rows x 128 bytes (128 or 256 codes)
  const uint32_t ablk = (uint32_t)p.NT * 128u;  // one activation box: NT rows x 64 BF16
  const uint32_t w_stage = wring_stage_bytes(FP4, p.kbps, p.RB);
  const uint32_t sc_off = w4_scale_off(p.kbps, p.RB);           // NVFP4: block scales within a stage
  const uint32_t sc_row = (uint32_t)p.kbps * 4u;                 // NVFP4: block-scale bytes per row and stage
  const uint32_t a_stage = w8_astage_bytes(p.kbps, p.NT);
  const uint32_t w_ring = base + 1024;
  const uint32_t a_ring = w_ring + (uint32_t)S * w_stage;
  const uint32_t r_tile = a_ring + (uint32_t)SA * a_stage;  // [NT][RB] BF16 residual tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KS = p.k_stages;
  const int G = p.groups;
  const int wins = p.kbps / G;  // MMA windows per stage
  const int n0 = (int)blockIdx.x * p.RB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&wfull[s]), 1);
      mbar_init(smem_u32(&wempty[s]), p.conv_warps);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(smem_u32(&afull[s]), 1);
      mbar_init(smem_u32(&aempty[s]), 1);
    }
    for (int t = 0; t < TS; ++t) {
      mbar_init(smem_u32(&tfull[t]), p.conv_warps);
      mbar_init(smem_u32(&tfree[t]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(rfull), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  // Tensor memory first: a CTA launched early by programmatic dependent launch
  // waits here (in the allocation) until the previous kernel's CTA on this SM
  // releases its columns.  Letting it stream its first weight stages before
  // the allocation measured slower (15.9 against 10.8 us per call).
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmR);
    if (FP4) prefetch_tmap(&tmS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------- weight-code producer (TMA)
    // The codes do not depend on the preceding kernel (they must not be
    // written by it), so they stream from the start, paced only by the
    // converters releasing ring slots.
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      int slot = 0, issued = 0;
      uint32_t par = 0;
      for (int s = 0; s < KS; ++s) {
        if (s >= S && !mbar_wait_sleepy_or_abort(smem_u32(&wempty[slot]), par ^ 1u, abort_flag)) {
          if (!*abort_flag) report_error(p.err, kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        const uint32_t wb = smem_u32(&wfull[slot]);
        const uint32_t st = w_ring + (uint32_t)slot * w_stage;
        if constexpr (FP4) {
          // kbps/4 boxes of 256 codes (128 bytes) per row, then the block scales.
          mbar_arrive_expect_tx(wb, sc_off + (uint32_t)p.RB * sc_row);
          for (int j = 0; j < p.kbps / 4; ++j)
            tma_load_2d(st + (uint32_t)j * wbox, &tmW, (s * p.kbps + 4 * j) * (kTcKBlock / 2), n0, wb, pol_w);
          tma_load_2d(st + sc_off, &tmS, s * p.kbps * 4, n0, wb, pol_w);
        } else {
          mbar_arrive_expect_tx(wb, w_stage);
          for (int j = 0; j < p.kbps / 2; ++j)
            tma_load_2d(st + (uint32_t)j * wbox, &tmW, (s * p.kbps + 2 * j) * kTcKBlock, n0, wb, pol_w);
        }
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
  } else if (warp == kW8AWarp) {
    // ------------------------------ activation and residual producer (TMA)
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_r = policy_evict_first();
      pdl_wait();  // A and R may come from the preceding kernel
      int slot = 0, issued = 0;
      uint32_t par = 0;
      for (int s = 0; s < KS; ++s) {
        if (s >= SA && !mbar_wait_sleepy_or_abort(smem_u32(&aempty[slot]), par ^ 1u, abort_flag)) {
          if (!*abort_flag) report_error(p.err, kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        const uint32_t ab = smem_u32(&afull[slot]);
        mbar_arrive_expect_tx(ab, a_stage);
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(a_ring + (uint32_t)slot * a_stage + (uint32_t)j * ablk, &tmA, (s * p.kbps + j) * kTcKBlock,
                      0, ab, pol_a);
        if (s == 0) {  // the residual tile, needed only by the epilogue
          const uint32_t rb = smem_u32(rfull);
          mbar_arrive_expect_tx(rb, (uint32_t)p.RB * p.NT * 2u);
          tma_load_2d(r_tile, &tmR, n0, 0, rb, pol_r);
        }
        issued = s + 1;
        if (++slot == SA) {
          slot = 0;
          par ^= 1u;
        }
      }
      bool ok = issued == 0 || mbar_wait(smem_u32(rfull), 0);
      for (int t = issued > SA ? issued - SA : 0; t < issued && ok; ++t)
        ok = mbar_wait(smem_u32(&afull[t % SA]), (t / SA) & 1);
      if (!ok) report_error(p.err, kErrDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTcTileRows, G * p.NT);
      const uint64_t adesc0 = smem_desc_sw128(a_ring);
      const uint32_t wslot0 = tmem + (uint32_t)p.acc_cols;
      bool ok = true;
      int slot = 0, ts = 0;
      uint32_t par = 0, tpar = 0;
      uint64_t ad = adesc0;
      uint32_t accum = 0;
      const uint64_t a_win = (uint64_t)((uint32_t)G * ablk >> 4);  // activations of one MMA window
      const uint32_t tstage = (uint32_t)wins * kW8SlotCols;  // TMEM columns of one widened stage
      for (int s = 0; s < KS; ++s) {
        if (!mbar_wait_or_abort(smem_u32(&afull[slot]), par, abort_flag) ||
            !mbar_wait_or_abort(smem_u32(&tfull[ts]), tpar, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // No index arithmetic per MMA: operand addresses advance by fixed
        // steps and the accumulate flag is a register the first MMA clears.
        uint32_t wa = wslot0 + (uint32_t)ts * tstage;
        uint64_t aw = ad;
        for (int w = 0; w < wins; ++w) {
#pragma unroll
          for (int kk = 0; kk < kTcKBlock / 16; ++kk) {
            // K step: 8 TMEM columns of widened codes, 32 bytes of activations
            mma_bf16_tmem_a(tmem, wa + (uint32_t)(kk * 8), aw + (uint64_t)(kk * 2), idesc, accum);
            accum = 1u;
          }
          wa += (uint32_t)kW8SlotCols;
          aw += a_win;
        }
        mma_commit(smem_u32(&tfree[ts]));
        mma_commit(smem_u32(&aempty[slot]));
        if (++ts == TS) {
          ts = 0;
          tpar ^= 1u;
        }
        ad += a_stage >> 4;
        if (++slot == SA) {
          slot = 0;
          par ^= 1u;
          ad = adesc0;
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
    // ------------------------------------------------------------ converters
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;     // which 32 codes of each 64-code block row
    const int L = q * 32 + lane;          // TMEM lane = row of the MMA window
    const bool epi = half == 0;
    // Scale of the output column this lane may own (a weight: readable before the dependency wait).
    const bool owner = epi && L < p.RB && n0 + L < p.N;
    const float sc = owner ? (FP4 ? p.gs : p.scale[n0 + L] * kE4m3Unscale) : 0.f;
    if (q * 32 < G * p.RB) {  // warp-uniform: the quarter holds rows of the window
      int g = L / p.RB, r = L - g * p.RB;
      if (g >= G) {  // lanes past the window duplicate a real row (their TMEM rows are never read)
        g = 0;
        r = L % p.RB;
      }
      const uint32_t row_off = (uint32_t)r * 128u;
      const uint32_t swz = (uint32_t)(r & 7);
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)p.acc_cols + (uint32_t)half * 16u;
      const uint32_t tstage = (uint32_t)wins * kW8SlotCols;
      bool ok = true;
      int slot = 0, ts = 0;
      uint32_t par = 0, tpar = 0;
      int pend = -1;  // tensor-memory stage whose stores are still in flight
      for (int s = 0; s < KS; ++s) {
        ok = mbar_wait_or_abort(smem_u32(&wfull[slot]), par, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // Windows are read and widened two at a time (independent work for
        // the scheduler to overlap) and stored into this stage's slot.
        const uint32_t wst = w_ring + (uint32_t)slot * w_stage;
        const uint32_t ws = wst + row_off;
        for (int w0 = 0; w0 < wins; w0 += 2) {
          uint32_t o[2][16];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int kb = (w0 + u < wins ? w0 + u : w0) * G + g;  // K block of this lane within the stage
            if constexpr (FP4) {
              // 32 codes = one 16-byte chunk of the 128-byte row of box kb/4,
              // and their two block scales.
              const uint32_t c = (uint32_t)((kb & 3) * 2 + half);
              const uint4 v = lds128(ws + (uint32_t)(kb >> 2) * wbox + ((c ^ swz) << 4));
              uint16_t sc2;
              asm volatile("ld.shared.u16 %0, [%1];"
                           : "=h"(sc2)
                           : "r"(wst + sc_off + (uint32_t)r * sc_row + (uint32_t)kb * 4u + (uint32_t)half * 2u));
              uint32_t s0, s1;
              e4m3x2_block_scales_f16(sc2, s0, s1);
              w4_widen32(v, s0, s1, o[u]);
            } else {
              const uint32_t c0 = (uint32_t)((kb & 1) * 4 + half * 2);  // first 16-byte chunk of the row
              const uint32_t rowp = ws + (uint32_t)(kb >> 1) * wbox;
              const uint4 v0 = lds128(rowp + ((c0 ^ swz) << 4));
              const uint4 v1 = lds128(rowp + (((c0 + 1u) ^ swz) << 4));
              const uint32_t x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
              w8_widen32(x, o[u]);
            }
          }
          if (w0 + 2 >= wins) {  // the stage's codes are all in registers
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&wempty[slot]));
          }
          if (w0 == 0) {
            // The previous stage's stores have had this widening to complete:
            // wait for them and hand that stage to the MMA.
            if (pend >= 0) {
              tmem_wait_st();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&tfull[pend]));
            }
            if (s >= TS) {
              ok = mbar_wait_sleepy_or_abort(smem_u32(&tfree[ts]), tpar ^ 1u, abort_flag);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
            }
            tc_fence_after();
          }
          const uint32_t ta = tl + (uint32_t)ts * tstage + (uint32_t)w0 * kW8SlotCols;
          tmem_st16(ta, o[0]);
          if (w0 + 1 < wins) tmem_st16(ta + kW8SlotCols, o[1]);
        }
        if (!ok) break;
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
        }
        pend = ts;
        if (++ts == TS) {
          ts = 0;
          tpar ^= 1u;
        }
      }
      tmem_wait_st();
      if (ok && pend >= 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tfull[pend]));
      }
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitFull);
        *abort_flag = 1;
      }
    }
    if (epi) {
      // ---------------------------------------------------------- epilogue
      bool ok = mbar_wait_sleepy_or_abort(smem_u32(acc_full), 0, abort_flag) &&
                mbar_wait_sleepy_or_abort(smem_u32(rfull), 0, abort_flag);
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      pdl_wait();  // Y may be read by the preceding kernel (already satisfied: the residual tile came after it)
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
      if constexpr (kDecode) {
        // Decode form: the thread on lane r < RB owns output column n0 + r
        // and holds group 0's sums; the thread on lane RB + r holds group
        // 1's and hands them over through the drained weight ring.
        const bool helper = G == 2 && L >= p.RB && L < 2 * p.RB;
        const int r = owner ? L : L - p.RB;
        const uint32_t xch = w_ring + (uint32_t)(helper || owner ? r : 0) * 80u;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        if (ok && q * 32 < G * p.RB) {
          if (G == 1 || (q + 1) * 32 <= p.RB) {
            tmem_ld16(taddr, v);
          } else if (q * 32 >= p.RB) {
            tmem_ld16(taddr + 16u, v);
          } else {
            float v1[16];
            tmem_ld16(taddr, v);
            tmem_ld16(taddr + 16u, v1);
            if (L >= p.RB) {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = v1[i];
            }
          }
        }
        if (ok && helper) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(xch + (uint32_t)i * 4u), "f"(v[i]),
                         "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                         : "memory");
        }
        named_bar_sync(1, 128);
        if (ok && owner) {
          if (G == 2) {
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              float a0, a1, a2, a3;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                           : "r"(xch + (uint32_t)i * 4u)
                           : "memory");
              v[i] += a0;
              v[i + 1] += a1;
              v[i + 2] += a2;
              v[i + 3] += a3;
            }
          }
          const unsigned short* rt = reinterpret_cast<const unsigned short*>(sb + (r_tile - base)) + L;
          __nv_bfloat16* yp = p.Y + n0 + L;
#pragma unroll
          for (int m = 0; m < 16; ++m)
            if (m < p.M) {
              const float res = __uint_as_float((uint32_t)rt[m * p.RB] << 16);
              yp[(size_t)m * p.ldy] = __float2bfloat16_rn(fmaf(v[m], sc, res));
            }
        }
      } else {
        // General form: every lane stages its diagonal block row (group g,
        // row r) in the drained rings, then each thread sums the groups of
        // one (row, 16-token chunk) in group order and stores.
        const int etid = threadIdx.x - 64;
        const int g = L / p.RB, r = L % p.RB;
        const int chunks = p.NT / 16;
        const int ldp = p.NT + 4;
        float* part = reinterpret_cast<float*>(sb + 1024);
        if (ok) {
          for (int c = 0; c < G * chunks; ++c) {
            float v[16];
            tmem_ld16(taddr + (uint32_t)(c * 16), v);
            if (g < G && c / chunks == g) {
              float* dst = part + ((size_t)g * p.RB + r) * ldp + (c % chunks) * 16;
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
          }
        }
        named_bar_sync(1, 128);
        if (ok) {
          const unsigned short* rt = reinterpret_cast<const unsigned short*>(sb + (r_tile - base));
          for (int item = etid; item < p.RB * chunks; item += 128) {
            const int rr = item % p.RB, c16 = item / p.RB;
            const int n = n0 + rr;
            if (n >= p.N) continue;
            const float scn = FP4 ? p.gs : p.scale[n] * kE4m3Unscale;
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
            for (int gg = 0; gg < G; ++gg) {
              const float* src = part + ((size_t)gg * p.RB + rr) * ldp + c16 * 16;
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 w4 = *reinterpret_cast<const float4*>(src + i);
                acc[i] += w4.x;
                acc[i + 1] += w4.y;
                acc[i + 2] += w4.z;
                acc[i + 3] += w4.w;
              }
            }
            const int m0 = c16 * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (m0 + i < p.M) {
                const float res = __uint_as_float((uint32_t)rt[(m0 + i) * p.RB + rr] << 16);
                p.Y[(size_t)(m0 + i) * p.ldy + n] = __float2bfloat16_rn(fmaf(acc[i], scn, res));
              }
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

// ------------------------------------------------------------------ host side
namespace detail {

// 2-D tensor map over a row-major byte matrix [rows, cols] with row stride ld
// bytes: boxes of box_rows x box_cols bytes, 128-byte swizzle.
inline bool make_tmap_u8(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld,
                         int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A byte matrix [rows, cols] (row stride ld bytes) in boxes of box_rows x
// box_cols bytes without swizzle (the NVFP4 block scales: read per row).
inline bool make_tmap_u8_plain(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld,
                               int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same over BF16 [rows, cols] (row stride ld elements), no swizzle: the
// residual tile is read row by row from shared memory.
inline bool make_tmap_plain_bf16(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld,
                                 int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace detail

inline int w8_rows_per_cta(int sms, int N) {
  const int rb = (N + sms - 1) / sms;
  return (rb + 7) / 8 * 8;
}

inline bool w8_supported(int sms, int M, int N, int K) {
  return M >= 1 && M <= kW8MaxTokens && N >= 8 && K >= 8 && N % 8 == 0 && K % 8 == 0 &&
         w8_rows_per_cta(sms, N) <= kTcTileRows;
}

// Default: two-deep rings of the largest stages (8, else 4, else 2 K blocks)
// that keep the CTA at or under ~110 KB of shared memory, so that the next
// call's CTA is already resident on the SM (waiting in its tensor-memory
// allocation) when this one finishes.  Measured at N = 7168, K = 3584, M = 1-16:
// few large stages beat deep rings of small ones (10.8 us against 13.3 us
// for four K blocks per stage with a six-deep ring): every stage costs a
// hand-off between the converter warps and the MMA thread.
inline void w8_default_config(int sms, int M, int N, int K, sgr_config* c, bool fp4 = false) {
  (void)K;
  std::memset(c, 0, sizeof *c);
  c->path = SGR_PATH_W8;
  c->ctas_per_sm = 1;
  c->token_tile = (M + 15) / 16 * 16;
  c->stages = 2;
  c->prefetch_stages = 2;
  const int rb = w8_rows_per_cta(sms, N);
  // NVFP4 above 8 tokens: 32-row slabs (four packed K blocks fill the 128-row
  // window, every tensor-memory lane quarter converts; measured at N = 7168,
  // K = 3584, M = 16: 11.1 against 11.4 us; slower at M <= 8).
  if (fp4 && M > 8 && (N + 31) / 32 <= 2 * sms) c->rows_per_stage = 32;
  const size_t budget = 110u * 1024u;
  c->k_blocks_per_stage = fp4 ? 4 : 2;
  for (int kb = 8; kb >= (fp4 ? 4 : 2); kb /= 2)
    if (w8_smem_bytes(2, 2, kb, c->rows_per_stage > 0 ? c->rows_per_stage : rb, c->token_tile, fp4) <= budget) {
      c->k_blocks_per_stage = kb;
      return;
    }
}

// stages = depth of the weight-code ring, prefetch_stages = depth of the
// activation ring (0: 2).
inline int w8_plan(const sgr_config& c, int sms, int M, int N, int K, W8Params* p, int* grid, size_t* smem,
                   bool fp4 = false) {
  if (!w8_supported(sms, M, N, K)) return SGR_ERR_UNSUPPORTED;
  if (c.path != SGR_PATH_AUTO && c.path != SGR_PATH_W8) return SGR_ERR_UNSUPPORTED;
  const int nt = c.token_tile;
  if (nt < 16 || nt > kW8MaxTokens || nt % 16 != 0 || nt < M) return SGR_ERR_UNSUPPORTED;
  const int kb = c.k_blocks_per_stage;
  if (kb < 2 || kb > 8 || kb % 2 != 0) return SGR_ERR_UNSUPPORTED;
  if (fp4 && kb % 4 != 0) return SGR_ERR_UNSUPPORTED;  // whole 256-code boxes; 16-byte block-scale boxes
  if (c.ctas_per_sm != 1) return SGR_ERR_UNSUPPORTED;
  if (c.stages < 2 || c.stages > kW8MaxStages) return SGR_ERR_UNSUPPORTED;
  const int sa = c.prefetch_stages > 0 ? c.prefetch_stages : 2;
  if (sa < 2 || sa > kW8MaxAStages) return SGR_ERR_UNSUPPORTED;
  const int rb = c.rows_per_stage > 0 ? c.rows_per_stage : w8_rows_per_cta(sms, N);
  if (rb % 8 != 0 || rb > kTcTileRows) return SGR_ERR_UNSUPPORTED;
  const size_t sm = w8_smem_bytes(c.stages, sa, kb, rb, nt, fp4);
  if (sm > 232448) return SGR_ERR_UNSUPPORTED;
  p->M = M;
  p->N = N;
  p->K = K;
  p->RB = rb;
  p->NT = nt;
  p->kbps = kb;
  p->k_stages = (K + kTcKBlock * kb - 1) / (kTcKBlock * kb);
  p->stages = c.stages;
  p->a_stages = sa;
  p->groups = 1;
  for (int gcount = 4; gcount >= 2; gcount /= 2)
    if (gcount * rb <= kTcTileRows && gcount * nt <= 256 && kb % gcount == 0) {
      p->groups = gcount;
      break;
    }
  // The general epilogue stages [groups][RB][NT+4] floats in the drained rings.
  const size_t rings = (size_t)c.stages * wring_stage_bytes(fp4, kb, rb) + (size_t)sa * w8_astage_bytes(kb, nt);
  while (p->groups > 1 && (size_t)p->groups * rb * (nt + 4) * 4 > rings) p->groups /= 2;
  if ((size_t)p->groups * rb * (nt + 4) * 4 > rings) return SGR_ERR_UNSUPPORTED;
  if (kb / p->groups > kW8MaxWins) return SGR_ERR_UNSUPPORTED;
  // Tensor memory: the accumulator, then as many widened stages as fit in
  // 256 columns (two CTAs per SM), or in 512 if fewer than two fit.
  p->acc_cols = detail::round_up(p->groups * nt, 32);
  const int stage_cols = kb / p->groups * kW8SlotCols;
  p->tmem_cols = 256;
  if ((p->tmem_cols - p->acc_cols) / stage_cols < 2) p->tmem_cols = 512;
  p->slots = (p->tmem_cols - p->acc_cols) / stage_cols;
  if (p->slots > kW8MaxSlots) p->slots = kW8MaxSlots;
  if (p->slots < 2) return SGR_ERR_UNSUPPORTED;
  const int quarters = (p->groups * rb + 31) / 32;
  p->conv_warps = 2 * quarters;
  *grid = (N + rb - 1) / rb;
  *smem = sm;
  return SGR_OK;
}

inline cudaError_t w8_init_device() {
  cudaError_t e = set_kernel_smem_attrs(reinterpret_cast<const void*>(w8_rows_kernel<false, false>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(w8_rows_kernel<false, true>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(w8_rows_kernel<true, false>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(w8_rows_kernel<true, true>));
  return e;
}

inline int w8_launch(const sgr_config& c, int sms, unsigned* err, const void* A, long long lda, const void* Wq,
                     long long ldw, const float* scale, const void* R, long long ldr, void* Y, long long ldy, int M,
                     int N, int K, bool pdl, cudaStream_t stream) {
  W8Params p;
  int grid = 0;
  size_t smem = 0;
  int rc = w8_plan(c, sms, M, N, K, &p, &grid, &smem);
  if (rc != SGR_OK) return rc;
  CUtensorMap tmW, tmA, tmR;
  if (!detail::make_tmap_u8(&tmW, Wq, N, K, ldw, p.RB, 2 * kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap(&tmA, A, M, K, lda, p.NT, kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap_plain_bf16(&tmR, R, M, N, ldr, p.NT, p.RB)) return SGR_ERR_LAUNCH;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.scale = scale;
  p.ldr = ldr;
  p.ldy = ldy;
  p.err = err;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kW8Threads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  auto fn = w8_decode_epi(p) ? w8_rows_kernel<false, true> : w8_rows_kernel<false, false>;
  if (cudaLaunchKernelEx(&lc, fn, tmW, tmA, tmR, tmW, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

// NVFP4 weights on the same kernel: Wq4 [N, K/2] bytes (row stride ldw), bs
// [N, ceil(K/16)] E4M3 block scales (row stride ldbs), tensor scale gs.
inline int w4_launch(const sgr_config& c, int sms, unsigned* err, const void* A, long long lda, const void* Wq4,
                     long long ldw, const void* bs, long long ldbs, float gs, const void* R, long long ldr, void* Y,
                     long long ldy, int M, int N, int K, bool pdl, cudaStream_t stream) {
  W8Params p;
  int grid = 0;
  size_t smem = 0;
  int rc = w8_plan(c, sms, M, N, K, &p, &grid, &smem, true);
  if (rc != SGR_OK) return rc;
  CUtensorMap tmW, tmA, tmR, tmS;
  if (!detail::make_tmap_u8(&tmW, Wq4, N, K / 2, ldw, p.RB, 2 * kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap(&tmA, A, M, K, lda, p.NT, kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap_plain_bf16(&tmR, R, M, N, ldr, p.NT, p.RB)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap_u8_plain(&tmS, bs, N, (K + 15) / 16, ldbs, p.RB, p.kbps * 4)) return SGR_ERR_LAUNCH;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.scale = nullptr;
  p.gs = gs;
  p.ldr = ldr;
  p.ldy = ldy;
  p.err = err;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kW8Threads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  auto fn = w8_decode_epi(p) ? w8_rows_kernel<true, true> : w8_rows_kernel<true, false>;
  if (cudaLaunchKernelEx(&lc, fn, tmW, tmA, tmR, tmS, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

}  // namespace sgr
