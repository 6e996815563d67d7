// sgr_simt.cuh -- bandwidth-bound SIMT path for small M (decode-sized batches).
//
// Computes Y[m,n] = bf16_rn( sum_k A[m,k] * W[n,k] + R[m,n] ) for m < M <= MT,
// accumulating in FP32 and rounding once in the epilogue.  The operation is
// the one benchmarked on the vLLM "benchmark_k3_cutedsl_residual.py" page
// (BF16[M,3584] @ BF16[7168,3584].T + BF16[M,7168], FP32 accumulation, BF16
// out); the SIMT structure follows the main loop of the vLLM
// "fused_add_multicast_skinny_gemm" kernel (vectorised 16-byte W loads,
// FP32 register accumulators, warp-shuffle then shared-memory K reduction,
// residual fused into the epilogue), re-planned for GB300:
//
//  * Persistent grid: CTA c owns the contiguous W rows [N*c/G, N*(c+1)/G),
//    i.e. one contiguous slab of HBM, so the grid is sized to the SM count
//    instead of N/outputs_per_block CTAs.
//  * W is streamed exactly once by one producer thread issuing 1-D bulk
//    copies (cp.async.bulk, L2 evict-first) of `rows_per_stage` whole rows
//    into a `stages`-deep shared-memory ring guarded by mbarriers.  The first
//    stages are requested before griddepcontrol.wait, so with programmatic
//    dependent launch the weight stream overlaps the previous kernel's tail.
//  * 7 consumer warps (224 threads) own a fixed K slice each: thread t owns
//    the 16-byte vectors t, t+224, ... of every row, so its slice of A is
//    loaded once (after griddepcontrol.wait) and stays in registers.
//  * Rows are reduced in batches of 32/MT rows so that each lane holds 32
//    partial sums; one transposing butterfly (31 shuffles) leaves lane l
//    with the warp's total for output l, the 7 warps' totals meet in shared
//    memory, and warp 0 adds R (loaded early, while W streams), rounds once
//    and stores.
//
// The W8 instantiation is the low-bit weight variant (FP8 E4M3 codes Wq with
// one FP32 scale per output column, the quantized-weight decode direction of
// the bitsandbytes "QLORA-2" page): the ring carries rows of K codes (half
// the bytes), each 16-byte vector holds 16 codes, which are widened exactly
// in registers (sgr_e4m3.cuh) before the FP32 FMAs, and the epilogue computes
// fmaf(sum, scale[n] * 2^8, R) with one rounding.
//
// The NVFP4 instantiation streams 4-bit E2M1 codes (two per byte, element 2i
// in the low nibble) with one E4M3 scale per 16 elements of a row and one
// FP32 scale for the tensor.  Each ring record is a row's K/2 code bytes
// followed by its block scales (padded to 16 bytes); each 16-byte vector
// holds 32 codes, converted two at a time to FP16 by the hardware conversion
// and multiplied by their block scale in FP16 (exact: 2 x 4 significant bits,
// magnitudes 2^-10 .. 2688), then widened to FP32 for the FMAs; the epilogue
// computes fmaf(sum, gs, R) with one rounding.
#pragma once

#include <cuda_bf16.h>

#include "sgr_e4m3.cuh"
#include "sgr_ptx.cuh"

namespace sgr {

constexpr int kSimtConsumerWarps = 7;
constexpr int kSimtConsumers = kSimtConsumerWarps * 32;  // 224 threads
constexpr int kSimtThreads = kSimtConsumers + 32;        // + one producer warp
constexpr int kSimtRPrefetch = 4;  // reduction batches whose residuals are loaded early

// Weight formats of the kernel (template parameter WF).
enum : int { kWfBf16 = 0, kWfE4m3 = 1, kWfNvfp4 = 2 };

// Bytes of one NVFP4 ring record: a row's K/2 code bytes, then its ceil(K/16)
// block scales padded to 16 bytes (K a multiple of 32).
__host__ __device__ constexpr uint32_t simt_w4_scale_bytes(int K) { return (uint32_t)(((K + 15) / 16 + 15) / 16 * 16); }
__host__ __device__ constexpr uint32_t simt_w4_record_bytes(int K) { return (uint32_t)(K / 2) + simt_w4_scale_bytes(K); }

struct SimtParams {
  const __nv_bfloat16* A;  // [M, K], row stride lda (elements)
  const __nv_bfloat16* W;  // [N, K], contiguous rows (BF16 weights)
  const uint8_t* Wq;       // E4M3: [N, K] contiguous rows of codes; NVFP4: [N, K/2] bytes, row stride ldw
  const float* scale;      // [N] per-column scales (E4M3 only)
  const uint8_t* bs;       // NVFP4: [N, ceil(K/16)] E4M3 block scales, row stride ldbs bytes
  long long ldw, ldbs;     // NVFP4 row strides (bytes, multiples of 16)
  float gs;                // NVFP4 tensor scale
  const __nv_bfloat16* R;  // [M, N], row stride ldr
  __nv_bfloat16* Y;        // [M, N], row stride ldy
  long long lda, ldr, ldy;
  int M, N, K;
  int rows_per_stage;  // W rows per ring stage
  int stages;          // ring depth
  unsigned* err;       // device error word
};

// Shared-memory layout (dynamic): [full bars][empty bars][partials 2x7x32 f32][pad][ring]
__host__ __device__ constexpr size_t simt_ring_offset(int stages) {
  return ((size_t)stages * 16 + 2 * kSimtConsumerWarps * 32 * 4 + 127) / 128 * 128;
}

__host__ __device__ constexpr size_t simt_smem_bytes(int stages, int rows_per_stage, int K, int elem_bytes = 2) {
  return simt_ring_offset(stages) + (size_t)stages * rows_per_stage * K * elem_bytes;
}

// Butterfly over 32 lanes that also transposes: on entry each lane holds 32
// partial sums x[0..31]; on exit lane l returns the sum over all lanes of x[l].
template <int CNT>
__device__ __forceinline__ void transpose_reduce_step(float (&x)[32], int lane) {
  const bool upper = (lane & CNT) != 0;
#pragma unroll
  for (int i = 0; i < CNT; ++i) {
    const float send = upper ? x[i] : x[i + CNT];
    const float keep = upper ? x[i + CNT] : x[i];
    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, CNT);
  }
}

__device__ __forceinline__ float transpose_reduce32(float (&x)[32], int lane) {
  transpose_reduce_step<16>(x, lane);
  transpose_reduce_step<8>(x, lane);
  transpose_reduce_step<4>(x, lane);
  transpose_reduce_step<2>(x, lane);
  transpose_reduce_step<1>(x, lane);
  return x[0];
}

// MT: rows of A handled (M <= MT, rows >= M masked); VPT: 16-byte K vectors
// per consumer thread (K <= 224 * EPV * VPT); WF: weight format (BF16, E4M3
// codes + per-column scales, NVFP4 codes + block scales + tensor scale).
template <int MT, int VPT, int WF = kWfBf16>
__global__ void __launch_bounds__(kSimtThreads,
                                  (WF == kWfNvfp4 ? (MT <= 2 ? 2 : 1) : (MT <= 2 ? 3 : (MT <= 4 ? 2 : 1))))
    simt_skinny_kernel(const SimtParams p) {
  constexpr bool W8 = WF == kWfE4m3;
  constexpr bool W4 = WF == kWfNvfp4;
  constexpr int B = 32 / MT;                      // rows per reduction batch
  constexpr int EPV = W4 ? 32 : (W8 ? 16 : 8);    // weight elements per 16-byte vector
  constexpr bool kPackedA = MT * VPT * EPV > 64;  // keep A as bf16x2 when large
  extern __shared__ __align__(128) unsigned char smem[];

  const int S = p.stages;
  const int RS = p.rows_per_stage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + S;
  float* partial = reinterpret_cast<float*>(empty + S);  // [2][7][32]
  const __nv_bfloat16* ring =
      reinterpret_cast<const __nv_bfloat16*>(smem + simt_ring_offset(S));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int n0 = (int)((long long)p.N * c / G);
  const int n1 = (int)((long long)p.N * (c + 1) / G);
  const int nrows = n1 - n0;
  const int nstages = (nrows + RS - 1) / RS;
  const int KV = W4 ? (p.K >> 5) : (W8 ? (p.K >> 4) : (p.K >> 3));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kSimtConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncwarp();
  __syncthreads();
  // The dependent grid may be scheduled now: its own griddepcontrol.wait
  // still orders its reads of our outputs after this grid completes.
  pdl_launch_dependents();

  if (warp == kSimtConsumerWarps) {
    // ---------------- producer: stream this CTA's W slab through the ring
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t row_bytes = W4 ? simt_w4_record_bytes(p.K) : (uint32_t)p.K * (W8 ? 1u : 2u);
      const char* wbase = (W8 ? reinterpret_cast<const char*>(p.Wq) : reinterpret_cast<const char*>(p.W)) +
                          (size_t)n0 * row_bytes;
      // NVFP4: each record is gathered from the code row and the scale row.
      const char* cbase = reinterpret_cast<const char*>(p.Wq) + (W4 ? (size_t)n0 * (size_t)p.ldw : 0);
      const char* sbase = reinterpret_cast<const char*>(p.bs) + (W4 ? (size_t)n0 * (size_t)p.ldbs : 0);
      const uint32_t code_bytes = (uint32_t)(p.K / 2), scale_bytes = simt_w4_scale_bytes(p.K);
      // Ring position kept by increments: no integer division on the
      // per-stage path of this single issuing thread.
      int issued = 0;
      int slot = 0;
      uint32_t par = 0;  // ring round parity of `slot`
      const uint32_t ring0 = smem_u32(ring);
      const uint32_t stage_bytes = (uint32_t)RS * row_bytes;
      uint32_t dst = ring0;
      const char* src = wbase;
      int left = nrows;
      for (int s = 0; s < nstages; ++s) {
        if (s >= S && !mbar_wait(smem_u32(&empty[slot]), par ^ 1u)) {
          report_error(p.err, kErrWaitEmpty);
          break;
        }
        const uint32_t bytes = left < RS ? (uint32_t)left * row_bytes : stage_bytes;
        const uint32_t fb = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(fb, bytes);
        if constexpr (W4) {
          const int rows = left < RS ? left : RS;
          for (int r = 0; r < rows; ++r) {
            const uint32_t d = dst + (uint32_t)r * row_bytes;
            bulk_g2s(d, cbase, code_bytes, fb, pol);
            bulk_g2s(d + code_bytes, sbase, scale_bytes, fb, pol);
            cbase += p.ldw;
            sbase += p.ldbs;
          }
        } else {
          bulk_g2s(dst, src, bytes, fb, pol);
        }
        issued = s + 1;
        left -= RS;
        src += stage_bytes;
        dst += stage_bytes;
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
          dst = ring0;
        }
      }
      // Before this CTA can exit, every copy it issued must have landed.
      for (int t = max(0, issued - S); t < issued; ++t) {
        if (!mbar_wait(smem_u32(&full[t % S]), (t / S) & 1)) {
          report_error(p.err, kErrDrain);
          break;
        }
      }
    }
    return;
  }

  // ---------------- consumers
  pdl_wait();  // A and R may be produced by the preceding kernel; Y may be read by it

  // This thread's K slice of A (EPV elements per vector), loaded once.
  float af[kPackedA ? 1 : MT][kPackedA ? 1 : VPT][EPV];
  uint32_t ap[kPackedA ? MT : 1][kPackedA ? VPT : 1][EPV / 2];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int vid = threadIdx.x + v * kSimtConsumers;
#pragma unroll
      for (int h = 0; h < EPV / 8; ++h) {
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (m < p.M && vid < KV)
          q = *reinterpret_cast<const uint4*>(p.A + (size_t)m * p.lda + (size_t)vid * EPV + h * 8);
        if constexpr (kPackedA) {
          ap[m][v][4 * h + 0] = q.x; ap[m][v][4 * h + 1] = q.y; ap[m][v][4 * h + 2] = q.z; ap[m][v][4 * h + 3] = q.w;
        } else {
          af[m][v][8 * h + 0] = bf16lo(q.x); af[m][v][8 * h + 1] = bf16hi(q.x);
          af[m][v][8 * h + 2] = bf16lo(q.y); af[m][v][8 * h + 3] = bf16hi(q.y);
          af[m][v][8 * h + 4] = bf16lo(q.z); af[m][v][8 * h + 5] = bf16hi(q.z);
          af[m][v][8 * h + 6] = bf16lo(q.w); af[m][v][8 * h + 7] = bf16hi(q.w);
        }
      }
    }
  }

  // Residuals of the first batches, loaded now so the epilogue does not wait
  // on memory (warp 0 stores; lane l handles output l of each batch).
  constexpr int kB = 32 / MT;
  float rpre[kSimtRPrefetch];
  float spre[W8 ? kSimtRPrefetch : 1];  // scales * 2^8 of the same outputs (E4M3)
#pragma unroll
  for (int b = 0; b < kSimtRPrefetch; ++b) {
    const int j = lane / MT, m = lane % MT, row = b * kB + j;
    rpre[b] = (warp == 0 && row < nrows && m < p.M)
                  ? __bfloat162float(p.R[(size_t)m * p.ldr + n0 + row])
                  : 0.f;
    if constexpr (W8) spre[b] = (warp == 0 && row < nrows) ? p.scale[n0 + row] * kE4m3Unscale : 0.f;
  }

  bool ok = true;
  int buf = 0;
  int bi = 0;  // reduction batch index
  int slot = 0, rr = 0;   // ring slot of the current stage, row within the stage
  uint32_t phase = 0;     // parity of the current stage's fill of that slot
  const uint32_t ring_base = smem_u32(ring);
  const uint32_t row_bytes = W4 ? simt_w4_record_bytes(p.K) : (uint32_t)p.K * (W8 ? 1u : 2u);
  const uint32_t code_bytes = (uint32_t)(p.K / 2);  // NVFP4: block scales follow the codes
  uint32_t row_addr = ring_base;
  for (int base = 0; base < nrows; base += B, ++bi) {
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;

#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (base + j < nrows) {
        if (rr == 0 && ok && !mbar_wait(smem_u32(&full[slot]), phase)) {
          report_error(p.err, kErrWaitFull);
          ok = false;
        }
        if (ok) {
#pragma unroll
          for (int v = 0; v < VPT; ++v) {
            const int vid = threadIdx.x + v * kSimtConsumers;
            if (vid < KV) {
              const uint4 q = lds128(row_addr + (uint32_t)vid * 16u);
              if constexpr (W4) {
                // Block scales of codes [0, 16) and [16, 32) of this vector, as FP16.
                uint16_t sc2;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(sc2) : "r"(row_addr + code_bytes + (uint32_t)vid * 2u));
                uint32_t s0, s1;
                e4m3x2_block_scales_f16(sc2, s0, s1);
                const uint32_t x[4] = {q.x, q.y, q.z, q.w};
                // One 8-code word at a time: decode, then its FMAs for every token.
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  uint32_t hx[4];
                  e2m1x8_to_f16x2(x[i], hx);
                  float w8[8];
#pragma unroll
                  for (int b = 0; b < 4; ++b) {
                    uint32_t h = hx[b];
                    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h) : "r"(i < 2 ? s0 : s1));  // exact
                    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\t"
                        "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, u;\n\t}"
                        : "=f"(w8[2 * b]), "=f"(w8[2 * b + 1]) : "r"(h));
                  }
#pragma unroll
                  for (int m = 0; m < MT; ++m) {
                    float t = acc[j * MT + m];
                    if constexpr (kPackedA) {
#pragma unroll
                      for (int e = 0; e < 4; ++e) {
                        t = fmaf(bf16lo(ap[m][v][4 * i + e]), w8[2 * e], t);
                        t = fmaf(bf16hi(ap[m][v][4 * i + e]), w8[2 * e + 1], t);
                      }
                    } else {
#pragma unroll
                      for (int e = 0; e < 8; ++e) t = fmaf(af[m][v][8 * i + e], w8[e], t);
                    }
                    acc[j * MT + m] = t;
                  }
                }
              } else {
              float w[EPV];
              uint32_t wp[EPV / 2];  // weights as BF16 pairs
              if constexpr (W8) {
                const uint32_t x[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  wp[2 * i] = e4m3x2_to_bf16x2_scaled<0x9180u>(x[i]);
                  wp[2 * i + 1] = e4m3x2_to_bf16x2_scaled<0xB3A2u>(x[i]);
                }
              } else {
                wp[0] = q.x; wp[1] = q.y; wp[2] = q.z; wp[3] = q.w;
              }
#pragma unroll
              for (int i = 0; i < EPV / 2; ++i) {
                w[2 * i] = bf16lo(wp[i]);
                w[2 * i + 1] = bf16hi(wp[i]);
              }
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                float t = acc[j * MT + m];
                if constexpr (kPackedA) {
#pragma unroll
                  for (int e = 0; e < EPV / 2; ++e) {
                    t = fmaf(bf16lo(ap[m][v][e]), w[2 * e], t);
                    t = fmaf(bf16hi(ap[m][v][e]), w[2 * e + 1], t);
                  }
                } else {
#pragma unroll
                  for (int e = 0; e < EPV; ++e) t = fmaf(af[m][v][e], w[e], t);
                }
                acc[j * MT + m] = t;
              }
              }
            }
          }
        }
        // Release the stage after its last row.
        if (rr == RS - 1 || base + j == nrows - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
        }
        row_addr += row_bytes;
        if (++rr == RS) {
          rr = 0;
          if (++slot == S) {
            slot = 0;
            phase ^= 1u;
            row_addr = ring_base;
          }
        }
      }
    }

    // K reduction: within the warp, then across the 7 consumer warps.
    const float mine = transpose_reduce32(acc, lane);
    partial[(buf * kSimtConsumerWarps + warp) * 32 + lane] = mine;
    named_bar_sync(1, kSimtConsumers);
    if (warp == 0) {
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kSimtConsumerWarps; ++w)
        total += partial[(buf * kSimtConsumerWarps + w) * 32 + lane];
      const int j = lane / MT, m = lane % MT;
      if (base + j < nrows && m < p.M) {
        const int n = n0 + base + j;
        float r = 0.f;
#pragma unroll
        for (int k = 0; k < kSimtRPrefetch; ++k)
          if (k == bi) r = rpre[k];
        if (bi >= kSimtRPrefetch) r = __bfloat162float(p.R[(size_t)m * p.ldr + n]);
        if constexpr (W8) {
          float sc = 0.f;
#pragma unroll
          for (int k = 0; k < kSimtRPrefetch; ++k)
            if (k == bi) sc = spre[k];
          if (bi >= kSimtRPrefetch) sc = p.scale[n] * kE4m3Unscale;
          p.Y[(size_t)m * p.ldy + n] = __float2bfloat16_rn(fmaf(total, sc, r));
        } else if constexpr (W4) {
          p.Y[(size_t)m * p.ldy + n] = __float2bfloat16_rn(fmaf(total, p.gs, r));
        } else {
          p.Y[(size_t)m * p.ldy + n] = __float2bfloat16_rn(total + r);
        }
      }
    }
    buf ^= 1;
  }
}

}  // namespace sgr
