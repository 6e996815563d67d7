// sgr_rows.cuh -- tensor-core row-slab path for decode-sized M.
//
// Same operation as the other kernels: Y[m,n] = bf16_rn( sum_k A[m,k] W[n,k]
// + R[m,n] ) with FP32 accumulation and one rounding (vLLM
// "benchmark_k3_cutedsl_residual.py", module docstring).
//
// Decomposition: like the SIMT kernel (and unlike the stream-K tensor-core
// kernel) every CTA owns a contiguous slab of RB whole rows of W, RB =
// ceil(N / SMs) rounded up to 8 (48 for N = 7168 on 152 SMs), so no output
// element is split across CTAs: no workspace, no counters, no fixup tail.
// The slab is streamed once with 2-D TMA boxes of RB rows x 64 K into a
// shared-memory ring and multiplied on the tensor core with
// tcgen05.mma M=128 (W rows) x N=NT (tokens) x K=16.  The ring stores only
// the RB loaded rows per K block; the MMA's 128-row window over-reads into the
// following bytes of shared memory (the next W blocks, then the A ring that
// follows the W ring, then slack if needed), and those extra rows only feed
// TMEM lanes >= RB, which the epilogue never reads (each output row of an MMA
// depends only on its own operand row).  At about 100 KB of shared memory per
// CTA the next call's CTA fits on the same SM, so with programmatic dependent
// launch it streams its weights while this one finishes.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA (W for the first stages
// before griddepcontrol.wait, A after it); warp 1 owns TMEM and lane 0 issues
// the MMAs; warps 2-5 are the epilogue: they load their residual values while
// the MMAs run, then tcgen05.ld the accumulator, add, round once and store.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sgr_ptx.cuh"
#include "sgr_tc.cuh"
#include "skinny_gemm_residual.h"

namespace sgr {

constexpr int kRowsThreads = 192;
constexpr int kRowsMaxTokens = 256;
constexpr int kRowsPrefetchTokens = 32;  // residual values held in registers before the MMAs end
constexpr uint32_t kRowsSlack = kTcTileRows * 128u;  // MMA window over-read past the ring

struct RowsParams {
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  long long ldr, ldy;
  unsigned* err;
  int M, N, K;
  int RB;        // W rows per CTA (multiple of 8, <= 128)
  int NT;        // token tile = MMA N (multiple of 16, >= M)
  int k_stages;  // ceil(K / (64 * kbps))
  int kbps;      // 64-wide K blocks per stage
  int stages;    // ring depth
  int chains;    // independent TMEM accumulators (1, 2 or 4), summed in the epilogue
  int tmem_cols;
};

__host__ __device__ inline uint32_t rows_stage_bytes(int kbps, int rb, int nt) {
  return (uint32_t)kbps * ((uint32_t)rb * 128u + (uint32_t)nt * 128u);
}

// Bytes past the end of the A ring that the last W block's 128-row MMA window
// can touch (the W ring is followed by the A ring, which absorbs the rest).
__host__ __device__ inline uint32_t rows_tail_slack(int stages, int kbps, int rb, int nt) {
  const uint32_t over = kRowsSlack - (uint32_t)rb * 128u;
  const uint32_t a_ring = (uint32_t)stages * kbps * nt * 128u;
  return over > a_ring ? over - a_ring : 0u;
}

__host__ __device__ inline size_t rows_smem_bytes(int stages, int kbps, int rb, int nt) {
  return 1024 /* alignment slack */ + 1024 /* barriers */ +
         (size_t)stages * rows_stage_bytes(kbps, rb, nt) + rows_tail_slack(stages, kbps, rb, nt);
}

// 16 accumulator columns summed over the chains, chain 0 first (fixed order).
__device__ __forceinline__ void rows_ld_chains(uint32_t taddr, int nt, int chains, float (&v)[16]) {
  tmem_ld16(taddr, v);
  for (int c = 1; c < chains; ++c) {
    float w[16];
    tmem_ld16(taddr + (uint32_t)(c * nt), w);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += w[i];
  }
}

__global__ void __launch_bounds__(kRowsThreads, 1)
    rows_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                       const RowsParams p) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(sb);  // [S]
  uint64_t* empty = full + S;                         // [S]
  uint64_t* acc_full = empty + S;                     // [1]
  uint64_t* drain = acc_full + 1;                     // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t wblk = (uint32_t)p.RB * 128u;   // bytes of one W box (RB rows x 128 B)
  const uint32_t ablk = (uint32_t)p.NT * 128u;   // bytes of one A box
  const uint32_t w_stage = (uint32_t)p.kbps * wblk;
  const uint32_t a_stage = (uint32_t)p.kbps * ablk;
  const uint32_t stage_bytes = w_stage + a_stage;  // bytes one stage brings in
  const uint32_t w_ring = base + 1024;                         // [stages][kbps] W boxes
  const uint32_t a_ring = w_ring + (uint32_t)S * w_stage;      // [stages][kbps] A boxes

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * p.RB;
  const int KS = p.k_stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmA);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();  // the dependent grid still waits for our completion before reading

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      const int pre = KS < S ? KS : S;
      for (int s = 0; s < pre; ++s) {
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        const uint32_t ws = w_ring + (uint32_t)s * w_stage;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(ws + (uint32_t)j * wblk, &tmW, (s * p.kbps + j) * kTcKBlock, n0, fb, pol_w);
      }
      pdl_wait();
      for (int s = 0; s < pre; ++s) {
        const uint32_t as = a_ring + (uint32_t)s * a_stage;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(as + (uint32_t)j * ablk, &tmA, (s * p.kbps + j) * kTcKBlock, 0,
                      smem_u32(&full[s]), pol_a);
      }
      int issued = pre;
      for (int s = pre; s < KS; ++s) {
        const int slot = s % S;
        if (!mbar_wait_or_abort(smem_u32(&empty[slot]), ((s / S) - 1) & 1, abort_flag)) {
          if (!*abort_flag) report_error(p.err, kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        const uint32_t fb = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        const uint32_t ws = w_ring + (uint32_t)slot * w_stage;
        const uint32_t as = a_ring + (uint32_t)slot * a_stage;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(ws + (uint32_t)j * wblk, &tmW, (s * p.kbps + j) * kTcKBlock, n0, fb, pol_w);
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(as + (uint32_t)j * ablk, &tmA, (s * p.kbps + j) * kTcKBlock, 0, fb, pol_a);
        issued = s + 1;
      }
      for (int t = issued > S ? issued - S : 0; t < issued; ++t)
        if (!mbar_wait(smem_u32(&full[t % S]), (t / S) & 1)) {
          report_error(p.err, kErrDrain);
          break;
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTcTileRows, p.NT);
      // Descriptors differ only in their start-address field (address >> 4):
      // build the ring bases once and add offsets.
      const uint64_t wdesc0 = smem_desc_sw128(w_ring);
      const uint64_t adesc0 = smem_desc_sw128(a_ring);
      bool ok = true;
      for (int s = 0; s < KS; ++s) {
        const int slot = s % S;
        if (!mbar_wait_or_abort(smem_u32(&full[slot]), (s / S) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t wd = wdesc0 + ((uint64_t)(slot * w_stage) >> 4);
        const uint64_t ad = adesc0 + ((uint64_t)(slot * a_stage) >> 4);
        for (int j = 0; j < p.kbps; ++j) {
#pragma unroll
          for (int kk = 0; kk < kTcKBlock / 16; ++kk) {
            // K step kk goes to accumulator chain kk % chains.
            const int chain = kk & (p.chains - 1);
            const bool first = (s == 0) && (j == 0) && (kk < p.chains);
            mma_bf16(tmem + (uint32_t)(chain * p.NT), wd + ((j * wblk + kk * 32u) >> 4),
                     ad + ((j * ablk + kk * 32u) >> 4), idesc, first ? 0u : 1u);
          }
        }
        mma_commit(smem_u32(&empty[slot]));
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
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (q * 32 < p.RB) {  // warp-uniform: this quarter holds loaded rows
      pdl_wait();
      const int n = n0 + row;
      const bool live = row < p.RB && n < p.N;
      float r[kRowsPrefetchTokens];
#pragma unroll
      for (int i = 0; i < kRowsPrefetchTokens; ++i)
        r[i] = (live && i < p.M) ? __bfloat162float(p.R[(size_t)i * p.ldr + n]) : 0.f;
      bool ok = mbar_wait_or_abort(smem_u32(acc_full), 0, abort_flag);
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      if (ok) {
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        // Tokens [0, 32): residuals already in registers (static indices).
#pragma unroll
        for (int half = 0; half < kRowsPrefetchTokens / 16; ++half) {
          const int col0 = half * 16;
          if (col0 < p.NT) {
            float v[16];
            rows_ld_chains(taddr + (uint32_t)col0, p.NT, p.chains, v);
            if (live) {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (col0 + i < p.M)
                  p.Y[(size_t)(col0 + i) * p.ldy + n] = __float2bfloat16_rn(v[i] + r[col0 + i]);
            }
          }
        }
        // Tokens [32, NT): residuals loaded per group of 16.
        for (int col0 = kRowsPrefetchTokens; col0 < p.NT; col0 += 16) {
          float v[16], rr[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            rr[i] = (live && col0 + i < p.M) ? __bfloat162float(p.R[(size_t)(col0 + i) * p.ldr + n]) : 0.f;
          rows_ld_chains(taddr + (uint32_t)col0, p.NT, p.chains, v);
          if (live) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (col0 + i < p.M) p.Y[(size_t)(col0 + i) * p.ldy + n] = __float2bfloat16_rn(v[i] + rr[i]);
          }
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
inline int rows_per_cta(int sms, int N) {
  const int rb = (N + sms - 1) / sms;
  return (rb + 7) / 8 * 8;
}

inline bool rows_supported(int sms, int M, int N, int K) {
  return M >= 1 && M <= kRowsMaxTokens && N >= 8 && K >= 8 && N % 8 == 0 && K % 8 == 0 &&
         rows_per_cta(sms, N) <= kTcTileRows;
}

// Default: 4 K blocks per stage and the deepest ring (up to 4 stages) that
// keeps the CTA at or under ~110 KB of shared memory, so that the next call's
// CTA can be resident on the same SM; smaller stages if even 2 do not fit.
inline void rows_default_config(int sms, int M, int N, int K, sgr_config* c) {
  (void)K;
  c->path = SGR_PATH_TC_ROWS;
  c->ctas_per_sm = 1;
  c->token_tile = (M + 15) / 16 * 16;
  c->rows_per_stage = 0;
  const int rb = rows_per_cta(sms, N);
  const size_t budget = 110u * 1024u;
  for (int kb = 4; kb >= 1; kb /= 2)
    for (int st = 4; st >= 2; --st)
      if (rows_smem_bytes(st, kb, rb, c->token_tile) <= budget) {
        c->k_blocks_per_stage = kb;
        c->stages = st;
        return;
      }
  c->k_blocks_per_stage = 1;
  c->stages = 2;
}

inline int rows_plan(const sgr_config& c, int sms, int M, int N, int K, RowsParams* p, int* grid,
                     size_t* smem) {
  if (!rows_supported(sms, M, N, K)) return SGR_ERR_UNSUPPORTED;
  const int nt = c.token_tile;
  if (nt < 16 || nt > kRowsMaxTokens || nt % 16 != 0 || nt < M) return SGR_ERR_UNSUPPORTED;
  if (c.k_blocks_per_stage < 1 || c.k_blocks_per_stage > 8) return SGR_ERR_UNSUPPORTED;
  if (c.ctas_per_sm != 1) return SGR_ERR_UNSUPPORTED;
  if (c.stages < 2 || c.stages > 32) return SGR_ERR_UNSUPPORTED;
  const int rb = rows_per_cta(sms, N);
  const size_t sm = rows_smem_bytes(c.stages, c.k_blocks_per_stage, rb, nt);
  if (sm > 232448) return SGR_ERR_UNSUPPORTED;
  const int kstage_elems = kTcKBlock * c.k_blocks_per_stage;
  p->M = M;
  p->N = N;
  p->K = K;
  p->RB = rb;
  p->NT = nt;
  p->k_stages = (K + kstage_elems - 1) / kstage_elems;
  p->kbps = c.k_blocks_per_stage;
  p->stages = c.stages;
  p->chains = nt <= 128 ? 4 : 2;  // chains * NT <= 512 TMEM columns
  p->tmem_cols = detail::pow2_at_least(p->chains * nt);
  *grid = (N + rb - 1) / rb;
  *smem = sm;
  return SGR_OK;
}

inline cudaError_t rows_init_device() {
  return set_kernel_smem_attrs(reinterpret_cast<const void*>(rows_skinny_kernel));
}

inline int rows_launch(const sgr_config& c, int sms, unsigned* err, const void* A, long long lda,
                       const void* W, const void* R, long long ldr, void* Y, long long ldy, int M,
                       int N, int K, bool pdl, cudaStream_t stream) {
  RowsParams p;
  int grid = 0;
  size_t smem = 0;
  int rc = rows_plan(c, sms, M, N, K, &p, &grid, &smem);
  if (rc != SGR_OK) return rc;
  CUtensorMap tmW, tmA;
  if (!detail::make_tmap(&tmW, W, N, K, K, p.RB, kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap(&tmA, A, M, K, lda, p.NT, kTcKBlock)) return SGR_ERR_LAUNCH;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.ldr = ldr;
  p.ldy = ldy;
  p.err = err;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kRowsThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&lc, rows_skinny_kernel, tmW, tmA, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

}  // namespace sgr
