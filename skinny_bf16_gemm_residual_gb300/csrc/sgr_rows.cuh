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
// (Except under the 2-CTA K split, k_split = 2, for long K with few rows per
// SM, as in the down-projection N = 3584, K = 7168: each slab goes to a
// 2-CTA cluster whose rank r streams the r-th half of K, i.e. 48-row slabs of
// half of K instead of 24-row slabs of all of it, and the epilogue adds the
// peer's partial sums read through distributed shared memory; rank 0
// finishes the slab's first RB / 2 columns, rank 1 the others.)
// The slab is streamed once with 2-D TMA boxes of RB rows x 64 K into a
// shared-memory ring and multiplied on the tensor core with
// tcgen05.mma M=128 (W rows) x N=G*NT (tokens) x K=16.
//
// Diagonal packing: the W boxes of consecutive K blocks sit back to back in
// the ring, so a 128-row MMA window starting at block j holds block j in rows
// [0, RB), block j+1 in rows [RB, 2 RB), ...; the activation boxes sit back to
// back too, so an N = G*NT window holds the tokens of blocks j .. j+G-1.  One
// MMA then computes G useful diagonal blocks D[g RB + r, g NT + t] (block
// j+g of W against block j+g of A) plus cross terms that are never read.
// With RB = 48 this is G = 2: half the MMAs and half the shared-memory reads
// of the W operand, which is what bounds a 16-token MMA.  The epilogue sums
// the G diagonal blocks (in g order) through shared memory.  The ring stores only
// the RB loaded rows per K block; the MMA's 128-row window over-reads into the
// following bytes of shared memory (the next W blocks, then the A ring that
// follows the W ring, then slack if needed), and those extra rows only feed
// TMEM lanes >= RB, which the epilogue never reads (each output row of an MMA
// depends only on its own operand row).  At about 100 KB of shared memory per
// CTA the next call's CTA fits on the same SM, so with programmatic dependent
// launch it streams its weights while this one finishes.
//
// Warp roles: warp 0 lane 0 issues TMA (W for the first stages before
// griddepcontrol.wait, A after it); warp 1 owns TMEM and its lane 0 issues
// the MMAs, or, with two issuers (16-token tiles, 224 threads), the even MMA
// windows of every stage while lane 0 of warp 6 issues the odd ones into a
// second accumulator (one thread issues a small-N MMA only every ~75 cycles,
// which left the last stage's MMAs exposed after its weights landed; the
// epilogue adds the two accumulators in a fixed order); warps 2-5 are the
// epilogue: they load their residual values while the MMAs run, then
// tcgen05.ld the accumulator, add, round once and store.
//
// One kernel instance per epilogue family (16-token tiles with one or two
// packed groups, and with three or four, both with 224 threads; 32- and
// 48-token tiles and the general form; 64-token tiles), each compiled with
// only its own epilogue code and issuer count.
//
// Warm-up pass: the first run of a code path in a CTA costs ~0.7 us more
// than the next (measured with the weight stream saturating L2: instruction
// and parameter fetches wait behind it), and the epilogue runs once, on the
// critical path after the last weights land.  So the 16- to 64-token
// epilogues run their instructions twice: first while the MMAs are still running, against tensor-
// memory columns no MMA writes, a scratch word of shared memory and stores
// predicated off, then for real.
//
// For up to 16 tokens the epilogue is one TMEM load, one shared-memory
// hand-over of group 1's partial sums and the stores, with the residuals and
// addresses prepared while the MMAs run: it sits on the critical path after
// the last weight byte lands, so it is kept short (counting each stage's
// packed groups on separate barriers, to start the last stage's MMAs early,
// measured slower).  Token tiles of 32, 48 and 64 use the same register form
// with the accumulator loaded in 16-column pieces (rows_epilogue_wide; the
// 64-token form in its own kernel instance because of its register count);
// only larger tiles stage partial sums through shared memory.
#pragma once

#include <cstring>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sgr_ptx.cuh"
#include "sgr_epi.cuh"
#include "sgr_tc.cuh"
#include "skinny_gemm_residual.h"

namespace sgr {

// Epilogue families (kernel instances) and their block sizes.
// kRowsEpi16: 16-token tiles with one or two packed groups; kRowsEpi16G4:
// 16-token tiles with three or four (short slabs); both with a second MMA
// issuer (224 threads).  The two are separate instances so that each keeps
// its register budget for two CTAs per SM without spills.
enum RowsEpi : int { kRowsEpi16 = 0, kRowsEpiWide = 1, kRowsEpi64 = 2, kRowsEpi16G4 = 3 };
__host__ __device__ constexpr bool rows_two_issuer_mode(int mode) { return mode == 0 || mode == 3; }
__host__ __device__ constexpr int rows_threads(int mode) { return rows_two_issuer_mode(mode) ? 224 : 192; }
__host__ __device__ inline int rows_epi_mode(int nt, int groups) {
  return nt == 16 ? (groups <= 2 ? kRowsEpi16 : kRowsEpi16G4)
                  : (nt == 64 && groups <= 2 ? kRowsEpi64 : kRowsEpiWide);
}
constexpr int kRowsMaxTokens = 256;
constexpr int kRowsPrefetchTokens = 16;  // residual values held in registers before the MMAs end
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
  int groups;    // K blocks packed into one MMA along its diagonal (1, 2 or 4)
  int prefetch;  // W stages requested before griddepcontrol.wait (1..stages)
  int issuers;   // MMA-issuing threads (1 or 2), each into its own accumulator
  int tmem_cols;
  int ksplit;    // 1, or 2: K split over a 2-CTA cluster (rank r takes K blocks from r k_stages kbps on)
};

// Scratch bytes of the decode epilogue's warm-up pass: the end of the
// 1024-byte barrier region (at most 32 stages: 2 x 32 + 3 barriers, the TMEM
// address and the abort flag end at byte 544).
constexpr uint32_t kRowsWarmScratch = 960;

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

// Scratch of the 17-64-token epilogues' warm-up pass, after the rings and
// the MMA window's over-read slack (no MMA reads it); the 16-token epilogues
// use the end of the barrier region instead.
constexpr uint32_t kRowsWideScratch = 512;

__host__ __device__ inline size_t rows_smem_bytes(int stages, int kbps, int rb, int nt) {
  return 1024 /* alignment slack */ + 1024 /* barriers */ +
         (size_t)stages * rows_stage_bytes(kbps, rb, nt) + rows_tail_slack(stages, kbps, rb, nt) +
         (nt > 16 ? kRowsWideScratch : 0);
}

// Shared-memory staging for the epilogue's sum over packed groups:
// [groups][RB][NT + 4] floats (the +4 spreads rows over banks).
__host__ __device__ inline size_t rows_stage_floats(int groups, int rb, int nt) {
  return (size_t)groups * rb * (nt + 4);
}

// One problem's operands: the tensor maps of W and A (in kernel parameter
// space) and the residual / output.
struct RowsIO {
  const CUtensorMap* tmW;
  const CUtensorMap* tmA;
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  long long ldr, ldy;
  int M;
};

// Bytes per row of the epilogues' hand-over buffers in the drained ring: the
// group-1 partial sums at rows [0, RB), and under the 2-CTA K split the
// partial sums the peer finishes at rows [RB, 2 RB).
__host__ __device__ inline uint32_t rows_xch_stride(int nt) { return nt == 16 ? 80u : (uint32_t)(nt + 4) * 4u; }

// 2-CTA K split: owner thread L of either rank holds that rank's partial sums
// v[0..T) of output column n0 + L; rank 0 finishes the columns L < RB / 2,
// rank 1 the others.  A thread whose column the peer finishes leaves its
// partial sums in its own drained ring at `xo`; every epilogue thread then
// arrives once on the peer's `ready` barrier (releasing those writes at
// cluster scope) and waits for the peer's 128 arrivals on its own; a
// finishing thread adds the peer's partial sums, read at the same offset of
// the peer's shared memory (the sum of two terms is the same in either
// order).  Returns false after a timed-out wait (reported).
template <int T>
__device__ __forceinline__ bool rows_pair_exchange(float (&v)[T], bool has, bool fin, uint32_t xo, uint64_t* ready,
                                                   uint32_t rank, volatile int* abort_flag, unsigned* err) {
  if (has && !fin) {
#pragma unroll
    for (int i = 0; i < T; i += 4)
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(xo + (uint32_t)i * 4u), "f"(v[i]), "f"(v[i + 1]),
                   "f"(v[i + 2]), "f"(v[i + 3])
                   : "memory");
  }
  mbar_arrive_remote(map_to_rank(smem_u32(ready), rank ^ 1u));
  bool got = mbar_wait_cluster(smem_u32(ready), 0, abort_flag);
  got = __all_sync(0xffffffffu, got);
  if (!got) {
    if (!*abort_flag) report_error(err, kErrWaitFixup);
    *abort_flag = 1;
    return false;
  }
  if (has && fin) {
    const uint32_t src = map_to_rank(xo, rank ^ 1u);
#pragma unroll
    for (int i = 0; i < T; i += 4) {
      const float4 o = ld_cluster_f32x4(src + (uint32_t)i * 4u);
      v[i] += o.x;
      v[i + 1] += o.y;
      v[i + 2] += o.z;
      v[i + 3] += o.w;
    }
  }
  return true;
}

// Epilogue for 17..64 tokens (token tile T = 32, 48 or 64) with at most two
// packed groups: the ownership of the 16-token decode epilogue (lane r < RB
// owns output column n0 + r, lane RB + r holds group 1's partial sums and
// hands them over through the drained ring), with T accumulator columns per
// group loaded in 16-column pieces and the residuals of all T token rows
// loaded into registers before the accumulator is ready.  Like the 16-token
// epilogue it first runs a warm-up pass over its instructions while the MMAs
// run (tensor-memory columns after the accumulator, which no MMA writes, the
// exchange in `scratch`, stores predicated off; kWarm false skips it).
// Under the 2-CTA K split (kSplit) the partial sums are completed by
// rows_pair_exchange before the residual add.  Called by the
// four epilogue warps (q: TMEM lane quarter of the warp).
template <int T, bool kWarm, bool kSplit>
__device__ __forceinline__ void rows_epilogue_wide(const RowsParams& p, const RowsIO& io, int n0, uint32_t tmem,
                                                   uint32_t w_ring, uint32_t scratch, uint64_t* acc_full,
                                                   uint64_t* ready, volatile int* abort_flag, int q, int lane) {
  constexpr int C = T / 16;
  const int L = q * 32 + lane;
  const int G = p.groups;
  const bool owner = L < p.RB && n0 + L < p.N;
  // Under the K split this rank stores column n0 + L only if fin (the rank is
  // read again where needed rather than held through the epilogue).
  constexpr bool split = kSplit;
  bool fin = true;
  if constexpr (kSplit) fin = (L < p.RB / 2) == (cluster_ctarank() == 0u);
  const bool helper = G == 2 && L >= p.RB && L < 2 * p.RB;
  const int r = owner ? L : L - p.RB;
  const uint32_t stride = rows_xch_stride(T);  // T floats + pad per row
  const uint32_t xch = w_ring + (uint32_t)(helper || owner ? r : 0) * stride;
  // Residuals kept as BF16 pairs (half the registers of FP32 values).
  const unsigned short* rp = reinterpret_cast<const unsigned short*>(io.R) + n0 + L;
  uint32_t res2[T / 2];
#pragma unroll
  for (int m = 0; m < T; m += 2) {
    const uint32_t lo = (owner && fin && m < io.M) ? rp[(size_t)m * io.ldr] : 0u;
    const uint32_t hi = (owner && fin && m + 1 < io.M) ? rp[(size_t)(m + 1) * io.ldr] : 0u;
    res2[m / 2] = lo | (hi << 16);
  }
#pragma unroll 1
  for (int pass = kWarm ? 0 : 1; pass < 2; ++pass) {
    int passv;  // opaque to the compiler: one copy of the loop body serves both passes
    asm volatile("mov.b32 %0, %1;" : "=r"(passv) : "r"(pass));
    const bool real = passv != 0;
    bool ok = true;
    if (real) {
      ok = mbar_wait_or_abort(smem_u32(acc_full), 0, abort_flag);
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      ok = __all_sync(0xffffffffu, ok);
    }
    tc_fence_after();
    float v[T];
#pragma unroll
    for (int i = 0; i < T; ++i) v[i] = 0.f;
    if (ok && q * 32 < G * p.RB) {  // warp-uniform: this warp holds rows of the MMA window in use
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (real ? 0u : (uint32_t)(G * T));
      // Columns [0, T) hold group 0's diagonal block, [T, 2T) group 1's.
      const bool straddle = G == 2 && q * 32 < p.RB && (q + 1) * 32 > p.RB;
      const uint32_t col0 = (G == 2 && q * 32 >= p.RB) ? (uint32_t)T : 0u;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        float a[16];
        tmem_ld16(taddr + col0 + (uint32_t)(16 * c), a);  // warp-collective
        if (straddle) {
          float b[16];
          tmem_ld16(taddr + (uint32_t)(T + 16 * c), b);
          if (L >= p.RB) {
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] = b[i];
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * c + i] = a[i];
      }
    }
    const uint32_t x = real ? xch : scratch;
    if (ok && helper) {
#pragma unroll
      for (int i = 0; i < T; i += 4)
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(x + (uint32_t)i * 4u), "f"(v[i]),
                     "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                     : "memory");
    }
    named_bar_sync(1, 128);
    if (ok && owner && G == 2) {
#pragma unroll
      for (int i = 0; i < T; i += 4) {
        float a0, a1, a2, a3;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                     : "r"(x + (uint32_t)i * 4u)
                     : "memory");
        v[i] += a0;
        v[i + 1] += a1;
        v[i + 2] += a2;
        v[i + 3] += a3;
      }
    }
    if constexpr (split)
      if (real)
        ok = rows_pair_exchange<T>(v, ok && owner, fin, xch + (uint32_t)p.RB * stride, ready, cluster_ctarank(),
                                 abort_flag, p.err) &&
           ok;
    if (ok && owner && fin) {
      __nv_bfloat16* yp = io.Y + n0 + L;
#pragma unroll
      for (int m = 0; m < T; ++m) {
        const float rm = (m & 1) ? bf16hi(res2[m / 2]) : bf16lo(res2[m / 2]);
        st_global_bf16_if(yp + (size_t)m * io.ldy, __float2bfloat16_rn(v[m] + rm), real && m < io.M);
      }
    }
  }
}

// One CTA: the RB-row slab of W starting at row n0 of the problem `io`, with
// the epilogue family kMode (the 64-token register epilogue needs more
// registers per thread: only its own instance has it, so that the others
// keep two CTAs per SM where their shared memory allows); kWideWarm: the
// 17-64-token register epilogues run their warm-up pass; kSplit: the 2-CTA
// K split (p.ksplit == 2), in instances of its own so that the others carry
// none of its code.
template <int kMode, bool kWideWarm, bool kSplit>
__device__ __forceinline__ void rows_run(const RowsParams& p, const RowsIO& io, int n0) {
  const int issuers = rows_two_issuer_mode(kMode) ? p.issuers : 1;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(sb);  // [S]
  uint64_t* empty = full + S;                         // [S]
  uint64_t* acc_full = empty + S;                     // [1]
  uint64_t* drain = acc_full + 1;                     // [1]
  uint64_t* ready = drain + 1;                        // [1] the K-split peer's partial sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr bool split = kSplit;  // p.ksplit == 2 (its own kernel instances)
  const uint32_t rank = split ? cluster_ctarank() : 0u;
  const uint32_t wblk = (uint32_t)p.RB * 128u;   // bytes of one W box (RB rows x 128 B)
  const uint32_t ablk = (uint32_t)p.NT * 128u;   // bytes of one A box
  const uint32_t w_stage = (uint32_t)p.kbps * wblk;
  const uint32_t a_stage = (uint32_t)p.kbps * ablk;
  const uint32_t stage_bytes = w_stage + a_stage;  // bytes one stage brings in
  const uint32_t w_ring = base + 1024;                         // [stages][kbps] W boxes
  const uint32_t a_ring = w_ring + (uint32_t)S * w_stage;      // [stages][kbps] A boxes
  const uint32_t wide_scratch =  // after the A ring and the MMA window's over-read slack
      a_ring + (uint32_t)S * a_stage + rows_tail_slack(S, p.kbps, p.RB, p.NT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KS = p.k_stages;
  const CUtensorMap* tmW = io.tmW;
  const CUtensorMap* tmA = io.tmA;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), (uint32_t)issuers);  // one commit per issuer and stage
    }
    mbar_init(smem_u32(acc_full), (uint32_t)issuers);
    mbar_init(smem_u32(drain), (uint32_t)issuers);
    if (split) mbar_init(smem_u32(ready), 128u);  // the peer's four epilogue warps
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(tmW);
    prefetch_tmap(tmA);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Under the K split the peer's barriers must exist before the first remote
  // arrive: every thread arrives here, and waits for this phase before its
  // first remote access (the epilogue warps) or at the end (the others).
  if (split) cluster_arrive();
  pdl_launch_dependents();  // the dependent grid still waits for our completion before reading

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      // W for the first `prefetch` stages before the dependency wait.  A
      // slot left free lets weights keep streaming while A (needed by the
      // first MMA) is fetched after the wait.
      const int pre = KS < p.prefetch ? KS : p.prefetch;
      // This rank's first K element (rank 1 of a K split may start or run
      // past K: those boxes are zero-filled and add nothing).
      const int kbase = (int)rank * KS * p.kbps * kTcKBlock;
      for (int s = 0; s < pre; ++s) {
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        const uint32_t ws = w_ring + (uint32_t)s * w_stage;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(ws + (uint32_t)j * wblk, tmW, kbase + (s * p.kbps + j) * kTcKBlock, n0, fb, pol_w);
      }
      pdl_wait();
      for (int s = 0; s < pre; ++s) {
        const uint32_t as = a_ring + (uint32_t)s * a_stage;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(as + (uint32_t)j * ablk, tmA, kbase + (s * p.kbps + j) * kTcKBlock, 0,
                      smem_u32(&full[s]), pol_a);
      }
      // Ring position kept by increments: no integer division on the
      // per-stage path of this single issuing thread.
      int issued = pre;
      int slot = pre == S ? 0 : pre;
      uint32_t par = pre == S ? 1u : 0u;  // ring round parity of `slot`
      uint32_t ws = w_ring + (uint32_t)slot * w_stage, as = a_ring + (uint32_t)slot * a_stage;
      int kx = kbase + pre * p.kbps * kTcKBlock;
      const int kstep = p.kbps * kTcKBlock;
      for (int s = pre; s < KS; ++s) {
        if (s >= S && !mbar_wait_or_abort(smem_u32(&empty[slot]), par ^ 1u, abort_flag)) {
          if (!*abort_flag) report_error(p.err, kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        const uint32_t fb = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(ws + (uint32_t)j * wblk, tmW, kx + j * kTcKBlock, n0, fb, pol_w);
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(as + (uint32_t)j * ablk, tmA, kx + j * kTcKBlock, 0, fb, pol_a);
        issued = s + 1;
        kx += kstep;
        ws += w_stage;
        as += a_stage;
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
          ws = w_ring;
          as = a_ring;
        }
      }
      for (int t = issued > S ? issued - S : 0; t < issued; ++t)
        if (!mbar_wait(smem_u32(&full[t % S]), (t / S) & 1)) {
          report_error(p.err, kErrDrain);
          break;
        }
    }
  } else if (warp == 1 || warp == 6) {
    // ----------------------------------------------------------- MMA issuers
    const int iss = rows_two_issuer_mode(kMode) && warp == 6 ? 1 : 0;
    if (lane == 0 && iss < issuers) {
      // Issuer i takes MMA windows i, i + issuers, ... of every stage into
      // accumulator i (G * NT columns each).  This thread's issue rate bounds
      // the kernel at 32-64 tokens, so its loop carries no index arithmetic
      // per MMA: window descriptors advance by a fixed step, and the
      // accumulate flag is a register the first MMA clears (recomputing the
      // first-window test and the offsets per MMA measured ~1.5 us slower
      // per call there).
      const uint32_t dacc = tmem + (uint32_t)(iss * p.groups * p.NT);
      const uint32_t idesc = idesc_bf16_f32(kTcTileRows, p.groups * p.NT);
      // Descriptors differ only in their start-address field (address >> 4):
      // build the ring bases once and add offsets.
      const uint64_t wdesc0 = smem_desc_sw128(w_ring);
      const uint64_t adesc0 = smem_desc_sw128(a_ring);
      const int j0 = iss * p.groups, jstep = issuers * p.groups;
      const uint64_t wfirst = (uint64_t)((uint32_t)j0 * wblk >> 4), afirst = (uint64_t)((uint32_t)j0 * ablk >> 4);
      const uint64_t wwin = (uint64_t)((uint32_t)jstep * wblk >> 4), awin = (uint64_t)((uint32_t)jstep * ablk >> 4);
      bool ok = true;
      int slot = 0;
      uint32_t par = 0;  // ring round parity of `slot`
      uint32_t accum = 0;
      uint64_t wd = wdesc0, ad = adesc0;
      for (int s = 0; s < KS; ++s) {
        if (!mbar_wait_or_abort(smem_u32(&full[slot]), par, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint64_t wj = wd + wfirst, aj = ad + afirst;
        for (int j = j0; j < p.kbps; j += jstep) {
#pragma unroll
          for (int kk = 0; kk < kTcKBlock / 16; ++kk) {
            mma_bf16(dacc, wj + (uint64_t)(kk * 2), aj + (uint64_t)(kk * 2), idesc, accum);  // K step: 32 bytes
            accum = 1u;
          }
          wj += wwin;
          aj += awin;
        }
        mma_commit(smem_u32(&empty[slot]));
        wd += w_stage >> 4;
        ad += a_stage >> 4;
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
          wd = wdesc0;
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
    // ------------------------------------------------------------ epilogue
    if (split) cluster_wait();  // the peer's barriers exist (the CTAs of a cluster start together)
    pdl_wait();  // R may come from the preceding kernel; Y may be read by it
    const int q = warp & 3;       // TMEM lane quarter this warp may access
    // Each instance compiles only its own forms: the 16-token ones always
    // apply to their instance (the planner packs G * RB <= 128 rows).
    if constexpr (kMode == kRowsEpi16) {
      // Decode epilogue (at most 16 tokens, at most two packed groups): the
      // thread on TMEM lane r < RB owns output column n0 + r and holds group
      // 0's partial sums; the thread on lane RB + r holds group 1's and hands
      // them over through shared memory.  Everything but the TMEM load, one
      // exchange and the stores is done before the accumulator is ready.
      const int L = q * 32 + lane;
      const int G = p.groups;
      const bool owner = L < p.RB && n0 + L < p.N;
      const bool fin = !split || ((L < p.RB / 2) == (rank == 0u));  // this rank stores column n0 + L
      const bool helper = G == 2 && L >= p.RB && L < 2 * p.RB;
      const int r = owner ? L : L - p.RB;
      const uint32_t xch = w_ring + (uint32_t)(helper || owner ? r : 0) * 80u;  // drained ring: 16 floats + pad per row
      uint32_t res2[kRowsPrefetchTokens / 2];  // residuals as BF16 pairs (half the registers)
      {
        const unsigned short* rp = reinterpret_cast<const unsigned short*>(io.R) + n0 + L;
#pragma unroll
        for (int m = 0; m < kRowsPrefetchTokens; m += 2) {
          const uint32_t lo = (owner && fin && m < io.M) ? rp[(size_t)m * io.ldr] : 0u;
          const uint32_t hi = (owner && fin && m + 1 < io.M) ? rp[(size_t)(m + 1) * io.ldr] : 0u;
          res2[m / 2] = lo | (hi << 16);
        }
      }
      // Pass 0 warms the code below while the MMAs run; pass 1 is the real
      // one.  The pass number goes through an opaque move so that the
      // compiler keeps one copy of the loop body for both passes.
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        int passv;
        asm volatile("mov.b32 %0, %1;" : "=r"(passv) : "r"(pass));
        const bool real = passv != 0;
        bool ok = true;
        if (real) {
          ok = mbar_wait_or_abort(smem_u32(acc_full), 0, abort_flag);
          if (!ok) {
            if (!*abort_flag) report_error(p.err, kErrWaitMma);
            *abort_flag = 1;
          }
          ok = __all_sync(0xffffffffu, ok);
        }
        tc_fence_after();
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        if (ok && q * 32 < G * p.RB) {  // warp-uniform: this warp holds rows of the MMA window in use
          // Accumulator i at columns [i C, (i + 1) C), C = G * 16; pass 0
          // reads the columns after them, which no MMA writes.
          const uint32_t C = (uint32_t)(G * kRowsPrefetchTokens);
          const uint32_t taddr =
              tmem + ((uint32_t)(q * 32) << 16) + (real ? 0u : (uint32_t)issuers * C);
          const bool two = issuers == 2;
          if (G == 1 || (q + 1) * 32 <= p.RB) {
            tmem_ld16_sum(taddr, C, two, v);  // group-0 columns only
          } else if (q * 32 >= p.RB) {
            tmem_ld16_sum(taddr + 16u, C, two, v);  // group-1 columns only
          } else {
            float v1[16];
            tmem_ld16_sum(taddr, C, two, v);
            tmem_ld16_sum(taddr + 16u, C, two, v1);
            if (L >= p.RB) {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = v1[i];
            }
          }
        }
        const uint32_t x = real ? xch : base + kRowsWarmScratch;
        if (ok && helper) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(x + (uint32_t)i * 4u), "f"(v[i]),
                         "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                         : "memory");
        }
        named_bar_sync(1, 128);
        if (ok && owner && G == 2) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            float a0, a1, a2, a3;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                         : "r"(x + (uint32_t)i * 4u)
                         : "memory");
            v[i] += a0;
            v[i + 1] += a1;
            v[i + 2] += a2;
            v[i + 3] += a3;
          }
        }
        if constexpr (split)
          if (real)
            ok = rows_pair_exchange<16>(v, ok && owner, fin, xch + (uint32_t)p.RB * 80u, ready, rank, abort_flag,
                                      p.err) &&
               ok;
        if (ok && owner && fin) {
          __nv_bfloat16* yp = io.Y + n0 + L;
#pragma unroll
          for (int m = 0; m < kRowsPrefetchTokens; ++m)
            st_global_bf16_if(yp + (size_t)m * io.ldy,
                              __float2bfloat16_rn(v[m] + ((m & 1) ? bf16hi(res2[m / 2]) : bf16lo(res2[m / 2]))),
                              real && m < io.M);
        }
      }
    } else if (kMode == kRowsEpiWide && p.NT == 32 && p.groups <= 2 && p.groups * p.RB <= kTcTileRows) {
      rows_epilogue_wide<32, kWideWarm, kSplit>(p, io, n0, tmem, w_ring, wide_scratch, acc_full, ready, abort_flag, q,
                                          lane);
    } else if (kMode == kRowsEpiWide && p.NT == 48 && p.groups <= 2 && p.groups * p.RB <= kTcTileRows) {
      rows_epilogue_wide<48, kWideWarm, kSplit>(p, io, n0, tmem, w_ring, wide_scratch, acc_full, ready, abort_flag, q,
                                          lane);
    } else if (kMode == kRowsEpi64 && p.NT == 64 && p.groups <= 2 && p.groups * p.RB <= kTcTileRows) {
      rows_epilogue_wide<64, kWideWarm, kSplit>(p, io, n0, tmem, w_ring, wide_scratch, acc_full, ready, abort_flag, q,
                                          lane);
    } else if (kMode == kRowsEpi16G4 && p.NT == kRowsPrefetchTokens && p.groups == 4 && p.RB == 32) {
      // 32-row slabs, four packed groups: warp quarter q holds group q whole.
      // Warps 1-3 hand their partial sums to warp 0's lanes (one output
      // column each) through shared memory; warp 0 adds them in group order.
      // A warm-up pass first, as in the two-group form above.
      const bool owner = q == 0 && n0 + lane < p.N;
      const uint32_t xch = w_ring + (uint32_t)lane * 80u;  // drained ring: [3][32] rows of 16 floats + pad
      uint32_t res2[kRowsPrefetchTokens / 2];  // residuals as BF16 pairs (half the registers)
      {
        const unsigned short* rp = reinterpret_cast<const unsigned short*>(io.R) + n0 + lane;
#pragma unroll
        for (int m = 0; m < kRowsPrefetchTokens; m += 2) {
          const uint32_t lo = (owner && m < io.M) ? rp[(size_t)m * io.ldr] : 0u;
          const uint32_t hi = (owner && m + 1 < io.M) ? rp[(size_t)(m + 1) * io.ldr] : 0u;
          res2[m / 2] = lo | (hi << 16);
        }
      }
      const uint32_t C = (uint32_t)(p.groups * kRowsPrefetchTokens);  // columns of one accumulator
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        int passv;  // opaque to the compiler: one copy of the loop body serves both passes
        asm volatile("mov.b32 %0, %1;" : "=r"(passv) : "r"(pass));
        const bool real = passv != 0;
        bool ok = true;
        if (real) {
          ok = mbar_wait_or_abort(smem_u32(acc_full), 0, abort_flag);
          if (!ok) {
            if (!*abort_flag) report_error(p.err, kErrWaitMma);
            *abort_flag = 1;
          }
          ok = __all_sync(0xffffffffu, ok);
        }
        tc_fence_after();
        const uint32_t x = real ? xch : base + kRowsWarmScratch;
        const uint32_t xs = real ? 32u * 80u : 0u;
        float v[16];
        if (ok) {
          tmem_ld16_sum(tmem + ((uint32_t)(q * 32) << 16) + (real ? 0u : (uint32_t)issuers * C) + (uint32_t)(q * 16),
                        C, issuers == 2, v);
          if (q > 0) {
            const uint32_t dst = x + (uint32_t)(q - 1) * xs;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + (uint32_t)i * 4u), "f"(v[i]),
                           "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                           : "memory");
          }
        }
        named_bar_sync(1, 128);
        if (ok && owner) {
#pragma unroll
          for (int gg = 0; gg < 3; ++gg) {
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              float a0, a1, a2, a3;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                           : "r"(x + (uint32_t)gg * xs + (uint32_t)i * 4u)
                           : "memory");
              v[i] += a0;
              v[i + 1] += a1;
              v[i + 2] += a2;
              v[i + 3] += a3;
            }
          }
          __nv_bfloat16* yp = io.Y + n0 + lane;
#pragma unroll
          for (int m = 0; m < kRowsPrefetchTokens; ++m)
            st_global_bf16_if(yp + (size_t)m * io.ldy,
                              __float2bfloat16_rn(v[m] + ((m & 1) ? bf16hi(res2[m / 2]) : bf16lo(res2[m / 2]))),
                              real && m < io.M);
        }
      }
    } else if constexpr (kMode == kRowsEpi16G4) {
      // The same for three or four packed groups (short slabs, e.g. 24 rows
      // when N = 3584): lane g*RB + r (g = 1 .. G-1) hands group g's partial
      // sums to the owner of row r, who adds them in g order.  Kept apart
      // from the two-group version above, which measured ~0.3 us faster per
      // call than this loop form with G = 2.  A warm-up pass first, as there.
      const int L = q * 32 + lane;
      const int G = p.groups;
      const int g = L / p.RB;  // packed group of this lane (>= G: unused lane)
      const int r = L - g * p.RB;
      const bool owner = g == 0 && n0 + r < p.N;
      const bool helper = g >= 1 && g < G;
      // drained ring: [G-1][RB] rows of 16 floats + 4 pad
      const uint32_t xch0 = w_ring + (uint32_t)r * 80u;
      const uint32_t xstep = (uint32_t)p.RB * 80u;
      uint32_t res2[kRowsPrefetchTokens / 2];  // residuals as BF16 pairs (half the registers)
      {
        const unsigned short* rp = reinterpret_cast<const unsigned short*>(io.R) + n0 + r;
#pragma unroll
        for (int m = 0; m < kRowsPrefetchTokens; m += 2) {
          const uint32_t lo = (owner && m < io.M) ? rp[(size_t)m * io.ldr] : 0u;
          const uint32_t hi = (owner && m + 1 < io.M) ? rp[(size_t)(m + 1) * io.ldr] : 0u;
          res2[m / 2] = lo | (hi << 16);
        }
      }
      const uint32_t C = (uint32_t)(G * kRowsPrefetchTokens);  // columns of one accumulator
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        int passv;  // opaque to the compiler: one copy of the loop body serves both passes
        asm volatile("mov.b32 %0, %1;" : "=r"(passv) : "r"(pass));
        const bool real = passv != 0;
        bool ok = true;
        if (real) {
          ok = mbar_wait_or_abort(smem_u32(acc_full), 0, abort_flag);
          if (!ok) {
            if (!*abort_flag) report_error(p.err, kErrWaitMma);
            *abort_flag = 1;
          }
          ok = __all_sync(0xffffffffu, ok);
        }
        tc_fence_after();
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
        if (ok && q * 32 < G * p.RB) {  // warp-uniform: this warp holds rows of the MMA window in use
          // The warp's lanes hold groups glo .. ghi: load their columns
          // (16 per group) and keep this lane's.
          const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (real ? 0u : (uint32_t)issuers * C);
          const int glo = (q * 32) / p.RB;
          const int ghi = min(G - 1, (q * 32 + 31) / p.RB);
          for (int gg = glo; gg <= ghi; ++gg) {
            float w[16];
            tmem_ld16(taddr + (uint32_t)(gg * 16), w);  // warp-collective
            if (gg == g) {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = w[i];
            }
            if (issuers == 2) {  // the second accumulator, added after the first
              tmem_ld16(taddr + C + (uint32_t)(gg * 16), w);
              if (gg == g) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] += w[i];
              }
            }
          }
        }
        const uint32_t x0 = real ? xch0 : base + kRowsWarmScratch;
        const uint32_t xs = real ? xstep : 0u;
        if (ok && helper) {
          const uint32_t dst = x0 + (uint32_t)(g - 1) * xs;
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + (uint32_t)i * 4u), "f"(v[i]),
                         "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                         : "memory");
        }
        named_bar_sync(1, 128);
        if (ok && owner) {
          for (int gg = 1; gg < G; ++gg) {
            const uint32_t src = x0 + (uint32_t)(gg - 1) * xs;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              float a0, a1, a2, a3;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                           : "r"(src + (uint32_t)i * 4u)
                           : "memory");
              v[i] += a0;
              v[i + 1] += a1;
              v[i + 2] += a2;
              v[i + 3] += a3;
            }
          }
          __nv_bfloat16* yp = io.Y + n0 + r;
#pragma unroll
          for (int m = 0; m < kRowsPrefetchTokens; ++m)
            st_global_bf16_if(yp + (size_t)m * io.ldy,
                              __float2bfloat16_rn(v[m] + ((m & 1) ? bf16hi(res2[m / 2]) : bf16lo(res2[m / 2]))),
                              real && m < io.M);
        }
      }
    } else {
      const int etid = threadIdx.x - 64;
      const int L = q * 32 + lane;  // TMEM lane = row of the MMA window
      const int g = L / p.RB, r = L % p.RB;
      const int G = p.groups;
      const int chunks = p.NT / 16;  // 16-column groups per token tile
      const int ldp = p.NT + 4;      // staging row stride (floats)
      float* part = reinterpret_cast<float*>(sb + 1024);  // reuses the drained ring
      // Residuals for the combine step (one row per thread when NT == 16).
      float rpre[kRowsPrefetchTokens];
      const bool pre = (p.NT == kRowsPrefetchTokens) && etid < p.RB && n0 + etid < p.N;
#pragma unroll
      for (int i = 0; i < kRowsPrefetchTokens; ++i)
        rpre[i] = (pre && i < io.M) ? __bfloat162float(io.R[(size_t)i * io.ldr + n0 + etid]) : 0.f;
      bool ok = mbar_wait_or_abort(smem_u32(acc_full), 0, abort_flag);
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      // Step 1: each lane copies its diagonal block row (group g, row r) to shared memory.
      if (ok) {
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        for (int c = 0; c < G * chunks; ++c) {
          float v[16];
          tmem_ld16(taddr + (uint32_t)(c * 16), v);  // warp-collective: every lane loads
          if (g < G && c / chunks == g) {
            float* dst = part + ((size_t)g * p.RB + r) * ldp + (c % chunks) * 16;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          }
        }
      }
      named_bar_sync(1, 128);
      // Step 2: sum the groups (g order), add the residual, round once, store.
      if (ok) {
        for (int item = etid; item < p.RB * chunks; item += 128) {
          const int rr = item % p.RB, c16 = item / p.RB;
          const int n = n0 + rr;
          if (n >= p.N) continue;
          float acc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] = 0.f;
          for (int gg = 0; gg < G; ++gg) {
            const float* src = part + ((size_t)gg * p.RB + rr) * ldp + c16 * 16;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 w = *reinterpret_cast<const float4*>(src + i);
              acc[i] += w.x;
              acc[i + 1] += w.y;
              acc[i + 2] += w.z;
              acc[i + 3] += w.w;
            }
          }
          const int m0 = c16 * 16;
          if (pre) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (m0 + i < io.M) io.Y[(size_t)(m0 + i) * io.ldy + n] = __float2bfloat16_rn(acc[i] + rpre[i]);
          } else {
            float rr16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              rr16[i] = (m0 + i < io.M) ? __bfloat162float(io.R[(size_t)(m0 + i) * io.ldr + n]) : 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (m0 + i < io.M) io.Y[(size_t)(m0 + i) * io.ldy + n] = __float2bfloat16_rn(acc[i] + rr16[i]);
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
  if (split) {
    // The producer and MMA warps close the start-up phase; then no CTA
    // leaves while its peer may still read its shared memory.
    if (warp == 0 || warp == 1 || warp == 6) cluster_wait();
    cluster_sync_all();
  }
}

// Two CTAs per SM where their shared memory allows (the register budget is
// sized for it; the default configuration of untabulated shapes relies on
// it), except for the 64-token instance.
template <int kMode, bool kSplit>
__global__ void __launch_bounds__(rows_threads(kMode), kMode == kRowsEpi64 ? 1 : 2)
    rows_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                       const RowsParams p) {
  const RowsIO io{&tmW, &tmA, p.R, p.Y, p.ldr, p.ldy, p.M};
  rows_run<kMode, true, kSplit>(p, io, (int)(blockIdx.x / (kSplit ? 2u : 1u)) * p.RB);  // a K-split pair shares its slab
}

// The instance for an epilogue family and K split (the 16-token form with
// three or four groups has no K-split instance).
inline const void* rows_kernel_fn(int mode, bool split) {
  if (split)
    return mode == kRowsEpi16   ? reinterpret_cast<const void*>(rows_skinny_kernel<kRowsEpi16, true>)
           : mode == kRowsEpi64 ? reinterpret_cast<const void*>(rows_skinny_kernel<kRowsEpi64, true>)
                                : reinterpret_cast<const void*>(rows_skinny_kernel<kRowsEpiWide, true>);
  return mode == kRowsEpi16     ? reinterpret_cast<const void*>(rows_skinny_kernel<kRowsEpi16, false>)
         : mode == kRowsEpi16G4 ? reinterpret_cast<const void*>(rows_skinny_kernel<kRowsEpi16G4, false>)
         : mode == kRowsEpi64   ? reinterpret_cast<const void*>(rows_skinny_kernel<kRowsEpi64, false>)
                                : reinterpret_cast<const void*>(rows_skinny_kernel<kRowsEpiWide, false>);
}

// Grouped launch: several independent problems with the same N and K and
// their own W, A, R, Y and token count (the experts of a mixture-of-experts
// layer).  CTA b works on slab b / count of problem b % count, so the CTAs
// that run at the same time stream different problems' weights.
constexpr int kRowsMaxGroups = 32;

struct RowsGroup {  // the tensor maps keep their own (64-byte or larger) alignment
  CUtensorMap tmW;
  CUtensorMap tmA;
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  long long ldr, ldy;
  int M;
};

struct RowsGroupList {
  RowsGroup g[kRowsMaxGroups];
  int count;
};

// kMode: the 16-token families for 16-token tiles, else kRowsEpiWide (whose
// 32/48-token epilogue here runs without its warm-up pass, which would cost
// this kernel register spills).  kSplit: the 2-CTA K split, the two CTAs of a
// cluster on the same slab of the same problem (16-48-token tiles).
template <int kMode, bool kSplit>
__global__ void __launch_bounds__(rows_threads(kMode), 2)
    rows_grouped_kernel(const __grid_constant__ RowsGroupList list, const RowsParams p) {
  const int unit = (int)blockIdx.x / (kSplit ? 2 : 1);
  const int e = unit % list.count;
  const int slab = unit / list.count;
  const RowsGroup& g = list.g[e];
  const RowsIO io{&g.tmW, &g.tmA, g.R, g.Y, g.ldr, g.ldy, g.M};
  rows_run<kMode, false, kSplit>(p, io, slab * p.RB);
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

inline int rows_plan(const sgr_config& c, int sms, int M, int N, int K, RowsParams* p, int* grid, size_t* smem);

// Default: 4 K blocks per stage and the deepest ring (up to 4 stages) that
// keeps the CTA at or under ~110 KB of shared memory, so that the next call's
// CTA can be resident on the same SM; smaller stages if even 2 do not fit.
// Slabs of at most 32 rows over a long K (K >= 4096) take the 2-CTA K split
// with the same ring: measured on GB300 at 1-64 tokens, N x K = 1024 x 4096,
// 2048 x 8192, 2560 x 10240, 4096 x 14336 ran in 0.54-0.76 of the unsplit
// time; 48-row slabs (7168 x 2048) ran slower split.
inline void rows_default_config(int sms, int M, int N, int K, sgr_config* c) {
  c->path = SGR_PATH_TC_ROWS;
  c->ctas_per_sm = 1;
  c->token_tile = (M + 15) / 16 * 16;
  c->rows_per_stage = 0;
  c->k_split = 0;
  const int rb = rows_per_cta(sms, N);
  const size_t budget = 110u * 1024u;
  c->k_blocks_per_stage = 1;
  c->stages = 2;
  bool found = false;
  for (int kb = 4; kb >= 1 && !found; kb /= 2)
    for (int st = 4; st >= 2 && !found; --st)
      if (rows_smem_bytes(st, kb, rb, c->token_tile) <= budget) {
        c->k_blocks_per_stage = kb;
        c->stages = st;
        found = true;
      }
  if (rb <= 32 && K >= 4096 && c->token_tile <= 64) {
    sgr_config s = *c;
    s.k_split = 2;
    RowsParams p;
    int grid = 0;
    size_t smem = 0;
    if (rows_plan(s, sms, M, N, K, &p, &grid, &smem) == SGR_OK) c->k_split = 2;
  }
}

inline int rows_plan(const sgr_config& c, int sms, int M, int N, int K, RowsParams* p, int* grid,
                     size_t* smem) {
  if (!rows_supported(sms, M, N, K)) return SGR_ERR_UNSUPPORTED;
  const int nt = c.token_tile;
  if (nt < 16 || nt > kRowsMaxTokens || nt % 16 != 0 || nt < M) return SGR_ERR_UNSUPPORTED;
  if (c.k_blocks_per_stage < 1 || c.k_blocks_per_stage > 8) return SGR_ERR_UNSUPPORTED;
  if (c.ctas_per_sm != 1) return SGR_ERR_UNSUPPORTED;
  if (c.stages < 2 || c.stages > 32) return SGR_ERR_UNSUPPORTED;
  if (c.k_split < 0 || c.k_split > 2) return SGR_ERR_UNSUPPORTED;
  const int ks = c.k_split == 2 ? 2 : 1;
  // W rows per CTA: N / SMs rounded up to 8 (N / (SMs / 2) under the K
  // split, whose two CTAs share a slab) unless the configuration names a
  // slab height (rows_per_stage; e.g. 32 rows: 224 CTAs for N = 7168, two per
  // SM, four K blocks per MMA).
  const int rb = c.rows_per_stage > 0 ? c.rows_per_stage : rows_per_cta(sms / ks > 0 ? sms / ks : 1, N);
  if (rb % 8 != 0 || rb > kTcTileRows) return SGR_ERR_UNSUPPORTED;
  const size_t sm = rows_smem_bytes(c.stages, c.k_blocks_per_stage, rb, nt);
  if (sm > 232448) return SGR_ERR_UNSUPPORTED;
  const int kstage_elems = kTcKBlock * c.k_blocks_per_stage;
  p->M = M;
  p->N = N;
  p->K = K;
  p->RB = rb;
  p->NT = nt;
  p->ksplit = ks;
  p->k_stages = (K + ks * kstage_elems - 1) / (ks * kstage_elems);  // per rank
  p->kbps = c.k_blocks_per_stage;
  p->stages = c.stages;
  p->prefetch = c.prefetch_stages > 0 ? c.prefetch_stages : (c.stages > 2 ? c.stages - 1 : c.stages);
  if (p->prefetch > c.stages) return SGR_ERR_UNSUPPORTED;
  // Diagonal packing: as many consecutive K blocks per MMA as fit in the
  // 128-row window and the 256-column N limit, dividing the stage's blocks,
  // with room to stage the epilogue's partial sums in the drained ring.
  // (At most two under the K split, whose epilogues take at most two.)
  p->groups = 1;
  for (int gcount = ks == 2 ? 2 : 4; gcount >= 2; gcount /= 2)
    if (gcount * rb <= kTcTileRows && gcount * nt <= 256 && c.k_blocks_per_stage % gcount == 0) {
      p->groups = gcount;
      break;
    }
  while (p->groups > 1 &&
         rows_stage_floats(p->groups, rb, nt) * 4 > (size_t)c.stages * rows_stage_bytes(c.k_blocks_per_stage, rb, nt))
    p->groups /= 2;
  if (rows_stage_floats(p->groups, rb, nt) * 4 > (size_t)c.stages * rows_stage_bytes(c.k_blocks_per_stage, rb, nt))
    return SGR_ERR_UNSUPPORTED;
  // Two MMA issuers where a 16-token epilogue (which adds the two
  // accumulators) serves the tile and every stage has at least two windows;
  // those epilogues also reserve as many columns again for their warm-up pass.
  const bool decode_epi = nt == kRowsPrefetchTokens && p->groups * rb <= kTcTileRows;
  p->issuers = decode_epi && c.k_blocks_per_stage >= 2 * p->groups ? 2 : 1;
  const int acc_cols = p->issuers * p->groups * nt;
  // The 17-64-token register epilogues (at most two groups) warm up too.
  const bool wide_epi = (nt == 32 || nt == 48 || nt == 64) && p->groups <= 2 && p->groups * rb <= kTcTileRows;
  p->tmem_cols = detail::pow2_at_least(decode_epi || wide_epi ? 2 * acc_cols : acc_cols);
  // The K split completes its partial sums in the 16-64-token register
  // epilogues (at most two groups), whose hand-over buffers then take two
  // rows per W row in the drained ring.
  if (ks == 2 && (!(decode_epi || wide_epi) || p->groups > 2 ||
                  (size_t)2 * rb * rows_xch_stride(nt) > (size_t)c.stages * rows_stage_bytes(c.k_blocks_per_stage, rb, nt)))
    return SGR_ERR_UNSUPPORTED;
  *grid = ks * ((N + rb - 1) / rb);
  *smem = sm;
  return SGR_OK;
}

inline cudaError_t rows_init_device() {
  cudaError_t e = cudaSuccess;
  for (int split = 0; split < 2; ++split)
    for (int mode : {kRowsEpi16, kRowsEpi16G4, kRowsEpiWide, kRowsEpi64})
      if (e == cudaSuccess) e = set_kernel_smem_attrs(rows_kernel_fn(mode, split != 0));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(rows_grouped_kernel<kRowsEpi16, false>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(rows_grouped_kernel<kRowsEpi16G4, false>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(rows_grouped_kernel<kRowsEpiWide, false>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(rows_grouped_kernel<kRowsEpi16, true>));
  if (e == cudaSuccess) e = set_kernel_smem_attrs(reinterpret_cast<const void*>(rows_grouped_kernel<kRowsEpiWide, true>));
  return e;
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
  const int mode = rows_epi_mode(p.NT, p.groups);
  lc.blockDim = dim3(rows_threads(mode), 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  if (p.ksplit == 2) {  // the two CTAs of a slab form a cluster
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = 2;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  lc.attrs = attr;
  lc.numAttrs = n_attr;
  auto fn = p.ksplit == 2 ? (mode == kRowsEpi16   ? rows_skinny_kernel<kRowsEpi16, true>
                             : mode == kRowsEpi64 ? rows_skinny_kernel<kRowsEpi64, true>
                                                  : rows_skinny_kernel<kRowsEpiWide, true>)
                          : (mode == kRowsEpi16     ? rows_skinny_kernel<kRowsEpi16, false>
                             : mode == kRowsEpi16G4 ? rows_skinny_kernel<kRowsEpi16G4, false>
                             : mode == kRowsEpi64   ? rows_skinny_kernel<kRowsEpi64, false>
                                                    : rows_skinny_kernel<kRowsEpiWide, false>);
  if (cudaLaunchKernelEx(&lc, fn, tmW, tmA, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

// Grouped launch of up to kRowsMaxGroups problems (all with M >= 1, M <= the
// plan's token tile) sharing N and K; the configuration is planned for the
// largest M.  One kernel launch; CTA count = slabs x problems.
struct RowsGroupArgs {
  const void* A;
  long long lda;
  const void* W;
  const void* R;
  long long ldr;
  void* Y;
  long long ldy;
  int M;
};

inline int rows_grouped_launch(const sgr_config& c, int sms, unsigned* err, const RowsGroupArgs* gs, int count,
                               int N, int K, bool pdl, cudaStream_t stream) {
  if (count < 1 || count > kRowsMaxGroups) return SGR_ERR_UNSUPPORTED;
  int m_max = 0;
  for (int i = 0; i < count; ++i) m_max = gs[i].M > m_max ? gs[i].M : m_max;
  RowsParams p;
  int grid = 0;
  size_t smem = 0;
  int rc = rows_plan(c, sms, m_max, N, K, &p, &grid, &smem);
  if (rc != SGR_OK) return rc;
  // Under the K split only the 16-48-token epilogues (the 64-token tile runs
  // the general epilogue here, which does not complete split sums).
  if (p.ksplit == 2 && p.NT > 48) return SGR_ERR_UNSUPPORTED;
  p.err = err;
  RowsGroupList list;
  std::memset(&list, 0, sizeof list);
  list.count = count;
  for (int i = 0; i < count; ++i) {
    RowsGroup& g = list.g[i];
    if (!detail::make_tmap(&g.tmW, gs[i].W, N, K, K, p.RB, kTcKBlock)) return SGR_ERR_LAUNCH;
    if (!detail::make_tmap(&g.tmA, gs[i].A, gs[i].M, K, gs[i].lda, p.NT, kTcKBlock)) return SGR_ERR_LAUNCH;
    g.R = static_cast<const __nv_bfloat16*>(gs[i].R);
    g.Y = static_cast<__nv_bfloat16*>(gs[i].Y);
    g.ldr = gs[i].ldr;
    g.ldy = gs[i].ldy;
    g.M = gs[i].M;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(grid * count), 1, 1);
  const int mode = p.NT == 16 ? rows_epi_mode(p.NT, p.groups) : kRowsEpiWide;  // 64-token tiles: the general epilogue
  lc.blockDim = dim3(rows_threads(mode), 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  if (p.ksplit == 2) {  // the two CTAs of a slab form a cluster
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = 2;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  lc.attrs = attr;
  lc.numAttrs = n_attr;
  auto fn = p.ksplit == 2 ? (mode == kRowsEpi16 ? rows_grouped_kernel<kRowsEpi16, true>
                                                : rows_grouped_kernel<kRowsEpiWide, true>)
                          : (mode == kRowsEpi16     ? rows_grouped_kernel<kRowsEpi16, false>
                             : mode == kRowsEpi16G4 ? rows_grouped_kernel<kRowsEpi16G4, false>
                                                    : rows_grouped_kernel<kRowsEpiWide, false>);
  if (cudaLaunchKernelEx(&lc, fn, list, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

}  // namespace sgr
