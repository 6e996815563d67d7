// sgr_pair.cuh -- tensor-core tile GEMM on CTA pairs (tcgen05 cta_group::2)
// for compute-bound token counts.
//
// Same operation as the other kernels: Y[m,n] = bf16_rn( sum_k A[m,k] W[n,k]
// + R[m,n] ) with FP32 accumulation and one rounding (vLLM
// "benchmark_k3_cutedsl_residual.py", module docstring and its correctness()
// reference).  Past the ridge point of tensor peak over HBM bandwidth (the
// roofline reasoning of the bitsandbytes "QLORA-2" comparison page,
// agents/kbit_gemm_context.md) the limit of a one-CTA 128 x NT tile is the
// operand feed from L2 into shared memory: each 64-wide K block brings
// (128 + NT) x 128 bytes for 128 x NT x 64 multiply-adds.  Here two CTAs on
// neighbouring SMs (a 2-CTA cluster) compute one 256-token x NT tile with
// M = 256 MMAs issued by one thread of the even CTA: each CTA loads its own
// 128 token rows of A and HALF of the W tile (NT/2 rows) into its own shared
// memory, and the tensor cores of the pair read both halves of W, so a CTA
// brings (128 + NT/2) x 128 bytes per K block for the same 128 x NT x 64
// multiply-adds.  No data is copied between the CTAs by software and no copy
// is sent to more than one CTA: each TMA load writes the shared memory of the
// CTA that issues it (its completion is counted on the even CTA's barrier,
// which the MMA thread waits on).
//
// Roles (192 threads per CTA).  Warp 0 lane 0: TMA producer of its CTA (the
// even CTA's also arms the stage's barrier with both CTAs' bytes).  Warp 1
// owns the pair's tensor memory (allocated by both CTAs together); in the
// even CTA its lane 0 issues the MMAs and commits stage releases and
// accumulator hand-offs to the barriers of both CTAs.  Warps 2-5: epilogue
// of each CTA, one output row (token) per thread from its CTA's half of the
// accumulator (TMEM lanes = the CTA's 128 tokens, columns = the NT W rows):
// residual row loaded when the tile starts, + accumulator, one rounding,
// 16-byte stores; then both CTAs' epilogues release the accumulator on the
// even CTA's barrier.  Two accumulators let the epilogue of one tile overlap
// the MMAs of the next.
//
// Persistent grid of 2 x min(tiles, pairs) CTAs, where pairs is the number of
// 2-CTA clusters the device runs at once (queried; SMs / 2 when every SM
// pairs up); pair u takes tiles u,
// u + P, ... with tile t = (t mod m_tiles) token tile, (t div m_tiles) W
// column tile, so concurrently running pairs share W tiles and A in L2.  W
// (input-only by the launch contract) is requested for the first ring stages
// before griddepcontrol.wait; A, R and Y are touched only after it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sgr_ptx.cuh"
#include "sgr_tc.cuh"
#include "sgr_gemm.cuh"
#include "skinny_gemm_residual.h"

namespace sgr {

constexpr int kPairThreads = 192;
constexpr int kPairM = 256;        // tokens per pair tile (MMA M)
constexpr int kPairHalf = 128;     // tokens per CTA (TMEM lanes)
constexpr int kPairMaxStages = 16;

struct PairParams {
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  long long ldr, ldy;
  unsigned* err;
  int M, N, K;
  int NT;        // W rows per pair tile = MMA N; each CTA loads NT / 2 of them
  int m_tiles;   // ceil(M / 256)
  int n_tiles;   // ceil(N / NT)
  int k_blocks;  // ceil(K / 64)
  int stages;    // ring depth
  int kbps;      // K blocks per ring stage (1, 2 or 4)
  int prefetch;  // W stages requested before griddepcontrol.wait (1..stages)
  int tmem_cols;
};

// One ring stage of one CTA: kbps K blocks of its A rows (128 x 64 boxes)
// then of its half of the W tile (NT/2 x 64 boxes).
__host__ __device__ inline uint32_t pair_stage_bytes(int nt, int kbps) {
  return (uint32_t)kbps * ((uint32_t)kPairHalf * 128u + (uint32_t)(nt / 2) * 128u);
}

__host__ __device__ inline size_t pair_smem_bytes(int stages, int nt, int kbps) {
  return 1024 /* alignment slack */ + 1024 /* barriers */ + (size_t)stages * pair_stage_bytes(nt, kbps);
}

// ------------------------------------------------------- cta_group::2 PTX
// Tensor memory of the CTA pair, allocated (and released) by one warp of
// each CTA together; the address is written to each CTA's shared memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A . B^T over the pair: A rows 0..127 from this CTA's shared memory
// and 128..255 from the other CTA's (same offset), B rows 0..N/2-1 from this
// CTA and N/2..N-1 from the other; D rows 0..127 in this CTA's tensor memory,
// 128..255 in the other's (same address).
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at cluster address `bar` (this CTA's or the other's)
// once the pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 2-D TMA load into this CTA's shared memory whose completion is counted on
// the barrier at cluster address `bar` (the even CTA's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// The residual row segment R[m, n0 .. n0 + NT) of one thread (zeros outside
// the matrix; N is a multiple of 8).
template <int NT>
__device__ __forceinline__ void pair_residual_row(const PairParams& p, int m, int n0, uint4 (&rv)[NT / 8]) {
  const bool row_ok = m < p.M;
  const __nv_bfloat16* src = p.R + (size_t)(row_ok ? m : 0) * p.ldr + n0;
#pragma unroll
  for (int j = 0; j < NT / 8; ++j)
    rv[j] = (row_ok && n0 + 8 * j < p.N) ? *reinterpret_cast<const uint4*>(src + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
}

template <int NT>
__global__ void __launch_bounds__(kPairThreads, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const PairParams p) {
  constexpr int HN = NT / 2;  // W rows loaded by each CTA
  static_assert(NT % 32 == 0 && HN % 8 == 0, "whole 32-column epilogue pieces and 8-row swizzle atoms");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(sb);  // [S]  both CTAs' copies landed (even CTA's used)
  uint64_t* empty = full + S;                         // [S]  the pair's MMAs are done with the slot
  uint64_t* acc_full = empty + S;                     // [2]  accumulator ready
  uint64_t* acc_empty = acc_full + 2;                 // [2]  both CTAs' epilogues done (even CTA's used)
  uint64_t* drain = acc_empty + 2;                    // [1]  MMA completion at exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int KP = p.kbps;
  const uint32_t a_box = (uint32_t)kPairHalf * 128u;  // one A box: 128 rows x 64 K
  const uint32_t w_box = (uint32_t)HN * 128u;         // one W box: NT/2 rows x 64 K
  const uint32_t a_part = (uint32_t)KP * a_box;       // A boxes at the start of a stage, W boxes after
  const uint32_t stage_bytes = pair_stage_bytes(NT, KP);
  const uint32_t ring = base + 1024;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int P = (int)gridDim.x / 2;      // pairs
  const int unit = (int)blockIdx.x / 2;  // this CTA's pair
  const int tiles = p.m_tiles * p.n_tiles;
  const int my_tiles = (tiles - unit + P - 1) / P;  // >= 1: pairs <= tiles
  const int KS = (p.k_blocks + KP - 1) / KP;        // ring stages per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 8);  // 4 epilogue warps in each CTA
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish_pair();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // both CTAs' barriers exist before any copy or MMA names them
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();  // the dependent grid still waits for our completion before reading

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();  // re-read by the pairs of the other token tiles
      const uint64_t pol_a = policy_evict_last();    // re-read for every W column tile
      const int total = my_tiles * KS;
      struct Cursor {
        int kx, t, m0, n0, kb;
      };
      // This CTA's rows of the tile: tokens m0 .. m0 + 127, W rows n0 .. n0 + HN - 1.
      auto coords = [&](Cursor& c) {
        c.m0 = (c.t % p.m_tiles) * kPairM + (int)rank * kPairHalf;
        c.n0 = (c.t / p.m_tiles) * NT + (int)rank * HN;
      };
      auto start = [&](Cursor& c) {
        c.kx = 0;
        c.kb = 0;
        c.t = unit;
        coords(c);
      };
      auto advance = [&](Cursor& c) {
        c.kx += KP * kTcKBlock;
        if (++c.kb == KS) {
          c.kb = 0;
          c.kx = 0;
          c.t += P;
          coords(c);
        }
      };
      auto arm = [&](int slot) {  // the even CTA arms the stage with both CTAs' bytes
        if (even) mbar_arrive_expect_tx(smem_u32(&full[slot]), 2u * stage_bytes);
      };
      const int pre = total < p.prefetch ? total : p.prefetch;  // <= S
      Cursor c;
      start(c);
      for (int it = 0; it < pre; ++it, advance(c)) {
        arm(it);
        const uint32_t fb = map_to_rank(smem_u32(&full[it]), 0);
        const uint32_t st = ring + (uint32_t)it * stage_bytes;
        for (int j = 0; j < KP; ++j)
          tma_load_2d_pair(st + a_part + (uint32_t)j * w_box, &tmW, c.kx + j * kTcKBlock, c.n0, fb, pol_w);
      }
      pdl_wait();
      {
        Cursor ca;
        start(ca);
        for (int it = 0; it < pre; ++it, advance(ca)) {
          const uint32_t fb = map_to_rank(smem_u32(&full[it]), 0);
          const uint32_t st = ring + (uint32_t)it * stage_bytes;
          for (int j = 0; j < KP; ++j)
            tma_load_2d_pair(st + (uint32_t)j * a_box, &tmA, ca.kx + j * kTcKBlock, ca.m0, fb, pol_a);
        }
      }
      int slot = pre == S ? 0 : pre;
      uint32_t par = pre == S ? 1u : 0u;  // ring round parity of `slot`
      uint32_t soff = (uint32_t)slot * stage_bytes;
      int issued = pre;
      for (int it = pre; it < total; ++it, advance(c)) {
        if (it >= S && !mbar_wait_or_abort(smem_u32(&empty[slot]), par ^ 1u, abort_flag)) {
          if (!*abort_flag) report_error(p.err, kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        arm(slot);
        const uint32_t fb = map_to_rank(smem_u32(&full[slot]), 0);
        const uint32_t st = ring + soff;
        for (int j = 0; j < KP; ++j) {
          tma_load_2d_pair(st + (uint32_t)j * a_box, &tmA, c.kx + j * kTcKBlock, c.m0, fb, pol_a);
          tma_load_2d_pair(st + a_part + (uint32_t)j * w_box, &tmW, c.kx + j * kTcKBlock, c.n0, fb, pol_w);
        }
        issued = it + 1;
        soff += stage_bytes;
        if (++slot == S) {
          slot = 0;
          soff = 0;
          par ^= 1u;
        }
      }
      // Drain: the MMAs release a slot only after reading both CTAs' copies,
      // so once the last stages are released every copy of this CTA has landed.
      for (int t = issued > S ? issued - S : 0; t < issued; ++t)
        if (!mbar_wait(smem_u32(&empty[t % S]), (t / S) & 1)) {
          report_error(p.err, kErrDrain);
          break;
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && even) {
      const uint32_t idesc = idesc_bf16_f32(kPairM, NT);
      const uint64_t adesc0 = smem_desc_sw128(ring);
      const uint64_t wdesc0 = smem_desc_sw128(ring + a_part);
      const uint32_t peer = 1u;
      bool ok = true;
      int slot = 0;
      uint32_t par = 0;
      uint64_t doff = 0;  // slot * stage_bytes >> 4 (descriptor start-address units)
      const uint64_t dstep = stage_bytes >> 4;
      const uint64_t a_win = (uint64_t)(a_box >> 4), w_win = (uint64_t)(w_box >> 4);  // one K block
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait_cluster(smem_u32(&acc_empty[buf]), ((i >> 1) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * NT);
        uint32_t accum = 0;
        for (int ks = 0; ks < KS; ++ks) {
          if (!mbar_wait_or_abort(smem_u32(&full[slot]), par, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // No index arithmetic per MMA: descriptors advance by fixed steps
          // and the accumulate flag is a register the tile's first MMA clears.
          uint64_t aj = adesc0 + doff, wj = wdesc0 + doff;
          for (int j = 0; j < KP; ++j) {
#pragma unroll
            for (int kk = 0; kk < kTcKBlock / 16; ++kk) {
              mma_bf16_pair(d, aj + (uint64_t)(kk * 2), wj + (uint64_t)(kk * 2), idesc, accum);  // K step: 32 bytes
              accum = 1u;
            }
            aj += a_win;
            wj += w_win;
          }
          mma_commit_pair(smem_u32(&empty[slot]));
          mma_commit_pair(map_to_rank(smem_u32(&empty[slot]), peer));
          doff += dstep;
          if (++slot == S) {
            slot = 0;
            doff = 0;
            par ^= 1u;
          }
        }
        if (ok) {
          mma_commit_pair(smem_u32(&acc_full[buf]));
          mma_commit_pair(map_to_rank(smem_u32(&acc_full[buf]), peer));
        }
      }
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      mma_commit_pair(smem_u32(drain));
      if (!mbar_wait(smem_u32(drain), 0)) report_error(p.err, kErrDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // R may come from the preceding kernel; Y may be read by it
    const int q = warp & 3;  // TMEM lane quarter = this CTA's tile rows [32 q, 32 q + 32)
    const uint32_t acc_empty0 = map_to_rank(smem_u32(&acc_empty[0]), 0);
    int t = unit;
    int m = (t % p.m_tiles) * kPairM + (int)rank * kPairHalf + q * 32 + lane;  // this thread's output row
    int n0 = (t / p.m_tiles) * NT;
    uint4 rv[NT / 8];
    pair_residual_row<NT>(p, m, n0, rv);
    for (int i = 0; i < my_tiles; ++i) {
      const int buf = i & 1;
      // Sleeping poll: warps 4 and 5 share sub-partitions with the copy and
      // MMA threads, whose issue slots a tight spin would take.
      bool ok = mbar_wait_sleepy_or_abort(smem_u32(&acc_full[buf]), (i >> 1) & 1, abort_flag);
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * NT);
      __nv_bfloat16* dst = p.Y + (size_t)(m < p.M ? m : 0) * p.ldy + n0;
#pragma unroll
      for (int cc = 0; cc < NT / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(taddr + (uint32_t)(cc * 32), v);  // warp-collective: every lane loads
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 r = rv[cc * 4 + j];
          const int e = j * 8;
          const uint4 y = make_uint4(add_round_bf16x2(v[e + 0], v[e + 1], r.x), add_round_bf16x2(v[e + 2], v[e + 3], r.y),
                                     add_round_bf16x2(v[e + 4], v[e + 5], r.z), add_round_bf16x2(v[e + 6], v[e + 7], r.w));
          if (m < p.M && n0 + cc * 32 + e < p.N) *reinterpret_cast<uint4*>(dst + cc * 32 + e) = y;
        }
      }
      // Accumulator buffer free (for this CTA's half) for the MMAs of tile i + 2.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc_empty0 + (uint32_t)(buf * 8));
      if (i + 1 < my_tiles) {  // next tile's residuals arrive during its main loop
        t += P;
        m = (t % p.m_tiles) * kPairM + (int)rank * kPairHalf + q * 32 + lane;
        n0 = (t / p.m_tiles) * NT;
        pair_residual_row<NT>(p, m, n0, rv);
      }
    }
  }

  __syncwarp();  // lane-0 roles rejoin their warp before the barriers
  tc_fence_before();
  __syncthreads();
  // The even CTA's MMAs (which read this CTA's shared memory and write its
  // tensor memory) are complete once its MMA thread has drained: no CTA
  // releases the pair's tensor memory or leaves before that.
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, (uint32_t)p.tmem_cols);
  }
  cluster_sync_all();
}

// ------------------------------------------------------------------ host side
inline bool pair_supported(int M, int N, int K) {
  return M >= 1 && N >= 16 && K >= 8 && N % 8 == 0 && K % 8 == 0;
}

// Tile width: the NT in {192, 256, 128, 96, 64} with the least work per SM
// (waves of tiles over the pairs x NT), the first listed winning ties.
inline int pair_default_nt(int pairs_avail, int M, int N) {
  const long long mt = (M + kPairM - 1) / kPairM;
  const long long pairs = pairs_avail > 0 ? pairs_avail : 1;
  const int cand[5] = {192, 256, 128, 96, 64};
  int best = cand[0];
  long long best_cost = -1;
  for (int nt : cand) {
    const long long tiles = mt * ((N + nt - 1) / nt);
    const long long cost = ((tiles + pairs - 1) / pairs) * nt;
    if (best_cost < 0 || cost < best_cost) {
      best = nt;
      best_cost = cost;
    }
  }
  return best;
}

inline int pair_default_stages(int nt, int kbps = 1) {
  long long st = (232448 - 2048) / pair_stage_bytes(nt, kbps);
  return (int)(st > kPairMaxStages ? kPairMaxStages : (st < 2 ? 2 : st));
}

inline void pair_default_config(int pairs, int M, int N, int K, sgr_config* c) {
  (void)K;
  c->path = SGR_PATH_PAIR;
  c->ctas_per_sm = 1;
  c->tile_n = pair_default_nt(pairs, M, N);
  // Two K blocks per stage: half the stage-release commits of one-block
  // stages, whose cost in the issuing thread measured larger than the loss
  // of ring depth.
  c->k_blocks_per_stage = 2;
  c->stages = pair_default_stages(c->tile_n, 2);
  c->prefetch_stages = 0;  // all stages
  c->token_tile = kPairM;
  c->rows_per_stage = 0;
  c->k_split = 0;
}

inline const void* pair_kernel_for(int nt) {
  switch (nt) {
    case 64: return reinterpret_cast<const void*>(pair_gemm_kernel<64>);
    case 96: return reinterpret_cast<const void*>(pair_gemm_kernel<96>);
    case 128: return reinterpret_cast<const void*>(pair_gemm_kernel<128>);
    case 192: return reinterpret_cast<const void*>(pair_gemm_kernel<192>);
    case 256: return reinterpret_cast<const void*>(pair_gemm_kernel<256>);
    default: return nullptr;
  }
}

// 2-CTA clusters of one-CTA-per-SM kernels that the device can run at once
// (fewer than SMs / 2 when the SMs of a processing cluster do not pair up),
// per device; 0 until queried.
inline int* pair_max_clusters_table() {
  static int table[64] = {0};
  return table;
}

// Kernel attributes, and the number of pairs a persistent grid may use on
// the current device (`dev`).
inline cudaError_t pair_init_device(int dev) {
  for (int nt : {64, 96, 128, 192, 256}) {
    cudaError_t e = set_kernel_smem_attrs(pair_kernel_for(nt));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2, 1, 1);
  lc.blockDim = dim3(kPairThreads, 1, 1);
  lc.dynamicSmemBytes = 232448 - 1024;  // any configuration above half an SM's shared memory: one CTA per SM
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(pair_gemm_kernel<192>), &lc);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) pair_max_clusters_table()[dev] = n;
  return cudaSuccess;
}

// Pairs a persistent grid may use: the queried cluster count of the device,
// else SMs / 2 (host-only planning without a device).
inline int pair_grid_pairs(int sms, int dev) {
  const int q = (dev >= 0 && dev < 64) ? pair_max_clusters_table()[dev] : 0;
  const int half = sms / 2 > 0 ? sms / 2 : 1;
  return q > 0 && q < half ? q : half;
}

// Checks a resolved configuration for this shape; fills the kernel params.
inline int pair_plan(const sgr_config& c, int pairs_avail, int M, int N, int K, PairParams* p, int* grid,
                     size_t* smem) {
  if (!pair_supported(M, N, K)) return SGR_ERR_UNSUPPORTED;
  const int nt = c.tile_n;
  if (!pair_kernel_for(nt)) return SGR_ERR_UNSUPPORTED;
  if (c.ctas_per_sm != 1) return SGR_ERR_UNSUPPORTED;
  if (c.token_tile != 0 && c.token_tile != kPairM) return SGR_ERR_UNSUPPORTED;
  if (c.k_split > 1) return SGR_ERR_UNSUPPORTED;
  const int kbps = c.k_blocks_per_stage == 0 ? 1 : c.k_blocks_per_stage;
  if (kbps != 1 && kbps != 2 && kbps != 4) return SGR_ERR_UNSUPPORTED;
  if (c.stages < 2 || c.stages > kPairMaxStages) return SGR_ERR_UNSUPPORTED;
  if (c.prefetch_stages < 0 || c.prefetch_stages > c.stages) return SGR_ERR_UNSUPPORTED;  // 0: all
  if (pairs_avail < 1) return SGR_ERR_UNSUPPORTED;
  const size_t sm = pair_smem_bytes(c.stages, nt, kbps);
  if (sm > 232448) return SGR_ERR_UNSUPPORTED;
  const long long m_tiles = (M + kPairM - 1) / kPairM;
  const long long n_tiles = (N + nt - 1) / nt;
  if (m_tiles * n_tiles > (1ll << 30)) return SGR_ERR_UNSUPPORTED;
  const long long tiles = m_tiles * n_tiles;
  const long long pairs = tiles < pairs_avail ? tiles : pairs_avail;
  p->M = M;
  p->N = N;
  p->K = K;
  p->NT = nt;
  p->m_tiles = (int)m_tiles;
  p->n_tiles = (int)n_tiles;
  p->k_blocks = (K + kTcKBlock - 1) / kTcKBlock;
  p->kbps = kbps;
  p->stages = c.stages;
  p->prefetch = c.prefetch_stages > 0 ? c.prefetch_stages : c.stages;
  p->tmem_cols = detail::pow2_at_least(2 * nt);
  *grid = (int)(2 * pairs);
  *smem = sm;
  return SGR_OK;
}

inline int pair_launch(const sgr_config& c, int pairs_avail, unsigned* err, const void* A, long long lda, const void* W,
                       const void* R, long long ldr, void* Y, long long ldy, int M, int N, int K, bool pdl,
                       cudaStream_t stream) {
  PairParams p;
  int grid = 0;
  size_t smem = 0;
  int rc = pair_plan(c, pairs_avail, M, N, K, &p, &grid, &smem);
  if (rc != SGR_OK) return rc;
  CUtensorMap tmA, tmW;
  if (!detail::make_tmap(&tmA, A, M, K, lda, kPairHalf, kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap(&tmW, W, N, K, K, p.NT / 2, kTcKBlock)) return SGR_ERR_LAUNCH;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.ldr = ldr;
  p.ldy = ldy;
  p.err = err;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kPairThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  attr[n_attr].id = cudaLaunchAttributeClusterDimension;
  attr[n_attr].val.clusterDim.x = 2;
  attr[n_attr].val.clusterDim.y = 1;
  attr[n_attr].val.clusterDim.z = 1;
  ++n_attr;
  lc.attrs = attr;
  lc.numAttrs = n_attr;
  cudaError_t e = cudaErrorInvalidValue;
  switch (p.NT) {
    case 64: e = cudaLaunchKernelEx(&lc, pair_gemm_kernel<64>, tmA, tmW, p); break;
    case 96: e = cudaLaunchKernelEx(&lc, pair_gemm_kernel<96>, tmA, tmW, p); break;
    case 128: e = cudaLaunchKernelEx(&lc, pair_gemm_kernel<128>, tmA, tmW, p); break;
    case 192: e = cudaLaunchKernelEx(&lc, pair_gemm_kernel<192>, tmA, tmW, p); break;
    case 256: e = cudaLaunchKernelEx(&lc, pair_gemm_kernel<256>, tmA, tmW, p); break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

}  // namespace sgr
