// sgr_gemm.cuh -- tensor-core tile GEMM for compute-bound token counts.
//
// Same operation as the other kernels: Y[m,n] = bf16_rn( sum_k A[m,k] W[n,k]
// + R[m,n] ) with FP32 accumulation and one rounding (vLLM
// "benchmark_k3_cutedsl_residual.py", module docstring and its correctness()
// reference).  Above a few hundred tokens the arithmetic intensity (about M
// FLOP per byte of W) passes the ridge point of tensor peak over HBM
// bandwidth (the roofline reasoning in the bitsandbytes "QLORA-2" comparison
// page, agents/kbit_gemm_context.md), so this kernel is organised around the
// tensor core instead of the weight stream.
//
// Operand roles (not swapped): a tile of 128 activation rows (tokens) is the
// MMA's M side and lives in TMEM lanes 0..127; a tile of NT rows of W (NT =
// 64, 128, 192 or 256) is the MMA's N side (TMEM columns).  Output tiles are
// 128 x NT.  NT is chosen per shape so that the tile count fills the SMs in
// whole waves (N = 7168 with NT = 192 gives 38 column tiles: 152 tiles at
// M = 512, 304 at M = 1024 on 152 SMs).  A problem with too few tiles for the
// SMs splits each tile's K over the S = 2, 3 or 4 CTAs of a cluster, which
// sum their partial accumulators through distributed shared memory (no
// workspace; see the modes below).
//
// Persistent grid of min(tiles, SMs) CTAs; CTA c takes tiles c, c + G, ...,
// each tile index t split as (t mod m_tiles, t div m_tiles), so the CTAs
// running at the same time share W column tiles and the whole of A in L2.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA loads of one 64-wide K
// block of A (128 x 64) and of W (NT x 64) per ring stage; warp 1 owns 2 x NT
// TMEM columns (two accumulators) and its lane 0 issues tcgen05.mma (4 per K
// block) and commits stage releases and accumulator hand-offs to mbarriers;
// warps 2-5 are the epilogue, one per 32-lane TMEM quarter, one output row
// per thread: the thread loads its row's NT residuals into registers when
// the tile starts (they arrive while the MMAs run), then adds the
// accumulator, rounds once to BF16 and stores 16-byte vectors.  Keeping the
// epilogue out of shared memory leaves all of it to the ring, whose depth is
// what hides the operand latency (about 1 us from L2 under full load).  The
// two accumulators let the epilogue of one tile run under the MMAs of the
// next.  W (input-only by the launch contract) is requested for the first
// ring stages before griddepcontrol.wait; A, R and Y are touched only after
// it.
//
// The single producer and MMA threads keep their ring position, K offset
// and tile coordinates by increments: an integer division on their
// per-stage path costs more issue time than the tensor core needs for a K
// block.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sgr_ptx.cuh"
#include "sgr_tc.cuh"
#include "skinny_gemm_residual.h"

namespace sgr {

constexpr int kTileThreads = 192;
constexpr int kTileM = 128;       // tokens per tile (MMA M, TMEM lanes)
constexpr int kTileEpiRows = 32;  // rows per epilogue warp (its TMEM lane quarter)
constexpr int kTileMaxN = 256;    // largest MMA N for M = 128
constexpr int kTileMaxStages = 16;

struct TileParams {
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  long long ldr, ldy;
  unsigned* err;
  int M, N, K;
  int NT;        // W rows per tile = MMA N (64, 128, 192 or 256)
  int m_tiles;   // ceil(M / 128)
  int n_tiles;   // ceil(N / NT)
  int k_blocks;  // ceil(K / 64)
  int stages;    // ring depth
  int kbps;      // K blocks per ring stage (1, 2 or 4): more contiguous bytes per W row and fetch
  int prefetch;  // W stages requested before griddepcontrol.wait (0..stages)
  int kb_split;  // K split over an S-CTA cluster: rank r takes K blocks [r kb_split, (r + 1) kb_split), the last rank the rest
  int tmem_cols;
};

// One ring stage: kbps K blocks of A (128 x 64 boxes) then of W (NT x 64).
__host__ __device__ inline uint32_t tile_stage_bytes(int nt, int kbps) {
  return (uint32_t)kbps * ((uint32_t)kTileM * 128u + (uint32_t)nt * 128u);
}

__host__ __device__ inline size_t tile_smem_bytes(int stages, int nt, int kbps) {
  return 1024 /* alignment slack */ + 1024 /* barriers */ + (size_t)stages * tile_stage_bytes(nt, kbps);
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Two 16-column TMEM loads (32x32b.x16) followed by one wait; the wait names
// every destination register so that no use can be scheduled before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr + 16u)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 16 TMEM columns with the wait naming every destination register.
__device__ __forceinline__ void tmem_ld16w(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// CH (16 or 32) consecutive TMEM columns of this thread's lane.
template <int CH>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[CH]) {
  static_assert(CH == 16 || CH == 32, "16 or 32 columns");
  if constexpr (CH == 32) {
    tmem_ld32(taddr, r);
  } else {
    tmem_ld16w(taddr, r);
  }
}

// acc (FP32 bits) + two BF16 residuals packed in `res`, rounded once to BF16x2.
__device__ __forceinline__ uint32_t add_round_bf16x2(uint32_t acc_lo, uint32_t acc_hi, uint32_t res) {
  const __nv_bfloat162 y =
      __floats2bfloat162_rn(__uint_as_float(acc_lo) + bf16lo(res), __uint_as_float(acc_hi) + bf16hi(res));
  return *reinterpret_cast<const uint32_t*>(&y);
}

// The residual row segment R[m, n0 .. n0 + NT) of one thread into registers
// (zeros outside the matrix; N is a multiple of 8, so a 16-byte chunk is
// either wholly inside or wholly outside).
template <int NT>
__device__ __forceinline__ void load_residual_row(const TileParams& p, int m, int n0, uint4 (&rv)[NT / 8]) {
  const bool row_ok = m < p.M;
  const __nv_bfloat16* src = p.R + (size_t)(row_ok ? m : 0) * p.ldr + n0;
#pragma unroll
  for (int j = 0; j < NT / 8; ++j)
    rv[j] = (row_ok && n0 + 8 * j < p.N) ? *reinterpret_cast<const uint4*>(src + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
}

// Modes (template parameter MODE = S, the CTAs per tile):
// kTilePlain (S = 1): persistent CTAs, each tile's whole K in one CTA.
// kTileSplitK, kTileSplit3, kTileSplit4 (S = 2, 3, 4): one tile per S-CTA
// cluster, rank r accumulating the r-th run of kb_split K blocks (the last
// rank the rest).  Rank r owns the tile's columns [r NT/S, (r+1) NT/S).  At
// the end every rank sends each other rank the columns that rank owns
// through distributed shared memory (into the receiver's drained ring, one
// slot per sender), then sums its own columns over the S partial
// accumulators in rank order (rank 0 first, whichever rank finished first,
// so the result is deterministic), adds the residual, rounds once and
// stores.  A slot holds the sender's columns in groups of four, each group
// as 128 rows of 16 bytes, so the 32 lanes of a warp (32 consecutive rows)
// write one contiguous 512-byte run per store: scattered 16-byte remote
// stores (one row per lane) measured 4-5x slower.  This multiplies the CTAs working on a problem with few tiles
// (M <= 256 at N = 7168) and divides each CTA's operand bytes and MMAs by S.
// Every CTA loads its own operands with plain TMA copies into its own
// shared memory.
enum : int { kTilePlain = 1, kTileSplitK = 2, kTileSplit3 = 3, kTileSplit4 = 4 };

// Threads per CTA: producer warp, MMA warp, four epilogue warps.  (A second
// MMA-issuing warp taking every other ring slot into its own accumulator was
// measured 1-4% slower here: with the whole ring in flight the K-block rate
// is set by the operand latency, not by the issuing thread's loop.)
__host__ __device__ constexpr int tile_threads(int mode) { return (void)mode, kTileThreads; }

template <int NT, int MODE>
__global__ void __launch_bounds__(tile_threads(MODE), 1)
    tile_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const TileParams p) {
  constexpr int KSPLIT = MODE;  // CTAs per tile
  constexpr int CL = MODE;      // CTAs per cluster

  static_assert(MODE >= 1 && MODE <= 4 && NT % MODE == 0 && (NT / MODE) % 16 == 0,
                "split tiles hand over whole 16-column pieces");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(sb);  // [S]  TMA -> MMA
  uint64_t* empty = full + S;                         // [S]  MMA -> TMA
  uint64_t* acc_full = empty + S;                     // [2]  MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;                 // [2]  epilogue (4 warps) -> MMA
  uint64_t* drain = acc_empty + 2;                    // [1]  MMA completion at exit
  uint64_t* peer_drained = drain + 1;                 // [1]  split: every other rank's ring is free
  uint64_t* received = peer_drained + 1;              // [1]  split: every other rank's columns have arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(received + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int KP = p.kbps;
  const uint32_t a_box = (uint32_t)kTileM * 128u;     // one A box: 128 rows x 64 K
  const uint32_t w_box = (uint32_t)NT * 128u;         // one W box: NT rows x 64 K
  const uint32_t a_part = (uint32_t)KP * a_box;       // A boxes at the start of a stage, W boxes after
  const uint32_t stage_bytes = tile_stage_bytes(NT, KP);
  const uint32_t ring = base + 1024;  // [S] x {KP A boxes, KP W boxes}

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int G = (int)gridDim.x / CL;      // tile-processing units (CTAs or clusters)
  const int unit = (int)blockIdx.x / CL;  // this CTA's unit
  // Tiles of a unit: (token tile, W column tile).
  const int mt_u = p.m_tiles;
  const int tiles = mt_u * p.n_tiles;
  const int my_tiles = (tiles - unit + G - 1) / G;  // >= 1: units <= tiles; 1 when split
  const int kb0 = KSPLIT > 1 ? (int)rank * p.kb_split : 0;
  const int KB = (KSPLIT > 1 && (int)rank < KSPLIT - 1) ? p.kb_split : p.k_blocks - kb0;  // K blocks of this CTA
  const int KS = (KB + KP - 1) / KP;  // ring stages per tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(peer_drained), KSPLIT > 1 ? KSPLIT - 1 : 1);
    mbar_init(smem_u32(received), KSPLIT > 1 ? (KSPLIT - 1) * 4 * 32 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmW);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (CL > 1) cluster_sync_all();  // the other ranks' barriers exist before any remote access
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();  // the dependent grid still waits for our completion before reading

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();  // re-read by the CTAs of the other token tiles
      const uint64_t pol_a = policy_evict_last();    // re-read for every W column tile
      const int total = my_tiles * KS;               // stages this CTA loads
      // Cursor over (local tile, K block) advanced by increments only: the
      // producer's per-stage path holds no integer division, which on this
      // single issuing thread costs more than the MMAs it feeds.
      struct Cursor {
        int kx, t, m0, n0, kb;
      };
      auto start = [&](Cursor& c) {
        c.kx = kb0 * kTcKBlock;
        c.kb = 0;
        c.t = unit;
        c.m0 = (c.t % mt_u) * kTileM;
        c.n0 = (c.t / mt_u) * NT;
      };
      auto advance = [&](Cursor& c) {
        c.kx += KP * kTcKBlock;
        if (++c.kb == KS) {
          c.kb = 0;
          c.kx = kb0 * kTcKBlock;
          c.t += G;
          c.m0 = (c.t % mt_u) * kTileM;
          c.n0 = (c.t / mt_u) * NT;
        }
      };
      // W box j of a stage.
      auto load_w = [&](uint32_t stage, int j, int kx, int n0, uint32_t fb) {
        tma_load_2d(stage + a_part + (uint32_t)j * w_box, &tmW, kx + j * kTcKBlock, n0, fb, pol_w);
      };
      const int pre = total < p.prefetch ? total : p.prefetch;  // <= S: slots 0 .. pre-1
      Cursor c;
      start(c);
      for (int it = 0; it < pre; ++it, advance(c)) {
        const uint32_t fb = smem_u32(&full[it]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        for (int j = 0; j < KP; ++j) load_w(ring + (uint32_t)it * stage_bytes, j, c.kx, c.n0, fb);
      }
      pdl_wait();
      {
        Cursor ca;
        start(ca);
        for (int it = 0; it < pre; ++it, advance(ca))
          for (int j = 0; j < KP; ++j)
            tma_load_2d(ring + (uint32_t)it * stage_bytes + (uint32_t)j * a_box, &tmA, ca.kx + j * kTcKBlock,
                        ca.m0, smem_u32(&full[it]), pol_a);
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
        const uint32_t fb = smem_u32(&full[slot]);
        const uint32_t st = ring + soff;
        mbar_arrive_expect_tx(fb, stage_bytes);
        for (int j = 0; j < KP; ++j) {
          tma_load_2d(st + (uint32_t)j * a_box, &tmA, c.kx + j * kTcKBlock, c.m0, fb, pol_a);
          load_w(st, j, c.kx, c.n0, fb);
        }
        issued = it + 1;
        soff += stage_bytes;
        if (++slot == S) {
          slot = 0;
          soff = 0;
          par ^= 1u;
        }
      }
      // Drain: every issued copy has landed before the CTA may exit.
      for (int t = issued > S ? issued - S : 0; t < issued; ++t)
        if (!mbar_wait(smem_u32(&full[t % S]), (t / S) & 1)) {
          report_error(p.err, kErrDrain);
          break;
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, NT);
      const uint64_t adesc0 = smem_desc_sw128(ring);
      const uint64_t wdesc0 = smem_desc_sw128(ring + a_part);
      bool ok = true;
      int slot = 0;
      uint32_t par = 0;   // ring round parity of `slot`
      uint64_t doff = 0;  // slot * stage_bytes >> 4 (descriptor start-address units)
      const uint64_t dstep = stage_bytes >> 4;
      const uint64_t a_win = (uint64_t)(a_box >> 4), w_win = (uint64_t)(w_box >> 4);  // one K block
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait_or_abort(smem_u32(&acc_empty[buf]), ((i >> 1) - 1) & 1, abort_flag)) {
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
              mma_bf16(d, aj + (uint64_t)(kk * 2), wj + (uint64_t)(kk * 2), idesc, accum);  // K step: 32 bytes
              accum = 1u;
            }
            aj += a_win;
            wj += w_win;
          }
          mma_commit(smem_u32(&empty[slot]));
          doff += dstep;
          if (++slot == S) {
            slot = 0;
            doff = 0;
            par ^= 1u;
          }
        }
        if (ok) mma_commit(smem_u32(&acc_full[buf]));
      }
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      mma_commit(smem_u32(drain));
      if (!mbar_wait(smem_u32(drain), 0)) report_error(p.err, kErrDrain);
    }
  } else if constexpr (KSPLIT == 1) {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // R may come from the preceding kernel; Y may be read by it
    const int q = warp & 3;  // TMEM lane quarter = tile rows [32 q, 32 q + 32)
    int t = unit;
    int m = (t % mt_u) * kTileM + q * kTileEpiRows + lane;  // this thread's output row
    int n0 = (t / mt_u) * NT;
    uint4 rv[NT / 8];
    load_residual_row<NT>(p, m, n0, rv);
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
      for (int c = 0; c < NT / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), v);  // warp-collective: every lane loads
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 r = rv[c * 4 + j];
          const int e = j * 8;
          const uint4 y = make_uint4(add_round_bf16x2(v[e + 0], v[e + 1], r.x), add_round_bf16x2(v[e + 2], v[e + 3], r.y),
                                     add_round_bf16x2(v[e + 4], v[e + 5], r.z), add_round_bf16x2(v[e + 6], v[e + 7], r.w));
          if (m < p.M && n0 + c * 32 + e < p.N) *reinterpret_cast<uint4*>(dst + c * 32 + e) = y;
        }
      }
      // Accumulator buffer free for the MMAs of tile i + 2.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[buf]));
      if (i + 1 < my_tiles) {  // next tile's residuals arrive during its main loop
        t += G;
        m = (t % mt_u) * kTileM + q * kTileEpiRows + lane;
        n0 = (t / mt_u) * NT;
        load_residual_row<NT>(p, m, n0, rv);
      }
    }
  } else {
    // ------------------------------------------------------- split epilogue
    pdl_wait();  // R may come from the preceding kernel; Y may be read by it
    constexpr int H = NT / KSPLIT;                 // columns each rank finishes
    constexpr int CH = H % 32 == 0 ? 32 : 16;      // columns per TMEM load
    constexpr uint32_t SLOT = (uint32_t)kTileM * (uint32_t)H * 4u;  // bytes of one sender's slot
    // Column group g (columns 4g .. 4g+3) of row r sits at (g * 128 + r) * 16.
    const int q = warp & 3;            // TMEM lane quarter = tile rows [32 q, 32 q + 32)
    const int row = q * 32 + lane;     // row within the tile
    const int m = (unit % p.m_tiles) * kTileM + row;
    const int own0 = (int)rank * H;    // first column (within the tile) this rank finishes
    const int n0 = (unit / p.m_tiles) * NT + own0;
    uint4 rv[H / 8];
    load_residual_row<H>(p, m, n0, rv);
    bool ok = mbar_wait_sleepy_or_abort(smem_u32(&acc_full[0]), 0, abort_flag);
    if (!ok) {
      if (!*abort_flag) report_error(p.err, kErrWaitMma);
      *abort_flag = 1;
    }
    ok = __all_sync(0xffffffffu, ok);
    // This rank's ring is drained (all its MMAs are done): tell the others.
    named_bar_sync(1, 128);
    if (threadIdx.x == 64)
      for (int o = 0; o < KSPLIT; ++o)
        if (o != (int)rank) mbar_arrive_remote(map_to_rank(smem_u32(peer_drained), (uint32_t)o));
    // Wait until every other rank's ring is drained, then write into rank o's
    // ring (slot of this sender) the columns of this accumulator that o finishes.
    bool peer_ok = mbar_wait_cluster(smem_u32(peer_drained), 0, abort_flag);
    peer_ok = __all_sync(0xffffffffu, peer_ok);
    tc_fence_after();
    const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
    if (ok && peer_ok) {
#pragma unroll
      for (int o = 0; o < KSPLIT; ++o) {
        if (o == (int)rank) continue;
        const uint32_t sidx = (int)rank < o ? rank : rank - 1u;  // this sender's slot at rank o
        const uint32_t dst = map_to_rank(ring + sidx * SLOT + (uint32_t)row * 16u, (uint32_t)o);
#pragma unroll
        for (int c = 0; c < H / CH; ++c) {
          uint32_t v[CH];
          tmem_ld_cols<CH>(taddr + (uint32_t)(o * H + c * CH), v);
#pragma unroll
          for (int j = 0; j < CH / 4; ++j)
            st_cluster_v4(dst + (uint32_t)((c * CH) / 4 + j) * (uint32_t)kTileM * 16u, v[4 * j], v[4 * j + 1],
                          v[4 * j + 2], v[4 * j + 3]);
        }
      }
    } else if (!peer_ok) {
      if (!*abort_flag) report_error(p.err, kErrWaitFixup);
      *abort_flag = 1;
    }
    // Every thread: its writes are released to each receiver.
    for (int o = 0; o < KSPLIT; ++o)
      if (o != (int)rank) mbar_arrive_remote(map_to_rank(smem_u32(received), (uint32_t)o));
    // Every other rank's partial of this rank's columns has arrived: sum in
    // rank order, add the residual, round, store.
    bool got = mbar_wait_cluster(smem_u32(received), 0, abort_flag);
    got = __all_sync(0xffffffffu, got);
    if (!got) {
      if (!*abort_flag) report_error(p.err, kErrWaitFixup);
      *abort_flag = 1;
    }
    if (ok && peer_ok && got) {
      const uint32_t src = ring + (uint32_t)row * 16u;
      __nv_bfloat16* yrow = p.Y + (size_t)(m < p.M ? m : 0) * p.ldy + n0;
#pragma unroll
      for (int c = 0; c < H / CH; ++c) {
        uint32_t v[CH];
        tmem_ld_cols<CH>(taddr + (uint32_t)(own0 + c * CH), v);
#pragma unroll
        for (int j = 0; j < CH / 8; ++j) {
          const int col = c * CH + 8 * j;
          float w[8];
#pragma unroll
          for (int r = 0; r < KSPLIT; ++r) {
            float part[8];
            if (r == (int)rank) {
#pragma unroll
              for (int e = 0; e < 8; ++e) part[e] = __uint_as_float(v[8 * j + e]);
            } else {
              const uint32_t sa = src + (uint32_t)(r < (int)rank ? r : r - 1) * SLOT + (uint32_t)(col / 4) * kTileM * 16u;
              const uint4 o0 = lds128(sa), o1 = lds128(sa + (uint32_t)kTileM * 16u);
              part[0] = __uint_as_float(o0.x), part[1] = __uint_as_float(o0.y);
              part[2] = __uint_as_float(o0.z), part[3] = __uint_as_float(o0.w);
              part[4] = __uint_as_float(o1.x), part[5] = __uint_as_float(o1.y);
              part[6] = __uint_as_float(o1.z), part[7] = __uint_as_float(o1.w);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = r == 0 ? part[e] : w[e] + part[e];
          }
          const uint4 rr = rv[col / 8];
          const uint4 y = make_uint4(
              add_round_bf16x2(__float_as_uint(w[0]), __float_as_uint(w[1]), rr.x),
              add_round_bf16x2(__float_as_uint(w[2]), __float_as_uint(w[3]), rr.y),
              add_round_bf16x2(__float_as_uint(w[4]), __float_as_uint(w[5]), rr.z),
              add_round_bf16x2(__float_as_uint(w[6]), __float_as_uint(w[7]), rr.w));
          if (m < p.M && n0 + col < p.N) *reinterpret_cast<uint4*>(yrow + col) = y;
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
  // No rank leaves while another may still write into its shared memory or
  // arrive on its barriers.
  if constexpr (CL > 1) cluster_sync_all();
}

// ------------------------------------------------------------------ host side
inline bool tile_supported(int M, int N, int K) {
  return M >= 1 && N >= 8 && K >= 8 && N % 8 == 0 && K % 8 == 0;
}

// Tile width and K split.  The default split is the 2-way one: 3- and 4-way
// splits (explicit configurations) measured slower at N = 7168 and M <= 128,
// their exchange of partial sums growing with the ranks faster than their K
// loops shrink.  With the K split over 2-CTA clusters (one tile per
// cluster, so it needs 2 x tiles <= SMs) the smallest width in {128, 192}
// that fits is taken while the problem has at most two 128-token tiles;
// otherwise the NT in {192, 256, 128, 64} with the least work per SM (waves
// of tiles x NT), the first listed winning ties.
inline void tile_default_shape(int sms, int M, int N, int K, int* nt_out, int* split_out) {
  const long long mt = (M + kTileM - 1) / kTileM;
  if (mt <= 2 && (K + kTcKBlock - 1) / kTcKBlock >= 2) {
    for (int nt : {128, 192}) {
      if (2 * mt * ((N + nt - 1) / nt) <= sms) {
        *nt_out = nt;
        *split_out = 2;
        return;
      }
    }
  }
  const int cand[4] = {192, 256, 128, 64};
  int best = cand[0];
  long long best_cost = -1;
  for (int nt : cand) {
    const long long tiles = mt * ((N + nt - 1) / nt);
    const long long cost = ((tiles + sms - 1) / sms) * nt;
    if (best_cost < 0 || cost < best_cost) {
      best = nt;
      best_cost = cost;
    }
  }
  *nt_out = best;
  *split_out = 1;
}

// Deepest ring that fits in the shared memory of one CTA.
inline int tile_default_stages(int nt, int kbps = 1) {
  long long st = (232448 - 2048) / tile_stage_bytes(nt, kbps);
  return (int)(st > kTileMaxStages ? kTileMaxStages : (st < 2 ? 2 : st));
}

inline void tile_default_config(int sms, int M, int N, int K, sgr_config* c) {
  c->path = SGR_PATH_TILE;
  c->ctas_per_sm = 1;
  tile_default_shape(sms, M, N, K, &c->tile_n, &c->k_split);
  c->stages = tile_default_stages(c->tile_n);
  c->prefetch_stages = 0;  // all stages
  c->token_tile = kTileM;
  c->k_blocks_per_stage = 1;
  c->rows_per_stage = 0;
}

// Tile widths each mode is built for: every width without a split; with an
// S-way split, widths whose share per rank (NT / S) is a whole number of
// 16-column pieces, limited to the ones that fill the SMs at N = 7168
// (S = 2: 64, 128, 192; S = 3: 192; S = 4: 128, 192, 256).
__host__ __device__ constexpr bool tile_has(int nt, int mode) {
  return mode == kTilePlain ? (nt == 64 || nt == 128 || nt == 192 || nt == 256)
         : mode == kTileSplitK ? (nt == 64 || nt == 128 || nt == 192)
         : mode == kTileSplit3 ? nt == 192
         : mode == kTileSplit4 ? (nt == 128 || nt == 192 || nt == 256)
                               : false;
}

// The kernel instantiation for a tile width and mode (nullptr if none).
template <int MODE>
inline const void* tile_kernel_mode(int nt) {
  switch (nt) {
    case 64:
      if constexpr (tile_has(64, MODE)) return reinterpret_cast<const void*>(tile_gemm_kernel<64, MODE>);
      break;
    case 128:
      if constexpr (tile_has(128, MODE)) return reinterpret_cast<const void*>(tile_gemm_kernel<128, MODE>);
      break;
    case 192:
      if constexpr (tile_has(192, MODE)) return reinterpret_cast<const void*>(tile_gemm_kernel<192, MODE>);
      break;
    case 256:
      if constexpr (tile_has(256, MODE)) return reinterpret_cast<const void*>(tile_gemm_kernel<256, MODE>);
      break;
    default:
      break;
  }
  return nullptr;
}

inline const void* tile_kernel_for(int nt, int mode) {
  switch (mode) {
    case kTilePlain: return tile_kernel_mode<kTilePlain>(nt);
    case kTileSplitK: return tile_kernel_mode<kTileSplitK>(nt);
    case kTileSplit3: return tile_kernel_mode<kTileSplit3>(nt);
    case kTileSplit4: return tile_kernel_mode<kTileSplit4>(nt);
    default: return nullptr;
  }
}

// Mode of a configuration: k_split 0 or 1 -> plain; 2, 3, 4 -> that split;
// anything else -> 0 (unsupported).
inline int tile_mode(const sgr_config& c) {
  const int split = c.k_split == 0 ? 1 : c.k_split;
  return split >= 1 && split <= 4 ? split : 0;
}

// Clusters of S = 2, 3, 4 CTAs (one CTA per SM) the device holds at once,
// per device, from cudaOccupancyMaxActiveClusters: a split launch has one
// tile per cluster and must fit in one wave.
inline int* tile_split_cluster_table() {
  static int table[64][5] = {{0}};
  return &table[0][0];
}

inline cudaError_t tile_init_device(int dev) {
  for (int mode = kTilePlain; mode <= kTileSplit4; ++mode)
    for (int nt : {64, 128, 192, 256}) {
      const void* fn = tile_kernel_for(nt, mode);
      if (!fn) continue;
      cudaError_t e = set_kernel_smem_attrs(fn);
      if (e != cudaSuccess) return e;
    }
  for (int S = 2; S <= 4; ++S) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)S, 1, 1);
    lc.blockDim = dim3((unsigned)kTileThreads, 1, 1);
    lc.dynamicSmemBytes = 232448 - 1024;  // above half an SM's shared memory: one CTA per SM
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, tile_kernel_for(192, S), &lc);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) tile_split_cluster_table()[dev * 5 + S] = n;
  }
  return cudaSuccess;
}

// Tiles an S-way split launch may have: the queried cluster count of the
// device, else SMs / S (host-only planning without a device).
inline int tile_split_capacity(int sms, int dev, int S) {
  const int q = (dev >= 0 && dev < 64 && S >= 2 && S <= 4) ? tile_split_cluster_table()[dev * 5 + S] : 0;
  const int even = S > 0 ? sms / S : 0;
  return q > 0 && q < even ? q : even;
}

// Checks a resolved configuration for this shape; fills the kernel params.
inline int tile_plan(const sgr_config& c, int sms, int M, int N, int K, TileParams* p, int* grid,
                     size_t* smem, int dev = -1) {
  if (!tile_supported(M, N, K)) return SGR_ERR_UNSUPPORTED;
  const int nt = c.tile_n;
  const int mode = tile_mode(c);
  if (!tile_kernel_for(nt, mode)) return SGR_ERR_UNSUPPORTED;
  if (c.ctas_per_sm != 1) return SGR_ERR_UNSUPPORTED;
  if (c.token_tile != 0 && c.token_tile != kTileM) return SGR_ERR_UNSUPPORTED;
  const int kbps = c.k_blocks_per_stage == 0 ? 1 : c.k_blocks_per_stage;
  if (kbps != 1 && kbps != 2 && kbps != 4) return SGR_ERR_UNSUPPORTED;
  if (c.stages < 2 || c.stages > kTileMaxStages) return SGR_ERR_UNSUPPORTED;
  if (c.prefetch_stages < 0 || c.prefetch_stages > c.stages) return SGR_ERR_UNSUPPORTED;  // 0: all
  const size_t sm = tile_smem_bytes(c.stages, nt, kbps);
  if (sm > 232448) return SGR_ERR_UNSUPPORTED;
  const long long m_tiles = (M + kTileM - 1) / kTileM;
  const long long n_tiles = (N + nt - 1) / nt;
  if (m_tiles * n_tiles > (1ll << 30)) return SGR_ERR_UNSUPPORTED;
  const long long tiles = m_tiles * n_tiles;
  const int k_blocks = (K + kTcKBlock - 1) / kTcKBlock;
  // Split over S ranks: each rank but the last takes ceil(k_blocks / S) K
  // blocks rounded up to whole stages (so that no stage reads into the next
  // rank's range), the last rank the rest.
  const int S = mode;
  const int kb_split = S > 1 ? ((k_blocks + S - 1) / S + kbps - 1) / kbps * kbps : k_blocks;
  if (S > 1) {
    // One tile per cluster, all clusters resident at once, every rank with
    // at least one K block, and the hand-over buffer (S - 1 slots of 128 rows
    // x NT/S floats) inside the ring.
    if (tiles > tile_split_capacity(sms, dev, S) || k_blocks - (S - 1) * kb_split < 1) return SGR_ERR_UNSUPPORTED;
    if ((size_t)(S - 1) * kTileM * (nt / S) * 4 > (size_t)c.stages * tile_stage_bytes(nt, kbps))
      return SGR_ERR_UNSUPPORTED;
  }
  p->M = M;
  p->N = N;
  p->K = K;
  p->NT = nt;
  p->m_tiles = (int)m_tiles;
  p->n_tiles = (int)n_tiles;
  p->k_blocks = k_blocks;
  p->kb_split = kb_split;
  p->kbps = kbps;
  p->stages = c.stages;
  p->prefetch = c.prefetch_stages > 0 ? c.prefetch_stages : c.stages;
  p->tmem_cols = detail::pow2_at_least(2 * nt);
  if (S > 1) {
    *grid = (int)(S * tiles);
  } else {
    *grid = (int)(tiles < sms ? tiles : sms);
  }
  *smem = sm;
  return SGR_OK;
}

template <int MODE>
inline cudaError_t tile_launch_mode(const cudaLaunchConfig_t* lc, int nt, const CUtensorMap& tmA, const CUtensorMap& tmW,
                                    const TileParams& p) {
  switch (nt) {
    case 64:
      if constexpr (tile_has(64, MODE)) return cudaLaunchKernelEx(lc, tile_gemm_kernel<64, MODE>, tmA, tmW, p);
      break;
    case 128:
      if constexpr (tile_has(128, MODE)) return cudaLaunchKernelEx(lc, tile_gemm_kernel<128, MODE>, tmA, tmW, p);
      break;
    case 192:
      if constexpr (tile_has(192, MODE)) return cudaLaunchKernelEx(lc, tile_gemm_kernel<192, MODE>, tmA, tmW, p);
      break;
    case 256:
      if constexpr (tile_has(256, MODE)) return cudaLaunchKernelEx(lc, tile_gemm_kernel<256, MODE>, tmA, tmW, p);
      break;
    default:
      break;
  }
  return cudaErrorInvalidValue;
}

inline int tile_launch(const sgr_config& c, int sms, int dev, unsigned* err, const void* A, long long lda,
                       const void* W, const void* R, long long ldr, void* Y, long long ldy, int M,
                       int N, int K, bool pdl, cudaStream_t stream) {
  TileParams p;
  int grid = 0;
  size_t smem = 0;
  int rc = tile_plan(c, sms, M, N, K, &p, &grid, &smem, dev);
  if (rc != SGR_OK) return rc;
  const int mode = tile_mode(c);
  CUtensorMap tmA, tmW;
  if (!detail::make_tmap(&tmA, A, M, K, lda, kTileM, kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap(&tmW, W, N, K, K, p.NT, kTcKBlock)) return SGR_ERR_LAUNCH;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.ldr = ldr;
  p.ldy = ldy;
  p.err = err;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3((unsigned)tile_threads(mode), 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  if (mode != kTilePlain) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = (unsigned)mode;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  lc.attrs = attr;
  lc.numAttrs = n_attr;
  cudaError_t e = cudaErrorInvalidValue;
  switch (mode) {
    case kTilePlain: e = tile_launch_mode<kTilePlain>(&lc, p.NT, tmA, tmW, p); break;
    case kTileSplitK: e = tile_launch_mode<kTileSplitK>(&lc, p.NT, tmA, tmW, p); break;
    case kTileSplit3: e = tile_launch_mode<kTileSplit3>(&lc, p.NT, tmA, tmW, p); break;
    case kTileSplit4: e = tile_launch_mode<kTileSplit4>(&lc, p.NT, tmA, tmW, p); break;
    default: break;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

}  // namespace sgr
