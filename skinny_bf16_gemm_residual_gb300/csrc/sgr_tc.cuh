// sgr_tc.cuh -- tensor-core path: tcgen05.mma with tensor-memory accumulators,
// fed by TMA, persistent stream-K over K, deterministic split-K fixup.
//
// Computes Y[m,n] = bf16_rn( sum_k A[m,k] * W[n,k] + R[m,n] ), the operation of
// the vLLM "benchmark_k3_cutedsl_residual.py" page (BF16 inputs, FP32
// accumulation, BF16 output), rounding once in the epilogue.
//
// Operand roles ("swap-AB"): a 128-row slab of W is the MMA's M side (it lives
// in TMEM lanes 0..127), a tile of NT activation rows (tokens) is the MMA's N
// side (TMEM columns).  At decode sizes (M <= 16) the token tile is 16 wide, so
// the tensor core does the whole contraction and the kernel is a pure W
// stream; at M >= 256 it is a regular tensor-core GEMM with 128 x NT tiles.
//
// Work decomposition: a unit is one ring stage = one (token tile, W tile,
// K stage of 64*kbps) triple; units are linearised W-tile-major, then token
// tile, then K, and CTA c of the persistent grid takes units
// [U*c/G, U*(c+1)/G).  A CTA's units split into segments of one output tile
// each.  A segment covering the tile's whole K is finished in place; the
// others write FP32 partial tiles to a workspace and the last CTA to arrive
// at the tile's counter sums every partial in K order (so results do not
// depend on arrival order), adds R, rounds and stores, and resets the counter.
// Every contributor arrives on the counter even after one of its waits ran
// out, so the counters are zero again at the end of every call.
// This replaces the vLLM page's one-CTA-per-outputs_per_block-rows grid,
// which leaves most of 152 SMs idle or in a ragged last wave.
//
// Warp roles (192 threads): warp 0 lane 0 issues TMA loads into a
// `stages`-deep shared-memory ring; warp 1 owns the tensor memory and its
// lane 0 issues tcgen05.mma (4 per 64-wide K block) and commits stage
// releases / accumulator hand-offs to mbarriers; warps 2-5 are the epilogue
// (tcgen05.ld of their 32-lane quarter, residual add, rounding, stores, and
// the split-K fixup).  Two TMEM accumulators let the epilogue of one segment
// overlap the MMAs of the next.  W is loaded before griddepcontrol.wait (it
// must not be produced by the preceding kernel); A, R, Y and the workspace
// are touched only after it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sgr_ptx.cuh"
#include "skinny_gemm_residual.h"

namespace sgr {

constexpr int kTcThreads = 192;
constexpr int kTcTileRows = 128;  // W rows per MMA tile (MMA M)
constexpr int kTcKBlock = 64;     // K elements per 128-byte swizzled row
constexpr int kTcMaxCtasPerSm = 2;
constexpr int kTcMaxTokenTile = 256;
constexpr int kTcMaxCounters = 1 << 20;

struct TcWorkspace {
  float* partials = nullptr;  // [G][2][NT][128] FP32 partial tiles
  unsigned* counters = nullptr;
  size_t partial_floats = 0;
  int counter_count = 0;
};

struct TcParams {
  const __nv_bfloat16* R;
  __nv_bfloat16* Y;
  long long ldr, ldy;
  float* ws;
  unsigned* counters;
  unsigned* err;
  long long units;  // n_tiles * m_tiles * k_stages
  int M, N, K;
  int NT;        // token tile = MMA N (multiple of 16, <= 256)
  int m_tiles;   // ceil(M / NT)
  int k_stages;  // ceil(K / (64 * kbps))
  int kbps;      // 64-wide K blocks per stage
  int stages;    // ring depth
  int chains;    // independent TMEM accumulators per buffer (1, 2 or 4)
  int tmem_cols;
  int abort_cta;  // self-test only: this CTA's epilogue acts as if its first wait ran out (-1: none)
};

__host__ __device__ inline uint32_t tc_stage_bytes(int kbps, int nt) {
  return (uint32_t)kbps * (kTcTileRows * 128u + (uint32_t)nt * 128u);
}

__host__ __device__ inline size_t tc_smem_bytes(int stages, int kbps, int nt) {
  return 1024 /* alignment slack */ + 1024 /* barriers */ + (size_t)stages * tc_stage_bytes(kbps, nt);
}

__device__ __forceinline__ long long tc_unit_begin(long long U, int G, int c) {
  return U * c / G;
}

// The CTA whose unit range contains unit u.
__device__ __forceinline__ int tc_cta_of(long long U, int G, long long u) {
  return (int)(((u + 1) * G - 1) / U);
}

// Wait that also returns (false) as soon as another role of the CTA aborted.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_test_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > SGR_WAIT_LIMIT_NS) return false;
  }
}

// The same for waits that may last microseconds (a consumer ahead of its
// producer, an epilogue waiting for the whole main loop, a CTA launched early
// by programmatic dependent launch): after a short spin the thread sleeps
// between polls (32 ns doubling to 256 ns), so that it does not take issue
// slots from the warps that do the work on the same SM sub-partition.
__device__ __forceinline__ bool mbar_wait_sleepy_or_abort(uint32_t bar, uint32_t parity,
                                                          volatile int* abort_flag) {
#pragma unroll 1
  for (int i = 0; i < 8; ++i)
    if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  unsigned ns = 32;
  while (true) {
    __nanosleep(ns);
    if (mbar_test_wait(bar, parity)) return true;
    if (ns < 256) ns <<= 1;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > SGR_WAIT_LIMIT_NS) return false;
  }
}

// 16 accumulator columns summed over the chains, chain 0 first (fixed order).
__device__ __forceinline__ void tc_ld_chains(uint32_t taddr, int nt, int chains, float (&v)[16]) {
  tmem_ld16(taddr, v);
  for (int c = 1; c < chains; ++c) {
    float w[16];
    tmem_ld16(taddr + (uint32_t)(c * nt), w);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += w[i];
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                     const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sb = smem_raw + (base - raw);
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(sb);  // [S]  TMA -> MMA
  uint64_t* empty = full + S;                         // [S]  MMA -> TMA
  uint64_t* acc_full = empty + S;                     // [2]  MMA -> epilogue
  uint64_t* acc_empty = acc_full + 2;                 // [2]  epilogue -> MMA
  uint64_t* drain = acc_empty + 2;                    // [1]  MMA completion at exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* abort_flag = bcast + 1;
  const uint32_t ring = base + 1024;
  const uint32_t w_bytes = (uint32_t)p.kbps * kTcTileRows * 128u;
  const uint32_t stage_bytes = tc_stage_bytes(p.kbps, p.NT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const long long U = p.units;
  const long long u0 = tc_unit_begin(U, G, c), u1 = tc_unit_begin(U, G, c + 1);
  const int count = (int)(u1 - u0);
  const int KS = p.k_stages;

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
    *abort_flag = 0;
    *bcast = 0;
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
  // The dependent grid may be scheduled now: its own griddepcontrol.wait
  // still orders its reads of our outputs after this grid completes.
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();  // W is streamed once
      const uint64_t pol_a = policy_evict_last();   // A is re-read by every W tile
      auto unit_coords = [&](long long u, int& kx, int& wy, int& ay) {
        const long long t = u / KS;
        const int ks = (int)(u - t * KS);
        kx = ks * p.kbps * kTcKBlock;
        wy = (int)(t / p.m_tiles) * kTcTileRows;
        ay = (int)(t % p.m_tiles) * p.NT;
      };
      const int pre = count < S ? count : S;
      // Weights for the first stages before the dependency wait.
      for (int i = 0; i < pre; ++i) {
        int kx, wy, ay;
        unit_coords(u0 + i, kx, wy, ay);
        const uint32_t fb = smem_u32(&full[i]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        const uint32_t st = ring + (uint32_t)i * stage_bytes;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(st + (uint32_t)j * (kTcTileRows * 128u), &tmW, kx + j * kTcKBlock, wy, fb, pol_w);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        int kx, wy, ay;
        unit_coords(u0 + i, kx, wy, ay);
        const uint32_t st = ring + (uint32_t)i * stage_bytes + w_bytes;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(st + (uint32_t)(j * p.NT * 128), &tmA, kx + j * kTcKBlock, ay,
                      smem_u32(&full[i]), pol_a);
      }
      int issued = pre;
      for (int i = pre; i < count; ++i) {
        const int slot = i % S;
        if (!mbar_wait_or_abort(smem_u32(&empty[slot]), ((i / S) - 1) & 1, abort_flag)) {
          if (!*abort_flag) report_error(p.err, kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        int kx, wy, ay;
        unit_coords(u0 + i, kx, wy, ay);
        const uint32_t fb = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        const uint32_t st = ring + (uint32_t)slot * stage_bytes;
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(st + (uint32_t)j * (kTcTileRows * 128u), &tmW, kx + j * kTcKBlock, wy, fb, pol_w);
        for (int j = 0; j < p.kbps; ++j)
          tma_load_2d(st + w_bytes + (uint32_t)(j * p.NT * 128), &tmA, kx + j * kTcKBlock, ay, fb, pol_a);
        issued = i + 1;
      }
      // Every copy this CTA issued must land before the CTA may exit.
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
      int i = 0;
      int buf = 0;
      int nuse[2] = {0, 0};
      bool ok = true;
      long long u = u0;
      while (ok && u < u1) {
        const long long t = u / KS;
        const long long seg_end = (t + 1) * KS < u1 ? (t + 1) * KS : u1;
        if (nuse[buf] > 0 &&
            !mbar_wait_or_abort(smem_u32(&acc_empty[buf]), (nuse[buf] - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * p.chains * p.NT);
        bool seg_start = true;
        for (; u < seg_end; ++u, ++i) {
          const int slot = i % S;
          if (!mbar_wait_or_abort(smem_u32(&full[slot]), (i / S) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = ring + (uint32_t)slot * stage_bytes;
          for (int j = 0; j < p.kbps; ++j) {
#pragma unroll
            for (int kk = 0; kk < kTcKBlock / 16; ++kk) {
              // K step kk accumulates into chain kk % chains (independent MMAs pipeline).
              const int chain = kk & (p.chains - 1);
              const uint64_t ad = smem_desc_sw128(st + (uint32_t)j * (kTcTileRows * 128u) + kk * 32u);
              const uint64_t bd = smem_desc_sw128(st + w_bytes + (uint32_t)(j * p.NT * 128) + kk * 32u);
              const bool first = seg_start && j == 0 && kk < p.chains;
              mma_bf16(d + (uint32_t)(chain * p.NT), ad, bd, idesc, first ? 0u : 1u);
            }
          }
          seg_start = false;
          mma_commit(smem_u32(&empty[slot]));  // stage free once these MMAs finish
        }
        if (!ok) break;
        mma_commit(smem_u32(&acc_full[buf]));  // accumulator ready
        ++nuse[buf];
        buf ^= 1;
      }
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      mma_commit(smem_u32(drain));
      if (!mbar_wait(smem_u32(drain), 0)) report_error(p.err, kErrDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // R may come from the preceding kernel; Y/workspace may be read by it
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int etid = threadIdx.x - 64;  // 0..127
    bool ok = true;
    int buf = 0;
    int nuse[2] = {0, 0};
    long long u = u0;
    while (u < u1) {
      const long long t = u / KS;
      const long long t_begin = t * KS, t_end = t_begin + KS;
      const long long seg_end = t_end < u1 ? t_end : u1;
      const bool complete = (u == t_begin) && (seg_end == t_end);
      const bool first_seg = (u == u0);
      const int n_tile = (int)(t / p.m_tiles), m_tile = (int)(t % p.m_tiles);
      const int n = n_tile * kTcTileRows + row;
      const int m_base = m_tile * p.NT;
      const int m_count = min(p.NT, p.M - m_base);
      if (ok && (c == p.abort_cta || !mbar_wait_or_abort(smem_u32(&acc_full[buf]), nuse[buf] & 1, abort_flag))) {
        if (!*abort_flag) report_error(p.err, kErrWaitMma);
        *abort_flag = 1;
        ok = false;
      }
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * p.chains * p.NT);
      float* part = p.ws + (size_t)(c * 2 + (first_seg ? 0 : 1)) * p.NT * kTcTileRows;
      if (ok) {
        for (int col0 = 0; col0 < p.NT; col0 += 16) {
          float v[16];
          if (complete) {
            // Residual loads first (independent of the accumulator), then one
            // rounding per element.
            float r[16];
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const int m = col0 + cc;
              r[cc] = (m < m_count && n < p.N)
                          ? __bfloat162float(p.R[(size_t)(m_base + m) * p.ldr + n])
                          : 0.f;
            }
            tc_ld_chains(taddr + (uint32_t)col0, p.NT, p.chains, v);
            if (n < p.N) {
#pragma unroll
              for (int cc = 0; cc < 16; ++cc) {
                const int m = col0 + cc;
                if (m < m_count)
                  p.Y[(size_t)(m_base + m) * p.ldy + n] = __float2bfloat16_rn(v[cc] + r[cc]);
              }
            }
          } else {
            tc_ld_chains(taddr + (uint32_t)col0, p.NT, p.chains, v);
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) part[(size_t)(col0 + cc) * kTcTileRows + row] = v[cc];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[buf]));
      ++nuse[buf];
      buf ^= 1;

      if (!complete) {
        // Split-K fixup: the last of the tile's segments to arrive reduces all.
        __threadfence();
        named_bar_sync(1, 128);
        const int c_first = tc_cta_of(U, G, t_begin);
        const int c_last = tc_cta_of(U, G, t_end - 1);
        if (etid == 0) {
          // Every contributor arrives, also one whose wait ran out (the error
          // word records that), so that the counter always returns to zero
          // and the next call that uses it starts clean.  A contributor
          // without its own partial (ok false) never runs the fixup.
          const unsigned prev = atomicAdd(&p.counters[t], 1u);
          const bool last = (prev == (unsigned)(c_last - c_first));
          if (last) p.counters[t] = 0u;  // every contributor has arrived: reset for the next call
          __threadfence();
          *bcast = (last && ok) ? 1 : 0;
        }
        named_bar_sync(1, 128);
        if (*bcast && n < p.N) {
          // Sum the partials in K order (contributor order), 16 tokens at a
          // time with all loads of a group in flight together.
          for (int mc = 0; mc < m_count; mc += 16) {
            float acc[16], r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              acc[i] = 0.f;
              r[i] = (mc + i < m_count) ? __bfloat162float(p.R[(size_t)(m_base + mc + i) * p.ldr + n]) : 0.f;
            }
            for (int cc = c_first; cc <= c_last; ++cc) {
              const int h = (cc == c_first && tc_unit_begin(U, G, cc) < t_begin) ? 1 : 0;
              const float* src = p.ws + (size_t)(cc * 2 + h) * p.NT * kTcTileRows + (size_t)mc * kTcTileRows + row;
              float v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = (mc + i < m_count) ? __ldcg(src + (size_t)i * kTcTileRows) : 0.f;
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[i] += v[i];
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (mc + i < m_count)
                p.Y[(size_t)(m_base + mc + i) * p.ldy + n] = __float2bfloat16_rn(acc[i] + r[i]);
          }
        }
      }
      u = seg_end;
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
namespace detail {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return (EncodeTiledFn) nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D BF16 row-major [rows, cols] with row stride ld (elements); box
// box_cols x box_rows with the 128-byte swizzle; out-of-bounds reads as zero.
inline bool make_tmap(CUtensorMap* m, const void* ptr, long long rows, long long cols, long long ld,
                      int box_rows, int box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int round_up(int x, int a) { return (x + a - 1) / a * a; }

inline int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace detail

inline bool tc_supported(int M, int N, int K) {
  return M >= 1 && N >= 8 && K >= 8 && (N % 8) == 0 && (K % 8) == 0 &&
         (long long)((N + kTcTileRows - 1) / kTcTileRows) * ((M + kTcMaxTokenTile - 1) / kTcMaxTokenTile) <=
             kTcMaxCounters;
}

// Token tile: one tile of round_up(M, 16) up to 256; beyond, equal tiles.
inline int tc_token_tile(int M) {
  const int tiles = (M + kTcMaxTokenTile - 1) / kTcMaxTokenTile;
  return detail::round_up((M + tiles - 1) / tiles, 16);
}

inline void tc_default_config(int sms, int M, int N, int K, sgr_config* c) {
  (void)sms;
  (void)N;
  (void)K;
  c->path = SGR_PATH_TC;
  c->ctas_per_sm = 1;
  c->token_tile = tc_token_tile(M);
  c->k_blocks_per_stage = 2;
  const size_t stage = tc_stage_bytes(c->k_blocks_per_stage, c->token_tile);
  int s = (int)((200u * 1024u) / stage);
  c->stages = s > 8 ? 8 : (s < 2 ? 2 : s);
  c->rows_per_stage = 0;
}

inline cudaError_t tc_init_device(int sms, TcWorkspace* ws) {
  const size_t g = (size_t)sms * kTcMaxCtasPerSm;
  ws->partial_floats = g * 2 * kTcMaxTokenTile * kTcTileRows;
  cudaError_t e = cudaMalloc(&ws->partials, ws->partial_floats * sizeof(float));
  if (e != cudaSuccess) return e;
  e = cudaMalloc(&ws->counters, (size_t)kTcMaxCounters * sizeof(unsigned));
  if (e != cudaSuccess) return e;
  ws->counter_count = kTcMaxCounters;
  e = cudaMemset(ws->counters, 0, (size_t)kTcMaxCounters * sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return set_kernel_smem_attrs(reinterpret_cast<const void*>(tc_skinny_kernel));
}

// Checks a resolved TC configuration for this shape; fills the kernel params.
inline int tc_plan(const sgr_config& c, int sms, int M, int N, int K, TcParams* p, int* grid,
                   size_t* smem) {
  const int nt = c.token_tile;
  if (nt < 16 || nt > kTcMaxTokenTile || nt % 16 != 0) return SGR_ERR_UNSUPPORTED;
  if (c.k_blocks_per_stage < 1 || c.k_blocks_per_stage > 8) return SGR_ERR_UNSUPPORTED;
  if (c.ctas_per_sm < 1 || c.ctas_per_sm > kTcMaxCtasPerSm) return SGR_ERR_UNSUPPORTED;
  if (c.stages < 2 || c.stages > 32) return SGR_ERR_UNSUPPORTED;
  const size_t sm = tc_smem_bytes(c.stages, c.k_blocks_per_stage, nt);
  if (sm > 232448) return SGR_ERR_UNSUPPORTED;
  const int n_tiles = (N + kTcTileRows - 1) / kTcTileRows;
  const int m_tiles = (M + nt - 1) / nt;
  const int kstage_elems = kTcKBlock * c.k_blocks_per_stage;
  const int k_stages = (K + kstage_elems - 1) / kstage_elems;
  if ((long long)n_tiles * m_tiles > kTcMaxCounters) return SGR_ERR_UNSUPPORTED;
  const long long units = (long long)n_tiles * m_tiles * k_stages;
  long long g = (long long)sms * c.ctas_per_sm;
  if (g > units) g = units;
  p->M = M;
  p->N = N;
  p->K = K;
  p->NT = nt;
  p->m_tiles = m_tiles;
  p->k_stages = k_stages;
  p->kbps = c.k_blocks_per_stage;
  p->stages = c.stages;
  p->units = units;
  p->chains = nt <= 64 ? 4 : (nt <= 128 ? 2 : 1);  // 2 buffers * chains * NT <= 512 TMEM columns
  p->tmem_cols = detail::pow2_at_least(2 * p->chains * nt);
  p->abort_cta = -1;
  *grid = (int)g;
  *smem = sm;
  return SGR_OK;
}

inline int tc_launch(const sgr_config& c, int sms, unsigned* err, TcWorkspace* ws, const void* A,
                     long long lda, const void* W, const void* R, long long ldr, void* Y, long long ldy,
                     int M, int N, int K, bool pdl, cudaStream_t stream, int abort_cta = -1) {
  TcParams p;
  int grid = 0;
  size_t smem = 0;
  int rc = tc_plan(c, sms, M, N, K, &p, &grid, &smem);
  if (rc != SGR_OK) return rc;
  if (abort_cta >= grid) return SGR_ERR_UNSUPPORTED;
  p.abort_cta = abort_cta;
  if (!ws->partials || (size_t)grid * 2 * p.NT * kTcTileRows > ws->partial_floats) return SGR_ERR_UNSUPPORTED;
  CUtensorMap tmW, tmA;
  if (!detail::make_tmap(&tmW, W, N, K, K, kTcTileRows, kTcKBlock)) return SGR_ERR_LAUNCH;
  if (!detail::make_tmap(&tmA, A, M, K, lda, p.NT, kTcKBlock)) return SGR_ERR_LAUNCH;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.ldr = ldr;
  p.ldy = ldy;
  p.ws = ws->partials;
  p.counters = ws->counters;
  p.err = err;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kTcThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&lc, tc_skinny_kernel, tmW, tmA, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

inline const void* tc_kernel_for(int M, int N, int K, const sgr_config* c, int* smem, int* threads) {
  (void)M;
  (void)N;
  (void)K;
  *smem = (int)tc_smem_bytes(c->stages, c->k_blocks_per_stage, c->token_tile);
  *threads = kTcThreads;
  return reinterpret_cast<const void*>(tc_skinny_kernel);
}

}  // namespace sgr
