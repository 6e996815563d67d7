// sgr_api.cu -- C ABI of the skinny BF16 GEMM + residual library: argument
// validation, per-device set-up, path/config selection and kernel launch.
// The operation and its argument rules are documented in
// include/skinny_gemm_residual.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "skinny_gemm_residual.h"
#include "sgr_simt.cuh"
#include "sgr_tc.cuh"
#include "sgr_rows.cuh"
#include "sgr_gemm.cuh"
#include "sgr_pair.cuh"
#include "sgr_w8.cuh"
#include "sgr_w8s.cuh"
#include "sgr_table.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxDynSmem = 232448;  // 227 KB, the per-CTA opt-in limit on sm_100-class GPUs
constexpr long long kMaxN = 1 << 24;
constexpr long long kMaxK = 1 << 20;
constexpr long long kMaxM = 1 << 20;
// Row strides in elements: keeps the overlap arithmetic far from 64-bit
// overflow and every byte stride below the tensor maps' 2^40 limit.
constexpr long long kMaxLd = 1LL << 36;

__device__ unsigned g_sgr_error_word;

// Device address of g_sgr_error_word per device, resolved once with that
// device current.  Allocates nothing, so the allocation-free entry point and
// the error query can use it without the workspace set-up of init_device.
struct ErrorWord {
  std::once_flag once;
  int status = SGR_ERR_DEVICE;
  unsigned* ptr = nullptr;
};
ErrorWord g_err_word[kMaxDevices];

int error_word(int dev, unsigned** out) {
  if (dev < 0 || dev >= kMaxDevices) return SGR_ERR_DEVICE;
  ErrorWord& w = g_err_word[dev];
  std::call_once(w.once, [&] {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || (prev != dev && cudaSetDevice(dev) != cudaSuccess)) {
      cudaGetLastError();
      return;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sgr_error_word) == cudaSuccess) {
      w.ptr = static_cast<unsigned*>(p);
      w.status = SGR_OK;
    } else {
      cudaGetLastError();
    }
    if (prev != dev) cudaSetDevice(prev);
  });
  *out = w.ptr;
  return w.status;
}

struct DeviceState {
  std::once_flag once;
  int status = SGR_ERR_DEVICE;
  int sms = 0;
  unsigned* err = nullptr;
  sgr::TcWorkspace ws{};
};
DeviceState g_dev[kMaxDevices];

// ------------------------------------------------------------ SIMT kernels
using SimtFn = void (*)(const sgr::SimtParams);

template <int MT>
SimtFn simt_fn_vpt(int vpt) {
  switch (vpt) {
    case 1: return sgr::simt_skinny_kernel<MT, 1>;
    case 2: return sgr::simt_skinny_kernel<MT, 2>;
    case 4: return sgr::simt_skinny_kernel<MT, 4>;
    default: return nullptr;
  }
}

SimtFn simt_fn(int mt, int vpt) {
  switch (mt) {
    case 1: return simt_fn_vpt<1>(vpt);
    case 2: return simt_fn_vpt<2>(vpt);
    case 4: return simt_fn_vpt<4>(vpt);
    case 8: return simt_fn_vpt<8>(vpt);
    case 16: return simt_fn_vpt<16>(vpt);
    default: return nullptr;
  }
}

// FP8-weight instantiations (M <= 8).
template <int MT>
SimtFn simt_w8_fn_vpt(int vpt) {
  switch (vpt) {
    case 1: return sgr::simt_skinny_kernel<MT, 1, sgr::kWfE4m3>;
    case 2: return sgr::simt_skinny_kernel<MT, 2, sgr::kWfE4m3>;
    case 4: return sgr::simt_skinny_kernel<MT, 4, sgr::kWfE4m3>;
    default: return nullptr;
  }
}

SimtFn simt_w8_fn(int mt, int vpt) {
  switch (mt) {
    case 1: return simt_w8_fn_vpt<1>(vpt);
    case 2: return simt_w8_fn_vpt<2>(vpt);
    case 4: return simt_w8_fn_vpt<4>(vpt);
    case 8: return simt_w8_fn_vpt<8>(vpt);
    default: return nullptr;
  }
}

// NVFP4-weight instantiations: at most 4 token rows per pass and one 32-code
// vector per thread and row (K <= 7168), the register budget in which they
// build without spills.
constexpr int kW4PassM = 4;

SimtFn simt_w4_fn(int mt, int vpt) {
  if (vpt != 1) return nullptr;
  switch (mt) {
    case 1: return sgr::simt_skinny_kernel<1, 1, sgr::kWfNvfp4>;
    case 2: return sgr::simt_skinny_kernel<2, 1, sgr::kWfNvfp4>;
    case 4: return sgr::simt_skinny_kernel<4, 1, sgr::kWfNvfp4>;
    default: return nullptr;
  }
}

// 32-code vectors per row slice: K a multiple of 32, K <= 224 * 32.
int simt_w4_vpt(int K) {
  if (K % 32 != 0) return 0;
  return K / 32 <= sgr::kSimtConsumers ? 1 : 0;
}

// 16-code vectors per row slice: K a multiple of 16, K <= 224 * 16 * 4.
int simt_w8_vpt(int K) {
  if (K % 16 != 0) return 0;
  const int kv = K / 16;
  if (kv <= sgr::kSimtConsumers) return 1;
  if (kv <= 2 * sgr::kSimtConsumers) return 2;
  if (kv <= 4 * sgr::kSimtConsumers) return 4;
  return 0;
}

int simt_mt(int M) {
  if (M <= 1) return 1;
  if (M <= 2) return 2;
  if (M <= 4) return 4;
  if (M <= 8) return 8;
  if (M <= 16) return 16;
  return 0;
}

int simt_vpt(int K) {
  const int kv = K / 8;
  if (kv <= sgr::kSimtConsumers) return 1;
  if (kv <= 2 * sgr::kSimtConsumers) return 2;
  if (kv <= 4 * sgr::kSimtConsumers) return 4;
  return 0;
}

// ------------------------------------------------------------ helpers
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Extent {
  uintptr_t lo, hi;  // [lo, hi) bytes
};

Extent extent(const void* p, long long rows, long long ld, long long cols) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(p);
  if (rows <= 0 || cols <= 0) return {b, b};
  return {b, b + static_cast<uintptr_t>(((rows - 1) * ld + cols) * 2)};
}

bool overlap(Extent a, Extent b) { return a.lo < b.hi && b.lo < a.hi && a.lo < a.hi && b.lo < b.hi; }

int validate(const void* A, long long lda, const void* W, const void* R, long long ldr,
             const void* Y, long long ldy, int M, int N, int K) {
  if (M < 0 || N < 0 || K < 0) return SGR_ERR_SHAPE;
  if (M == 0 || N == 0) return SGR_OK;  // empty: nothing is read or written
  if (M > kMaxM || N > kMaxN || K > kMaxK) return SGR_ERR_UNSUPPORTED;
  if (N % 8 != 0 || K % 8 != 0) return SGR_ERR_SHAPE;
  if (!R || !Y) return SGR_ERR_NULL;
  if (K > 0 && (!A || !W)) return SGR_ERR_NULL;
  if (ldr < N || ldy < N) return SGR_ERR_SHAPE;
  if (K > 0 && lda < K) return SGR_ERR_SHAPE;
  if (ldr > kMaxLd || ldy > kMaxLd || (K > 0 && lda > kMaxLd)) return SGR_ERR_UNSUPPORTED;
  if (ldr % 8 != 0 || ldy % 8 != 0 || (K > 0 && lda % 8 != 0)) return SGR_ERR_ALIGN;
  if (!aligned16(R) || !aligned16(Y)) return SGR_ERR_ALIGN;
  if (K > 0 && (!aligned16(A) || !aligned16(W))) return SGR_ERR_ALIGN;
  const Extent ey = extent(Y, M, ldy, N);
  if (K > 0) {
    if (overlap(ey, extent(A, M, lda, K))) return SGR_ERR_ALIAS;
    if (overlap(ey, extent(W, N, K, K))) return SGR_ERR_ALIAS;
  }
  const bool in_place = (Y == R) && (ldy == ldr);
  if (!in_place && overlap(ey, extent(R, M, ldr, N))) return SGR_ERR_ALIAS;
  return SGR_OK;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  if (*dev < 0 || *dev >= kMaxDevices) return SGR_ERR_DEVICE;
  return SGR_OK;
}

int init_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return SGR_ERR_DEVICE;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&] {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) {
      cudaGetLastError();
      st.status = SGR_ERR_DEVICE;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      st.status = SGR_ERR_DEVICE;
      return;
    }
    int ok = SGR_OK;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      ok = SGR_ERR_DEVICE;
    unsigned* errp = nullptr;
    if (ok == SGR_OK && error_word(dev, &errp) != SGR_OK) ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && cudaMemset(errp, 0, sizeof(unsigned)) != cudaSuccess) ok = SGR_ERR_DEVICE;
    const int mts[5] = {1, 2, 4, 8, 16};
    const int vpts[3] = {1, 2, 4};
    for (int mt : mts)
      for (int v : vpts) {
        if (ok == SGR_OK && sgr::set_kernel_smem_attrs(reinterpret_cast<const void*>(simt_fn(mt, v))) != cudaSuccess)
          ok = SGR_ERR_DEVICE;
        if (ok == SGR_OK && mt <= 8 &&
            sgr::set_kernel_smem_attrs(reinterpret_cast<const void*>(simt_w8_fn(mt, v))) != cudaSuccess)
          ok = SGR_ERR_DEVICE;
        if (ok == SGR_OK && mt <= kW4PassM && v == 1 &&
            sgr::set_kernel_smem_attrs(reinterpret_cast<const void*>(simt_w4_fn(mt, v))) != cudaSuccess)
          ok = SGR_ERR_DEVICE;
      }
    if (ok == SGR_OK && sgr::tc_init_device(sms, &st.ws) != cudaSuccess) ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && sgr::rows_init_device() != cudaSuccess) ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && sgr::tile_init_device(dev) != cudaSuccess) ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && sgr::pair_init_device(dev) != cudaSuccess) ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && sgr::w8_init_device() != cudaSuccess) ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && sgr::w8s_init_device() != cudaSuccess) ok = SGR_ERR_DEVICE;
    if (ok != SGR_OK) cudaGetLastError();
    st.sms = sms;
    st.err = errp;
    st.status = ok;
    if (prev != dev) cudaSetDevice(prev);
  });
  return st.status;
}

// The measured table entry for (N, K) that covers M: the first entry whose M
// is >= the call's M (entries are sorted by M), or nullptr.
const sgr::TableEntry* table_lookup(int M, int N, int K) {
  for (int i = 0; i < sgr::kTableSize; ++i) {
    const sgr::TableEntry& e = sgr::kTable[i];
    if (e.n == N && e.k == K && e.m >= M) return &e;
  }
  return nullptr;
}

// Library choice for a shape: the measured per-M table where it covers the
// shape; otherwise the row-slab tensor-core kernel up to 64 tokens (the SIMT
// kernel where the row slab does not fit), and the tile GEMM beyond.
int select_path(int M, int N, int K, int sms) {
  if (const sgr::TableEntry* e = table_lookup(M, N, K)) {
    if (e->path == SGR_PATH_SIMT && M <= 16 && simt_vpt(K) > 0) return SGR_PATH_SIMT;
    if (e->path == SGR_PATH_TC_ROWS && sgr::rows_supported(sms, M, N, K)) return SGR_PATH_TC_ROWS;
    if (e->path == SGR_PATH_TC && sgr::tc_supported(M, N, K)) return SGR_PATH_TC;
    if (e->path == SGR_PATH_TILE && sgr::tile_supported(M, N, K)) return SGR_PATH_TILE;
    if (e->path == SGR_PATH_PAIR && sgr::pair_supported(M, N, K) && sms >= 2) return SGR_PATH_PAIR;
  }
  if (M <= 64 && sgr::rows_supported(sms, M, N, K)) return SGR_PATH_TC_ROWS;
  if (M <= 2 && simt_vpt(K) > 0) return SGR_PATH_SIMT;
  if (sgr::tile_supported(M, N, K)) return SGR_PATH_TILE;
  if (sgr::tc_supported(M, N, K)) return SGR_PATH_TC;
  if (M <= 16 && simt_vpt(K) > 0) return SGR_PATH_SIMT;
  return -SGR_ERR_UNSUPPORTED;
}

void default_simt_config(int sms, int M, int K, sgr_config* c) {
  (void)sms;
  (void)M;
  c->path = SGR_PATH_SIMT;
  c->ctas_per_sm = 1;
  const int row_bytes = K * 2;
  c->rows_per_stage = row_bytes >= 16384 ? 1 : (16384 / row_bytes > 64 ? 64 : 16384 / row_bytes);
  const size_t stage = (size_t)c->rows_per_stage * row_bytes;
  const size_t budget = 200 * 1024 - sgr::simt_ring_offset(16);
  int s = (int)(budget / stage);
  c->stages = s > 16 ? 16 : (s < 2 ? 2 : s);
  c->k_blocks_per_stage = 0;
  c->token_tile = 0;
}

// The current device, or -1 when none is current.
int current_device_or_none() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  return dev;
}

// 2-CTA clusters available to the pair kernel on the current device (SMs / 2
// when no device is current or none was queried).
int pair_pairs(int dev_sms) {
  return sgr::pair_grid_pairs(dev_sms > 0 ? dev_sms : 2, current_device_or_none());
}

int resolve_config(int dev_sms, int M, int N, int K, const sgr_config* in, sgr_config* out) {
  std::memset(out, 0, sizeof *out);
  int path = in ? in->path : SGR_PATH_AUTO;
  const bool automatic = (path == SGR_PATH_AUTO);
  if (automatic) {
    path = select_path(M, N, K, dev_sms);
    if (path < 0) return -path;
  }
  if (path == SGR_PATH_SIMT) {
    if (M > 16 || simt_vpt(K) == 0) return SGR_ERR_UNSUPPORTED;
    default_simt_config(dev_sms, M, K, out);
  } else if (path == SGR_PATH_TC) {
    if (!sgr::tc_supported(M, N, K)) return SGR_ERR_UNSUPPORTED;
    sgr::tc_default_config(dev_sms, M, N, K, out);
  } else if (path == SGR_PATH_TC_ROWS) {
    if (!sgr::rows_supported(dev_sms, M, N, K)) return SGR_ERR_UNSUPPORTED;
    sgr::rows_default_config(dev_sms, M, N, K, out);
  } else if (path == SGR_PATH_TILE) {
    if (!sgr::tile_supported(M, N, K)) return SGR_ERR_UNSUPPORTED;
    sgr::tile_default_config(dev_sms > 0 ? dev_sms : 1, M, N, K, out);
  } else if (path == SGR_PATH_PAIR) {
    if (!sgr::pair_supported(M, N, K)) return SGR_ERR_UNSUPPORTED;
    sgr::pair_default_config(pair_pairs(dev_sms), M, N, K, out);
  } else {
    return SGR_ERR_UNSUPPORTED;
  }
  if (automatic) {  // measured configuration for this shape, if the table has one
    const sgr::TableEntry* e = table_lookup(M, N, K);
    if (e && e->path == path) {
      out->ctas_per_sm = e->ctas_per_sm;
      out->stages = e->stages;
      if (path == SGR_PATH_SIMT || path == SGR_PATH_TC_ROWS) out->rows_per_stage = e->rows_per_stage;
      const bool tiled = path == SGR_PATH_TILE || path == SGR_PATH_PAIR;
      if (path != SGR_PATH_SIMT && (!tiled || e->k_blocks_per_stage > 0))
        out->k_blocks_per_stage = e->k_blocks_per_stage;
      if (path == SGR_PATH_TC_ROWS || tiled) out->prefetch_stages = e->prefetch_stages;
      if (tiled && e->tile_n) out->tile_n = e->tile_n;
      if (path == SGR_PATH_TILE) out->k_split = e->k_split > 0 ? e->k_split : 1;
      if (path == SGR_PATH_TC_ROWS) out->k_split = e->k_split == 2 ? 2 : 0;  // as measured
    }
  }
  if (in) {
    for (int r : in->reserved)
      if (r != 0) return SGR_ERR_UNSUPPORTED;
    if (in->ctas_per_sm) out->ctas_per_sm = in->ctas_per_sm;
    if (in->rows_per_stage) out->rows_per_stage = in->rows_per_stage;
    if (in->stages) out->stages = in->stages;
    if (in->k_blocks_per_stage) out->k_blocks_per_stage = in->k_blocks_per_stage;
    if (in->token_tile) out->token_tile = in->token_tile;
    if (in->prefetch_stages) out->prefetch_stages = in->prefetch_stages;
    if (in->tile_n) out->tile_n = in->tile_n;
    // A chosen tile width runs unsplit unless the split is asked for too.
    if (in->k_split) out->k_split = in->k_split;
    else if (path == SGR_PATH_TILE && in->tile_n) out->k_split = 1;
    // A tile width chosen without a ring depth gets the deepest ring that fits it.
    if (path == SGR_PATH_TILE && (in->tile_n || in->k_blocks_per_stage) && !in->stages)
      out->stages = sgr::tile_default_stages(out->tile_n, out->k_blocks_per_stage > 0 ? out->k_blocks_per_stage : 1);
    if (path == SGR_PATH_PAIR && (in->tile_n || in->k_blocks_per_stage) && !in->stages)
      out->stages = sgr::pair_default_stages(out->tile_n, out->k_blocks_per_stage > 0 ? out->k_blocks_per_stage : 1);
  }
  if (out->ctas_per_sm < 1 || out->ctas_per_sm > 8 || out->stages < 1 || out->stages > 64)
    return SGR_ERR_UNSUPPORTED;
  if (path == SGR_PATH_TC) {
    sgr::TcParams tp;
    int grid = 0;
    size_t smem = 0;
    int rc = sgr::tc_plan(*out, dev_sms > 0 ? dev_sms : 1, M, N, K, &tp, &grid, &smem);
    if (rc != SGR_OK) return rc;
  }
  if (path == SGR_PATH_TC_ROWS) {
    sgr::RowsParams rp;
    int grid = 0;
    size_t smem = 0;
    int rc = sgr::rows_plan(*out, dev_sms > 0 ? dev_sms : 1, M, N, K, &rp, &grid, &smem);
    if (rc != SGR_OK) return rc;
  }
  if (path == SGR_PATH_TILE) {
    sgr::TileParams gp;
    int grid = 0;
    size_t smem = 0;
    int rc = sgr::tile_plan(*out, dev_sms > 0 ? dev_sms : 1, M, N, K, &gp, &grid, &smem, current_device_or_none());
    if (rc != SGR_OK) return rc;
  }
  if (path == SGR_PATH_PAIR) {
    sgr::PairParams pp;
    int grid = 0;
    size_t smem = 0;
    int rc = sgr::pair_plan(*out, pair_pairs(dev_sms), M, N, K, &pp, &grid, &smem);
    if (rc != SGR_OK) return rc;
  }
  if (path == SGR_PATH_SIMT) {
    if (out->rows_per_stage < 1 || out->rows_per_stage > 64) return SGR_ERR_UNSUPPORTED;
    if (sgr::simt_smem_bytes(out->stages, out->rows_per_stage, K) > (size_t)kMaxDynSmem)
      return SGR_ERR_UNSUPPORTED;
    if ((size_t)out->rows_per_stage * K * 2 >= (1u << 31)) return SGR_ERR_UNSUPPORTED;
  }
  return SGR_OK;
}

int launch_simt(const sgr_config& c, int sms, unsigned* err, const void* A, long long lda,
                const void* W, const void* R, long long ldr, void* Y, long long ldy, int M, int N,
                int K, unsigned flags, cudaStream_t stream) {
  SimtFn fn = simt_fn(simt_mt(M), simt_vpt(K));
  if (!fn) return SGR_ERR_UNSUPPORTED;
  sgr::SimtParams p;
  p.A = static_cast<const __nv_bfloat16*>(A);
  p.W = static_cast<const __nv_bfloat16*>(W);
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.lda = lda;
  p.ldr = ldr;
  p.ldy = ldy;
  p.M = M;
  p.N = N;
  p.K = K;
  p.rows_per_stage = c.rows_per_stage;
  p.stages = c.stages;
  p.err = err;
  long long grid = (long long)sms * c.ctas_per_sm;
  if (grid > N) grid = N;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(sgr::kSimtThreads, 1, 1);
  lc.dynamicSmemBytes = sgr::simt_smem_bytes(c.stages, c.rows_per_stage, K);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (flags & SGR_FLAG_NO_PDL) ? 0 : 1;
  if (cudaLaunchKernelEx(&lc, fn, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

int launch_simt_w8(const sgr_config& c, int sms, unsigned* err, const void* A, long long lda, const void* Wq,
                   const float* scale, const void* R, long long ldr, void* Y, long long ldy, int M, int N, int K,
                   unsigned flags, cudaStream_t stream) {
  SimtFn fn = simt_w8_fn(simt_mt(M), simt_w8_vpt(K));
  if (!fn) return SGR_ERR_UNSUPPORTED;
  sgr::SimtParams p;
  std::memset(&p, 0, sizeof p);
  p.A = static_cast<const __nv_bfloat16*>(A);
  p.Wq = static_cast<const uint8_t*>(Wq);
  p.scale = scale;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.lda = lda;
  p.ldr = ldr;
  p.ldy = ldy;
  p.M = M;
  p.N = N;
  p.K = K;
  p.rows_per_stage = c.rows_per_stage;
  p.stages = c.stages;
  p.err = err;
  long long grid = (long long)sms * c.ctas_per_sm;
  if (grid > N) grid = N;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(sgr::kSimtThreads, 1, 1);
  lc.dynamicSmemBytes = sgr::simt_smem_bytes(c.stages, c.rows_per_stage, K, 1);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (flags & SGR_FLAG_NO_PDL) ? 0 : 1;
  if (cudaLaunchKernelEx(&lc, fn, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

int run(const void* A, long long lda, const void* W, const void* R, long long ldr, void* Y,
        long long ldy, int M, int N, int K, const sgr_config* cfg, unsigned flags,
        void* stream_ptr) {
  int rc = validate(A, lda, W, R, ldr, Y, ldy, M, N, K);
  if (rc != SGR_OK) return rc;
  if (M == 0 || N == 0) return SGR_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (K == 0) {  // empty sum: Y = R
    if (Y == R) return SGR_OK;
    if (cudaMemcpy2DAsync(Y, (size_t)ldy * 2, R, (size_t)ldr * 2, (size_t)N * 2, (size_t)M,
                          cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_LAUNCH;
    }
    return SGR_OK;
  }
  int dev;
  if ((rc = current_device(&dev)) != SGR_OK) return rc;
  if ((rc = init_device(dev)) != SGR_OK) return rc;
  DeviceState& st = g_dev[dev];
  sgr_config c;
  if ((rc = resolve_config(st.sms, M, N, K, cfg, &c)) != SGR_OK) return rc;
  if (c.path == SGR_PATH_SIMT)
    return launch_simt(c, st.sms, st.err, A, lda, W, R, ldr, Y, ldy, M, N, K, flags, stream);
  if (c.path == SGR_PATH_TC_ROWS)
    return sgr::rows_launch(c, st.sms, st.err, A, lda, W, R, ldr, Y, ldy, M, N, K,
                            (flags & SGR_FLAG_NO_PDL) == 0, stream);
  if (c.path == SGR_PATH_TILE)
    return sgr::tile_launch(c, st.sms, dev, st.err, A, lda, W, R, ldr, Y, ldy, M, N, K,
                            (flags & SGR_FLAG_NO_PDL) == 0, stream);
  if (c.path == SGR_PATH_PAIR)
    return sgr::pair_launch(c, sgr::pair_grid_pairs(st.sms, dev), st.err, A, lda, W, R, ldr, Y, ldy, M, N, K,
                            (flags & SGR_FLAG_NO_PDL) == 0, stream);
  return sgr::tc_launch(c, st.sms, st.err, &st.ws, A, lda, W, R, ldr, Y, ldy, M, N, K,
                        (flags & SGR_FLAG_NO_PDL) == 0, stream);
}

// ------------------------------------------------------------ no-allocation variant
// Scratch for skinny_gemm_residual_noalloc: split-K tile counters followed by
// FP32 partial tiles, in one file-scope device array.  Every GPU that loads
// this library holds it (4 MiB + 16 KiB) until the process exits.  Host code
// must not use the symbol itself as a pointer: it is a host-side stand-in, and
// the device address comes from cudaGetSymbolAddress (once per device).
constexpr int kNoallocCounters = 4096;              // W tiles x token tiles
constexpr size_t kNoallocPartialFloats = 1u << 20;  // 4 MiB of FP32 partials
constexpr size_t kNoallocBytes = kNoallocCounters * sizeof(unsigned) + kNoallocPartialFloats * sizeof(float);
static __device__ __align__(256) unsigned char g_sgr_noalloc_scratch[kNoallocBytes];

struct NoallocState {
  std::once_flag once;
  int status = SGR_ERR_DEVICE;
  int sms = 0;
  unsigned char* scratch = nullptr;  // device address of g_sgr_noalloc_scratch
  unsigned* err = nullptr;           // device address of g_sgr_error_word
};
NoallocState g_noalloc[kMaxDevices];

// One-time set-up for the current device (which must be `dev`): resolve the
// device addresses of the scratch array and of the error word, and set the
// kernel's shared-memory attributes.  Allocates nothing.
int noalloc_setup(int dev) {
  NoallocState& st = g_noalloc[dev];
  std::call_once(st.once, [&] {
    int ok = SGR_OK;
    int sms = 0;
    void* scratch = nullptr;
    unsigned* errp = nullptr;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && cudaGetSymbolAddress(&scratch, g_sgr_noalloc_scratch) != cudaSuccess)
      ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK && error_word(dev, &errp) != SGR_OK) ok = SGR_ERR_DEVICE;
    if (ok == SGR_OK &&
        sgr::set_kernel_smem_attrs(reinterpret_cast<const void*>(sgr::tc_skinny_kernel)) != cudaSuccess)
      ok = SGR_ERR_DEVICE;
    if (ok != SGR_OK) cudaGetLastError();
    st.sms = sms;
    st.scratch = static_cast<unsigned char*>(scratch);
    st.err = errp;
    st.status = ok;
  });
  return st.status;
}

int run_noalloc(const void* A, long long lda, const void* W, const void* R, long long ldr, void* Y,
                long long ldy, int M, int N, int K, unsigned flags, void* stream_ptr) {
  int rc = validate(A, lda, W, R, ldr, Y, ldy, M, N, K);
  if (rc != SGR_OK) return rc;
  if (M == 0 || N == 0) return SGR_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (K == 0) {  // empty sum: Y = R
    if (Y == R) return SGR_OK;
    if (cudaMemcpy2DAsync(Y, (size_t)ldy * 2, R, (size_t)ldr * 2, (size_t)N * 2, (size_t)M,
                          cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_LAUNCH;
    }
    return SGR_OK;
  }
  if (!sgr::tc_supported(M, N, K)) return SGR_ERR_UNSUPPORTED;
  int dev;
  if ((rc = current_device(&dev)) != SGR_OK) return rc;
  if ((rc = noalloc_setup(dev)) != SGR_OK) return rc;
  NoallocState& st = g_noalloc[dev];
  sgr_config c;
  std::memset(&c, 0, sizeof c);
  sgr::tc_default_config(st.sms, M, N, K, &c);
  sgr::TcParams plan;
  int grid = 0;
  size_t smem = 0;
  if ((rc = sgr::tc_plan(c, st.sms, M, N, K, &plan, &grid, &smem)) != SGR_OK) return rc;
  const long long tiles = (long long)((N + sgr::kTcTileRows - 1) / sgr::kTcTileRows) * plan.m_tiles;
  const size_t partials = (size_t)grid * 2 * plan.NT * sgr::kTcTileRows;
  if (tiles > kNoallocCounters || partials > kNoallocPartialFloats) return SGR_ERR_UNSUPPORTED;
  sgr::TcWorkspace ws;
  ws.counters = reinterpret_cast<unsigned*>(st.scratch);
  ws.counter_count = kNoallocCounters;
  ws.partials = reinterpret_cast<float*>(st.scratch + kNoallocCounters * sizeof(unsigned));
  ws.partial_floats = kNoallocPartialFloats;
  // The array keeps the previous call's contents: counters must start at zero.
  if (cudaMemsetAsync(ws.counters, 0, (size_t)tiles * sizeof(unsigned), stream) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return sgr::tc_launch(c, st.sms, st.err, &ws, A, lda, W, R, ldr, Y, ldy, M, N, K,
                        (flags & SGR_FLAG_NO_PDL) == 0, stream);
}

// ------------------------------------------------------------ FP8 weights
// Argument rules of skinny_gemm_residual_w8: those of the BF16 entry points
// for A, R and Y; Wq is [N, K] bytes with row stride ldw (>= K, a multiple of
// 16, 16-byte aligned base); scale holds N floats (4-byte aligned).
int validate_w8(const void* A, long long lda, const void* Wq, long long ldw, const float* scale, const void* R,
                long long ldr, const void* Y, long long ldy, int M, int N, int K) {
  if (M < 0 || N < 0 || K < 0) return SGR_ERR_SHAPE;
  if (M == 0 || N == 0) return SGR_OK;
  if (M > kMaxM || N > kMaxN || K > kMaxK) return SGR_ERR_UNSUPPORTED;
  if (N % 8 != 0 || K % 8 != 0) return SGR_ERR_SHAPE;
  if (!R || !Y) return SGR_ERR_NULL;
  if (K > 0 && (!A || !Wq || !scale)) return SGR_ERR_NULL;
  if (ldr < N || ldy < N) return SGR_ERR_SHAPE;
  if (K > 0 && (lda < K || ldw < K)) return SGR_ERR_SHAPE;
  if (ldr > kMaxLd || ldy > kMaxLd || (K > 0 && (lda > kMaxLd || ldw > kMaxLd))) return SGR_ERR_UNSUPPORTED;
  if (ldr % 8 != 0 || ldy % 8 != 0 || (K > 0 && (lda % 8 != 0 || ldw % 16 != 0))) return SGR_ERR_ALIGN;
  if (!aligned16(R) || !aligned16(Y)) return SGR_ERR_ALIGN;
  if (K > 0 && (!aligned16(A) || !aligned16(Wq) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0))
    return SGR_ERR_ALIGN;
  const Extent ey = extent(Y, M, ldy, N);
  if (K > 0) {
    if (overlap(ey, extent(A, M, lda, K))) return SGR_ERR_ALIAS;
    const uintptr_t wb = reinterpret_cast<uintptr_t>(Wq);
    if (overlap(ey, Extent{wb, wb + static_cast<uintptr_t>((long long)(N - 1) * ldw + K)})) return SGR_ERR_ALIAS;
    const uintptr_t sb = reinterpret_cast<uintptr_t>(scale);
    if (overlap(ey, Extent{sb, sb + static_cast<uintptr_t>(N) * 4u})) return SGR_ERR_ALIAS;
  }
  const bool in_place = (Y == R) && (ldy == ldr);
  if (!in_place && overlap(ey, extent(R, M, ldr, N))) return SGR_ERR_ALIAS;
  return SGR_OK;
}

// The CUDA-core FP8 kernel runs M <= 8 with contiguous code rows (one bulk
// copy per ring stage) and K a multiple of 16.
bool simt_w8_supported(int M, int K, long long ldw) {
  return M >= 1 && M <= 8 && ldw == K && simt_w8_vpt(K) > 0;
}

// The library chooses the CUDA-core kernel up to this many tokens (measured
// at N = 7168, K = 3584: 10.7 us at M = 1 for both kernels, 11.5 against
// 10.8 us at M = 2, the tensor-core kernel ahead from there on).
constexpr int kW8SimtMaxM = 1;

// The FP8 tensor-core path with split activations up to this many tokens
// (measured at N = 7168, K = 3584, graph of 8 calls over distinct code
// copies: 8.2-8.7 us at M = 1-4 and 9.8-10.0 us at M = 5-8 against 10.8 us
// for the widening kernel; the widening kernel ahead at M = 12-16, 10.9-11.0
// against 11.9-12.2 us, where converting all of A in every CTA costs more
// than it saves).
constexpr int kW8sAutoMaxM = 8;

// CUDA-core FP8 configuration: ring stages of two code rows, 4 stages,
// CTAs per SM by token count (the register footprint grows with M).
void default_simt_w8_config(int M, sgr_config* c) {
  std::memset(c, 0, sizeof *c);
  c->path = SGR_PATH_SIMT;
  c->ctas_per_sm = M <= 2 ? 3 : (M <= 4 ? 2 : 1);
  c->rows_per_stage = 2;
  c->stages = 4;
}

// Configuration of the FP8-weight kernels: the library default for this
// shape, then any non-zero field of `in` (path AUTO, W8 or SIMT).
int resolve_config_w8(int sms, int M, int N, int K, long long ldw, const sgr_config* in, sgr_config* out) {
  int path = in ? in->path : SGR_PATH_AUTO;
  if (path == SGR_PATH_AUTO) {
    if (M <= kW8sAutoMaxM && sgr::w8s_supported(sms, M, N, K, ldw))
      path = SGR_PATH_W8S;
    else
      path = (M <= kW8SimtMaxM && simt_w8_supported(M, K, ldw)) ? SGR_PATH_SIMT : SGR_PATH_W8;
  }
  if (path == SGR_PATH_SIMT) {
    if (!simt_w8_supported(M, K, ldw)) return SGR_ERR_UNSUPPORTED;
    default_simt_w8_config(M, out);
    if (in) {
      for (int r : in->reserved)
        if (r != 0) return SGR_ERR_UNSUPPORTED;
      if (in->tile_n || in->k_split || in->k_blocks_per_stage || in->token_tile ||
          in->prefetch_stages)
        return SGR_ERR_UNSUPPORTED;
      if (in->ctas_per_sm) out->ctas_per_sm = in->ctas_per_sm;
      if (in->rows_per_stage) out->rows_per_stage = in->rows_per_stage;
      if (in->stages) out->stages = in->stages;
    }
    if (out->ctas_per_sm < 1 || out->ctas_per_sm > 8 || out->stages < 2 || out->stages > 16) return SGR_ERR_UNSUPPORTED;
    if (out->rows_per_stage < 1 || out->rows_per_stage > 64) return SGR_ERR_UNSUPPORTED;
    if (sgr::simt_smem_bytes(out->stages, out->rows_per_stage, K, 1) > (size_t)kMaxDynSmem)
      return SGR_ERR_UNSUPPORTED;
    return SGR_OK;
  }
  if (path == SGR_PATH_W8S) {
    if (!sgr::w8s_supported(sms, M, N, K, ldw)) return SGR_ERR_UNSUPPORTED;
    sgr::w8s_default_config(sms, M, N, K, out);
    if (in) {
      for (int r : in->reserved)
        if (r != 0) return SGR_ERR_UNSUPPORTED;
      if (in->tile_n || in->k_split || in->prefetch_stages) return SGR_ERR_UNSUPPORTED;
      if (in->ctas_per_sm) out->ctas_per_sm = in->ctas_per_sm;
      if (in->rows_per_stage) out->rows_per_stage = in->rows_per_stage;
      if (in->stages) out->stages = in->stages;
      if (in->k_blocks_per_stage) out->k_blocks_per_stage = in->k_blocks_per_stage;
      if (in->token_tile) out->token_tile = in->token_tile;
    }
    out->path = SGR_PATH_W8S;
    sgr::W8sParams p;
    int grid = 0;
    size_t smem = 0;
    return sgr::w8s_plan(*out, sms, M, N, K, ldw, &p, &grid, &smem);
  }
  if (path != SGR_PATH_W8) return SGR_ERR_UNSUPPORTED;
  if (!sgr::w8_supported(sms, M, N, K)) return SGR_ERR_UNSUPPORTED;
  sgr::w8_default_config(sms, M, N, K, out);
  if (in) {
    for (int r : in->reserved)
      if (r != 0) return SGR_ERR_UNSUPPORTED;
    if (in->tile_n || in->k_split) return SGR_ERR_UNSUPPORTED;
    if (in->ctas_per_sm) out->ctas_per_sm = in->ctas_per_sm;
    if (in->rows_per_stage) out->rows_per_stage = in->rows_per_stage;
    if (in->stages) out->stages = in->stages;
    if (in->k_blocks_per_stage) out->k_blocks_per_stage = in->k_blocks_per_stage;
    if (in->token_tile) out->token_tile = in->token_tile;
    if (in->prefetch_stages) out->prefetch_stages = in->prefetch_stages;
  }
  out->path = SGR_PATH_W8;
  sgr::W8Params p;
  int grid = 0;
  size_t smem = 0;
  return sgr::w8_plan(*out, sms, M, N, K, &p, &grid, &smem);
}

int run_w8(const void* A, long long lda, const void* Wq, long long ldw, const float* scale, const void* R,
           long long ldr, void* Y, long long ldy, int M, int N, int K, const sgr_config* cfg, unsigned flags,
           void* stream_ptr) {
  int rc = validate_w8(A, lda, Wq, ldw, scale, R, ldr, Y, ldy, M, N, K);
  if (rc != SGR_OK) return rc;
  if (M == 0 || N == 0) return SGR_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (K == 0) {  // empty sum: Y = R
    if (Y == R) return SGR_OK;
    if (cudaMemcpy2DAsync(Y, (size_t)ldy * 2, R, (size_t)ldr * 2, (size_t)N * 2, (size_t)M,
                          cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_LAUNCH;
    }
    return SGR_OK;
  }
  int dev;
  if ((rc = current_device(&dev)) != SGR_OK) return rc;
  if ((rc = init_device(dev)) != SGR_OK) return rc;
  DeviceState& st = g_dev[dev];
  sgr_config c;
  if ((rc = resolve_config_w8(st.sms, M, N, K, ldw, cfg, &c)) != SGR_OK) return rc;
  if (c.path == SGR_PATH_SIMT)
    return launch_simt_w8(c, st.sms, st.err, A, lda, Wq, scale, R, ldr, Y, ldy, M, N, K, flags, stream);
  if (c.path == SGR_PATH_W8S)
    return sgr::w8s_launch(c, st.sms, st.err, A, lda, Wq, ldw, scale, R, ldr, Y, ldy, M, N, K,
                           (flags & SGR_FLAG_NO_PDL) == 0, stream);
  return sgr::w8_launch(c, st.sms, st.err, A, lda, Wq, ldw, scale, R, ldr, Y, ldy, M, N, K,
                        (flags & SGR_FLAG_NO_PDL) == 0, stream);
}

// ------------------------------------------------------------ NVFP4 weights
// Argument rules of skinny_gemm_residual_w4: those of the BF16 entry points
// for A, R and Y; K a multiple of 32; Wq4 is [N, K/2] bytes with row stride
// ldw (>= K/2, a multiple of 16, 16-byte aligned base); bs is
// [N, ceil(K/16)] E4M3 block scales with row stride ldbs (a multiple of 16,
// >= ceil(K/16) rounded up to 16: every row is read in 16-byte units,
// padding included, so the buffer holds N rows of ldbs bytes or at least
// (N - 1) ldbs + that many), 16-byte aligned base.
long long w4_scale_row_bytes(int K) { return sgr::simt_w4_scale_bytes(K); }

int validate_w4(const void* A, long long lda, const void* Wq4, long long ldw, const void* bs, long long ldbs,
                const void* R, long long ldr, const void* Y, long long ldy, int M, int N, int K) {
  if (M < 0 || N < 0 || K < 0) return SGR_ERR_SHAPE;
  if (M == 0 || N == 0) return SGR_OK;
  if (M > kMaxM || N > kMaxN || K > kMaxK) return SGR_ERR_UNSUPPORTED;
  if (N % 8 != 0 || K % 8 != 0) return SGR_ERR_SHAPE;
  if (!R || !Y) return SGR_ERR_NULL;
  if (K > 0 && (!A || !Wq4 || !bs)) return SGR_ERR_NULL;
  if (ldr < N || ldy < N) return SGR_ERR_SHAPE;
  if (K > 0 && (lda < K || ldw < K / 2 || ldbs < w4_scale_row_bytes(K))) return SGR_ERR_SHAPE;
  if (ldr > kMaxLd || ldy > kMaxLd || (K > 0 && (lda > kMaxLd || ldw > kMaxLd || ldbs > kMaxLd)))
    return SGR_ERR_UNSUPPORTED;
  if (ldr % 8 != 0 || ldy % 8 != 0 || (K > 0 && (lda % 8 != 0 || ldw % 16 != 0 || ldbs % 16 != 0)))
    return SGR_ERR_ALIGN;
  if (!aligned16(R) || !aligned16(Y)) return SGR_ERR_ALIGN;
  if (K > 0 && (!aligned16(A) || !aligned16(Wq4) || !aligned16(bs))) return SGR_ERR_ALIGN;
  const Extent ey = extent(Y, M, ldy, N);
  if (K > 0) {
    if (overlap(ey, extent(A, M, lda, K))) return SGR_ERR_ALIAS;
    const uintptr_t wb = reinterpret_cast<uintptr_t>(Wq4);
    if (overlap(ey, Extent{wb, wb + static_cast<uintptr_t>((long long)(N - 1) * ldw + K / 2)})) return SGR_ERR_ALIAS;
    const uintptr_t sb = reinterpret_cast<uintptr_t>(bs);
    if (overlap(ey, Extent{sb, sb + static_cast<uintptr_t>((long long)(N - 1) * ldbs + w4_scale_row_bytes(K))}))
      return SGR_ERR_ALIAS;
  }
  const bool in_place = (Y == R) && (ldy == ldr);
  if (!in_place && overlap(ey, extent(R, M, ldr, N))) return SGR_ERR_ALIAS;
  return SGR_OK;
}

// CUDA-core NVFP4 configuration, the fastest measured at N = 7168, K = 3584
// (graph of 8 calls over distinct weight copies): ring stages of four
// records; two CTAs per SM with two stages for 1-2 tokens (10.5 / 12.1 us),
// one CTA with eight stages for 3-4 tokens (23.7 us), where the FMAs and the
// conversions, not the bytes, set the pace.
void default_simt_w4_config(int M, sgr_config* c) {
  std::memset(c, 0, sizeof *c);
  c->path = SGR_PATH_SIMT;
  c->ctas_per_sm = M <= 2 ? 2 : 1;
  c->rows_per_stage = 4;
  c->stages = M <= 2 ? 2 : 8;
}

size_t simt_w4_smem_bytes(int stages, int rows_per_stage, int K) {
  return sgr::simt_ring_offset(stages) + (size_t)stages * rows_per_stage * sgr::simt_w4_record_bytes(K);
}

// The library takes the CUDA-core kernel up to this many tokens where it can
// run (K a multiple of 32, at most 7168), the tensor-core widening kernel
// otherwise (measured at N = 7168, K = 3584, graph of 8 calls: 10.5 against
// 11.1 us at M = 1; 12.1 against 11.2 at M = 2; the tensor-core kernel flat
// at 11.1-11.5 us up to M = 16, the CUDA-core one 23.7 / 46.7 / 92.9 us at
// M = 4 / 8 / 16).
constexpr int kW4SimtMaxM = 1;
// Tokens per launch of the tensor-core NVFP4 kernel: its activation ring of
// two 4-block stages holds at most 128 token rows in shared memory.
constexpr int kW4TcPassM = 128;

// The path of an NVFP4 call, decided without a device: SGR_PATH_SIMT or
// SGR_PATH_W8 (the tensor-core widening kernel); 0 when refused.
int w4_path(int M, int K, const sgr_config* in) {
  int path = in ? in->path : SGR_PATH_AUTO;
  if (in) {
    for (int r : in->reserved)
      if (r != 0) return 0;
    if (in->tile_n || in->k_split) return 0;
  }
  if (path == SGR_PATH_AUTO) path = (M <= kW4SimtMaxM && simt_w4_vpt(K)) ? SGR_PATH_SIMT : SGR_PATH_W8;
  if (path == SGR_PATH_SIMT && !simt_w4_vpt(K)) return 0;
  return (path == SGR_PATH_SIMT || path == SGR_PATH_W8) ? path : 0;
}

int resolve_config_w4(int sms, int M, int N, int K, const sgr_config* in, sgr_config* out) {
  const int path = w4_path(M, K, in);
  if (!path) return SGR_ERR_UNSUPPORTED;
  if (path == SGR_PATH_SIMT) {
    default_simt_w4_config(M < kW4PassM ? M : kW4PassM, out);
    if (in) {
      if (in->k_blocks_per_stage || in->token_tile || in->prefetch_stages) return SGR_ERR_UNSUPPORTED;
      if (in->ctas_per_sm) out->ctas_per_sm = in->ctas_per_sm;
      if (in->rows_per_stage) out->rows_per_stage = in->rows_per_stage;
      if (in->stages) out->stages = in->stages;
    }
    if (out->ctas_per_sm < 1 || out->ctas_per_sm > 8 || out->stages < 2 || out->stages > 16) return SGR_ERR_UNSUPPORTED;
    if (out->rows_per_stage < 1 || out->rows_per_stage > 64) return SGR_ERR_UNSUPPORTED;
    if (simt_w4_smem_bytes(out->stages, out->rows_per_stage, K) > (size_t)kMaxDynSmem) return SGR_ERR_UNSUPPORTED;
    return SGR_OK;
  }
  M = M < kW4TcPassM ? M : kW4TcPassM;  // one pass
  if (!sgr::w8_supported(sms, M, N, K)) return SGR_ERR_UNSUPPORTED;
  sgr::w8_default_config(sms, M, N, K, out, true);
  if (in) {
    if (in->ctas_per_sm) out->ctas_per_sm = in->ctas_per_sm;
    if (in->rows_per_stage) out->rows_per_stage = in->rows_per_stage;
    if (in->stages) out->stages = in->stages;
    if (in->k_blocks_per_stage) out->k_blocks_per_stage = in->k_blocks_per_stage;
    if (in->token_tile) out->token_tile = in->token_tile;
    if (in->prefetch_stages) out->prefetch_stages = in->prefetch_stages;
  }
  sgr::W8Params p;
  int grid = 0;
  size_t smem = 0;
  return sgr::w8_plan(*out, sms, M, N, K, &p, &grid, &smem, true);
}

// One pass over at most kW4PassM token rows.
int launch_simt_w4(const sgr_config& c, int sms, unsigned* err, const void* A, long long lda, const void* Wq4,
                   long long ldw, const void* bs, long long ldbs, float gs, const void* R, long long ldr, void* Y,
                   long long ldy, int M, int N, int K, unsigned flags, cudaStream_t stream) {
  SimtFn fn = simt_w4_fn(simt_mt(M), simt_w4_vpt(K));
  if (!fn) return SGR_ERR_UNSUPPORTED;
  sgr::SimtParams p;
  std::memset(&p, 0, sizeof p);
  p.A = static_cast<const __nv_bfloat16*>(A);
  p.Wq = static_cast<const uint8_t*>(Wq4);
  p.bs = static_cast<const uint8_t*>(bs);
  p.ldw = ldw;
  p.ldbs = ldbs;
  p.gs = gs;
  p.R = static_cast<const __nv_bfloat16*>(R);
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.lda = lda;
  p.ldr = ldr;
  p.ldy = ldy;
  p.M = M;
  p.N = N;
  p.K = K;
  p.rows_per_stage = c.rows_per_stage;
  p.stages = c.stages;
  p.err = err;
  long long grid = (long long)sms * c.ctas_per_sm;
  if (grid > N) grid = N;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(sgr::kSimtThreads, 1, 1);
  lc.dynamicSmemBytes = simt_w4_smem_bytes(c.stages, c.rows_per_stage, K);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = (flags & SGR_FLAG_NO_PDL) ? 0 : 1;
  if (cudaLaunchKernelEx(&lc, fn, p) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_LAUNCH;
  }
  return SGR_OK;
}

constexpr int kW4MaxM = 256;  // decode-sized batches: at most 64 passes of 4 tokens

int run_w4(const void* A, long long lda, const void* Wq4, long long ldw, const void* bs, long long ldbs, float gs,
           const void* R, long long ldr, void* Y, long long ldy, int M, int N, int K, const sgr_config* cfg,
           unsigned flags, void* stream_ptr) {
  int rc = validate_w4(A, lda, Wq4, ldw, bs, ldbs, R, ldr, Y, ldy, M, N, K);
  if (rc != SGR_OK) return rc;
  if (M == 0 || N == 0) return SGR_OK;
  if (M > kW4MaxM) return SGR_ERR_UNSUPPORTED;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (K == 0) {  // empty sum: Y = R
    if (Y == R) return SGR_OK;
    if (cudaMemcpy2DAsync(Y, (size_t)ldy * 2, R, (size_t)ldr * 2, (size_t)N * 2, (size_t)M,
                          cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_LAUNCH;
    }
    return SGR_OK;
  }
  if (!w4_path(M, K, cfg)) return SGR_ERR_UNSUPPORTED;  // refused before any device work
  int dev;
  if ((rc = current_device(&dev)) != SGR_OK) return rc;
  if ((rc = init_device(dev)) != SGR_OK) return rc;
  DeviceState& st = g_dev[dev];
  sgr_config c;
  if ((rc = resolve_config_w4(st.sms, M, N, K, cfg, &c)) != SGR_OK) return rc;
  if (c.path == SGR_PATH_W8) {
    // Passes of at most kW4TcPassM token rows (one for M <= 128).
    for (int m0 = 0; m0 < M; m0 += kW4TcPassM) {
      const int mp = M - m0 < kW4TcPassM ? M - m0 : kW4TcPassM;
      sgr_config cp = c;
      if (mp < M && (!cfg || !cfg->token_tile)) cp.token_tile = (mp + 15) / 16 * 16;
      rc = sgr::w4_launch(cp, st.sms, st.err, static_cast<const __nv_bfloat16*>(A) + (size_t)m0 * lda, lda, Wq4,
                          ldw, bs, ldbs, gs, static_cast<const __nv_bfloat16*>(R) + (size_t)m0 * ldr, ldr,
                          static_cast<__nv_bfloat16*>(Y) + (size_t)m0 * ldy, ldy, mp, N, K,
                          (flags & SGR_FLAG_NO_PDL) == 0, stream);
      if (rc != SGR_OK) return rc;
    }
    return SGR_OK;
  }
  // Passes of at most kW4PassM token rows (each streams the weights again).
  for (int m0 = 0; m0 < M; m0 += kW4PassM) {
    const int mp = M - m0 < kW4PassM ? M - m0 : kW4PassM;
    rc = launch_simt_w4(c, st.sms, st.err, static_cast<const __nv_bfloat16*>(A) + (size_t)m0 * lda, lda, Wq4, ldw,
                        bs, ldbs, gs, static_cast<const __nv_bfloat16*>(R) + (size_t)m0 * ldr, ldr,
                        static_cast<__nv_bfloat16*>(Y) + (size_t)m0 * ldy, ldy, mp, N, K, flags, stream);
    if (rc != SGR_OK) return rc;
  }
  return SGR_OK;
}

// ------------------------------------------------------------ wait self-test
// One thread waits on an mbarrier that nothing arrives on, with a limit of
// `limit_ns` nanoseconds of %globaltimer instead of the kernels' one second,
// and reports the timeout through the device error word exactly as the
// kernels' waits do.  Exercises the failure path without faulting or hanging
// the GPU.
__global__ void sgr_selftest_wait_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ uint64_t bar;
  const uint32_t b = sgr::smem_u32(&bar);
  sgr::mbar_init(b, 1);
  sgr::fence_mbar_init();
  const uint64_t t0 = sgr::globaltimer_ns();
  bool done = false;
  while (!done && sgr::globaltimer_ns() - t0 <= limit_ns)
    for (int i = 0; i < 64 && !done; ++i) done = sgr::mbar_test_wait(b, 0);
  if (!done) sgr::report_error(err, sgr::kErrWaitFull);
}

int run_selftest_wait(unsigned limit_us, unsigned* code) {
  if (!code) return SGR_ERR_NULL;
  if (limit_us == 0 || limit_us > 100000) return SGR_ERR_UNSUPPORTED;
  int dev, rc;
  if ((rc = current_device(&dev)) != SGR_OK) return rc;
  if ((rc = init_device(dev)) != SGR_OK) return rc;
  DeviceState& st = g_dev[dev];
  unsigned zero = 0;
  if (cudaMemcpy(st.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  sgr_selftest_wait_kernel<<<1, 1>>>((unsigned long long)limit_us * 1000ull, st.err);
  if (cudaGetLastError() != cudaSuccess) return SGR_ERR_LAUNCH;
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(&v, st.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(st.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  *code = v;
  return SGR_OK;
}

// ------------------------------------------------------------ stream-K abort self-test
// One stream-K launch (the library's workspace, contiguous operands) in which
// CTA `cta` acts as if its first accumulator wait had run out: it records
// kErrWaitMma, raises its abort flag (its producer and MMA threads stop at
// their next wait and drain) and arrives on the split-K counters of its
// remaining segments without contributing a partial.  Exercises the abort
// path of the kernel without faulting or hanging anything.
int run_selftest_streamk_abort(const void* A, const void* W, const void* R, void* Y, int M, int N, int K, int cta,
                               unsigned* code) {
  if (!code) return SGR_ERR_NULL;
  if (M < 1 || N < 1 || K < 1) return SGR_ERR_SHAPE;
  int rc = validate(A, K, W, R, N, Y, N, M, N, K);
  if (rc != SGR_OK) return rc;
  if (cta < 0) return SGR_ERR_UNSUPPORTED;
  int dev;
  if ((rc = current_device(&dev)) != SGR_OK) return rc;
  if ((rc = init_device(dev)) != SGR_OK) return rc;
  DeviceState& st = g_dev[dev];
  sgr_config in = {};
  in.path = SGR_PATH_TC;
  sgr_config c;
  if ((rc = resolve_config(st.sms, M, N, K, &in, &c)) != SGR_OK) return rc;
  unsigned zero = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(st.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  rc = sgr::tc_launch(c, st.sms, st.err, &st.ws, A, K, W, R, N, Y, N, M, N, K, false, nullptr, cta);
  if (rc != SGR_OK) return rc;
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(&v, st.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(st.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  *code = v;
  return SGR_OK;
}

// ------------------------------------------------------------ grouped launch
int run_grouped(const sgr_group* groups, int num_groups, int N, int K, const sgr_config* cfg, unsigned flags,
                void* stream_ptr) {
  if (num_groups < 0) return SGR_ERR_UNSUPPORTED;
  if (num_groups > 0 && !groups) return SGR_ERR_NULL;
  if (cfg && cfg->path != SGR_PATH_AUTO && cfg->path != SGR_PATH_TC_ROWS) return SGR_ERR_UNSUPPORTED;
  int m_max = 0, active = 0;
  for (int i = 0; i < num_groups; ++i) {
    const sgr_group& g = groups[i];
    if (g.reserved != 0) return SGR_ERR_UNSUPPORTED;
    int rc = validate(g.A, g.lda, g.W, g.R, g.ldr, g.Y, g.ldy, g.M, N, K);
    if (rc != SGR_OK) return rc;
    if (g.M > sgr::kRowsMaxTokens) return SGR_ERR_UNSUPPORTED;
    if (g.M > 0) {
      ++active;
      m_max = g.M > m_max ? g.M : m_max;
    }
  }
  // No group's output may overlap another group's operands.
  for (int i = 0; i < num_groups; ++i) {
    const sgr_group& g = groups[i];
    if (g.M == 0 || N == 0) continue;
    const Extent ey = extent(g.Y, g.M, g.ldy, N);
    for (int j = 0; j < num_groups; ++j) {
      const sgr_group& h = groups[j];
      if (j == i || h.M == 0) continue;
      if (overlap(ey, extent(h.Y, h.M, h.ldy, N)) || overlap(ey, extent(h.R, h.M, h.ldr, N))) return SGR_ERR_ALIAS;
      if (K > 0 && (overlap(ey, extent(h.A, h.M, h.lda, K)) || overlap(ey, extent(h.W, N, K, K)))) return SGR_ERR_ALIAS;
    }
  }
  if (active == 0 || N == 0) return SGR_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (K == 0) {  // empty sums: Y = R per group
    for (int i = 0; i < num_groups; ++i) {
      const sgr_group& g = groups[i];
      if (g.M == 0 || g.Y == g.R) continue;
      if (cudaMemcpy2DAsync(g.Y, (size_t)g.ldy * 2, g.R, (size_t)g.ldr * 2, (size_t)N * 2, (size_t)g.M,
                            cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
        cudaGetLastError();
        return SGR_ERR_LAUNCH;
      }
    }
    return SGR_OK;
  }
  int dev, rc;
  if ((rc = current_device(&dev)) != SGR_OK) return rc;
  if ((rc = init_device(dev)) != SGR_OK) return rc;
  DeviceState& st = g_dev[dev];
  if (!sgr::rows_supported(st.sms, m_max, N, K)) return SGR_ERR_UNSUPPORTED;
  sgr_config in = {};
  if (cfg) in = *cfg;
  in.path = SGR_PATH_TC_ROWS;
  sgr_config c;
  if ((rc = resolve_config(st.sms, m_max, N, K, &in, &c)) != SGR_OK) return rc;
  // The default's K split where the grouped kernel has it (16-48-token tiles).
  if (in.k_split == 0 && c.token_tile > 48) c.k_split = 0;
  // Active groups in launches of up to 32.
  sgr::RowsGroupArgs batch[sgr::kRowsMaxGroups];
  int n = 0;
  for (int i = 0; i <= num_groups; ++i) {
    if (i < num_groups && groups[i].M > 0) {
      const sgr_group& g = groups[i];
      batch[n++] = sgr::RowsGroupArgs{g.A, g.lda, g.W, g.R, g.ldr, g.Y, g.ldy, g.M};
    }
    if (n == sgr::kRowsMaxGroups || (i == num_groups && n > 0)) {
      rc = sgr::rows_grouped_launch(c, st.sms, st.err, batch, n, N, K, (flags & SGR_FLAG_NO_PDL) == 0, stream);
      if (rc != SGR_OK) return rc;
      n = 0;
    }
  }
  return SGR_OK;
}

}  // namespace

extern "C" {

int skinny_gemm_residual(const void* A, const void* W, const void* R, void* Y, int M, int N,
                         int K, void* stream) {
  return run(A, K, W, R, N, Y, N, M, N, K, nullptr, 0u, stream);
}

int skinny_gemm_residual_ex(const void* A, int64_t lda, const void* W, const void* R,
                            int64_t ldr, void* Y, int64_t ldy, int M, int N, int K,
                            unsigned flags, void* stream) {
  return run(A, lda, W, R, ldr, Y, ldy, M, N, K, nullptr, flags, stream);
}

int skinny_gemm_residual_config(const void* A, int64_t lda, const void* W, const void* R,
                                int64_t ldr, void* Y, int64_t ldy, int M, int N, int K,
                                const sgr_config* cfg, unsigned flags, void* stream) {
  return run(A, lda, W, R, ldr, Y, ldy, M, N, K, cfg, flags, stream);
}

int sgr_validate(const void* A, int64_t lda, const void* W, const void* R, int64_t ldr,
                 const void* Y, int64_t ldy, int M, int N, int K) {
  return validate(A, lda, W, R, ldr, Y, ldy, M, N, K);
}

int sgr_select_path(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 8 || N % 8 || K % 8) return -SGR_ERR_SHAPE;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    sms = 152;  // no device visible: plan for a GB300 (152 SMs)
  }
  return select_path(M, N, K, sms);
}

int sgr_default_config(int device, int M, int N, int K, int path, sgr_config* cfg) {
  if (!cfg) return SGR_ERR_NULL;
  if (M < 1 || N < 8 || K < 8 || N % 8 || K % 8) return SGR_ERR_SHAPE;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  sgr_config in = {};
  in.path = path;
  if (path == SGR_PATH_W8 || path == SGR_PATH_W8S) return resolve_config_w8(sms, M, N, K, K, &in, cfg);
  return resolve_config(sms, M, N, K, &in, cfg);
}

int sgr_init(int device) { return init_device(device); }

int sgr_device_error(int device, unsigned* code, int clear) {
  if (!code) return SGR_ERR_NULL;
  unsigned* word = nullptr;
  int rc = error_word(device, &word);  // no workspace set-up: allocates nothing
  if (rc != SGR_OK) return rc;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess || (prev != device && cudaSetDevice(device) != cudaSuccess)) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  unsigned v = 0;
  cudaError_t e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(word, 0, sizeof v);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SGR_ERR_DEVICE;
  }
  *code = v;
  return SGR_OK;
}

int sgr_kernel_resources(int device, int path, int M, int N, int K, int* regs, int* local_bytes,
                         int* smem_bytes, int* threads) {
  if (!regs || !local_bytes || !smem_bytes || !threads) return SGR_ERR_NULL;
  sgr_config c;
  int rc = sgr_default_config(device, M, N, K, path, &c);
  if (rc != SGR_OK) return rc;
  cudaFuncAttributes fa;
  if (c.path == SGR_PATH_SIMT) {
    if (cudaFuncGetAttributes(&fa, simt_fn(simt_mt(M), simt_vpt(K))) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_DEVICE;
    }
    *smem_bytes = (int)sgr::simt_smem_bytes(c.stages, c.rows_per_stage, K);
    *threads = sgr::kSimtThreads;
  } else if (c.path == SGR_PATH_TC_ROWS) {
    sgr::RowsParams rp;
    int grid = 0;
    size_t smem = 0;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (sgr::rows_plan(c, sms, M, N, K, &rp, &grid, &smem) != SGR_OK) return SGR_ERR_UNSUPPORTED;
    const int mode = sgr::rows_epi_mode(rp.NT, rp.groups);
    const void* fn = sgr::rows_kernel_fn(mode, rp.ksplit == 2);
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_DEVICE;
    }
    *smem_bytes = (int)smem;
    *threads = sgr::rows_threads(mode);
  } else if (c.path == SGR_PATH_W8) {
    sgr::W8Params wp;
    int grid = 0;
    size_t smem = 0;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (sgr::w8_plan(c, sms, M, N, K, &wp, &grid, &smem) != SGR_OK) return SGR_ERR_UNSUPPORTED;
    if (cudaFuncGetAttributes(&fa, sgr::w8_decode_epi(wp) ? sgr::w8_rows_kernel<false, true>
                                                          : sgr::w8_rows_kernel<false, false>) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_DEVICE;
    }
    *smem_bytes = (int)smem;
    *threads = sgr::kW8Threads;
  } else if (c.path == SGR_PATH_W8S) {
    if (cudaFuncGetAttributes(&fa, sgr::w8s_in_regs(M, K) ? sgr::w8s_kernel<true> : sgr::w8s_kernel<false>) !=
        cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_DEVICE;
    }
    sgr::W8sParams wp;
    int grid = 0;
    size_t smem = 0;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (sgr::w8s_plan(c, sms, M, N, K, K, &wp, &grid, &smem) != SGR_OK) return SGR_ERR_UNSUPPORTED;
    *smem_bytes = (int)smem;
    *threads = sgr::kW8sThreads;
  } else if (c.path == SGR_PATH_PAIR) {
    if (cudaFuncGetAttributes(&fa, sgr::pair_kernel_for(c.tile_n)) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_DEVICE;
    }
    *smem_bytes = (int)sgr::pair_smem_bytes(c.stages, c.tile_n, c.k_blocks_per_stage > 0 ? c.k_blocks_per_stage : 1);
    *threads = sgr::kPairThreads;
  } else if (c.path == SGR_PATH_TILE) {
    if (cudaFuncGetAttributes(&fa, sgr::tile_kernel_for(c.tile_n, sgr::tile_mode(c))) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_DEVICE;
    }
    *smem_bytes = (int)sgr::tile_smem_bytes(c.stages, c.tile_n, c.k_blocks_per_stage > 0 ? c.k_blocks_per_stage : 1);
    *threads = sgr::tile_threads(sgr::tile_mode(c));
  } else {
    int s = 0, t = 0;
    const void* fn = sgr::tc_kernel_for(M, N, K, &c, &s, &t);
    if (!fn || cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
      cudaGetLastError();
      return SGR_ERR_DEVICE;
    }
    *smem_bytes = s;
    *threads = t;
  }
  *regs = fa.numRegs;
  *local_bytes = (int)fa.localSizeBytes;
  return SGR_OK;
}

const char* sgr_status_string(int status) {
  switch (status) {
    case SGR_OK: return "ok";
    case SGR_ERR_NULL: return "a required pointer is NULL";
    case SGR_ERR_SHAPE: return "bad shape: negative size, N or K not a multiple of 8, or row stride below row width";
    case SGR_ERR_ALIGN: return "misaligned: pointers must be 16-byte aligned and row strides multiples of 8 elements";
    case SGR_ERR_ALIAS: return "Y overlaps A, W, or R (other than Y == R exactly)";
    case SGR_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case SGR_ERR_LAUNCH: return "CUDA launch failed";
    case SGR_ERR_DEVICE: return "no usable CUDA device or device set-up failed";
    default: return "unknown status";
  }
}

int sgr_abi_version(void) { return SGR_ABI_VERSION; }

int skinny_gemm_residual_grouped(const sgr_group* groups, int num_groups, int N, int K,
                                 const sgr_config* cfg, unsigned flags, void* stream) {
  return run_grouped(groups, num_groups, N, K, cfg, flags, stream);
}

int skinny_gemm_residual_noalloc(const void* A, int64_t lda, const void* W, const void* R,
                                 int64_t ldr, void* Y, int64_t ldy, int M, int N, int K,
                                 unsigned flags, void* stream) {
  return run_noalloc(A, lda, W, R, ldr, Y, ldy, M, N, K, flags, stream);
}

int skinny_gemm_residual_w8(const void* A, int64_t lda, const void* Wq, int64_t ldw, const float* scale,
                            const void* R, int64_t ldr, void* Y, int64_t ldy, int M, int N, int K,
                            const sgr_config* cfg, unsigned flags, void* stream) {
  return run_w8(A, lda, Wq, ldw, scale, R, ldr, Y, ldy, M, N, K, cfg, flags, stream);
}

int sgr_validate_w8(const void* A, int64_t lda, const void* Wq, int64_t ldw, const float* scale, const void* R,
                    int64_t ldr, const void* Y, int64_t ldy, int M, int N, int K) {
  return validate_w8(A, lda, Wq, ldw, scale, R, ldr, Y, ldy, M, N, K);
}

int skinny_gemm_residual_w4(const void* A, int64_t lda, const void* Wq4, int64_t ldw, const void* bs, int64_t ldbs,
                            float gs, const void* R, int64_t ldr, void* Y, int64_t ldy, int M, int N, int K,
                            const sgr_config* cfg, unsigned flags, void* stream) {
  return run_w4(A, lda, Wq4, ldw, bs, ldbs, gs, R, ldr, Y, ldy, M, N, K, cfg, flags, stream);
}

int sgr_validate_w4(const void* A, int64_t lda, const void* Wq4, int64_t ldw, const void* bs, int64_t ldbs,
                    const void* R, int64_t ldr, const void* Y, int64_t ldy, int M, int N, int K) {
  return validate_w4(A, lda, Wq4, ldw, bs, ldbs, R, ldr, Y, ldy, M, N, K);
}

int sgr_selftest_wait_timeout(unsigned limit_us, unsigned* code) { return run_selftest_wait(limit_us, code); }

int sgr_selftest_streamk_abort(const void* A, const void* W, const void* R, void* Y, int M, int N, int K, int cta,
                               unsigned* code) {
  return run_selftest_streamk_abort(A, W, R, Y, M, N, K, cta, code);
}

}  // extern "C"
