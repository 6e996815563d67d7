// sgr_tc.cuh -- tensor-core (tcgen05 / tensor memory) path.  Placeholder:
// reports every shape as unsupported until the kernel lands.
#pragma once

#include <cuda_runtime.h>

#include "skinny_gemm_residual.h"

namespace sgr {

struct TcWorkspace {
  float* partials = nullptr;
  unsigned* counters = nullptr;
  size_t partial_floats = 0;
  int counter_count = 0;
};

inline bool tc_supported(int, int, int) { return false; }
inline cudaError_t tc_init_device(int, TcWorkspace*) { return cudaSuccess; }
inline void tc_default_config(int, int, int, int, sgr_config* c) { c->path = SGR_PATH_TC; }
inline int tc_launch(const sgr_config&, int, unsigned*, TcWorkspace*, const void*, long long,
                     const void*, const void*, long long, void*, long long, int, int, int, bool,
                     cudaStream_t) {
  return SGR_ERR_UNSUPPORTED;
}
inline const void* tc_kernel_for(int, int, int, const sgr_config*, int*, int*) { return nullptr; }

}  // namespace sgr
