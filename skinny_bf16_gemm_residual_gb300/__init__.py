"""Skinny BF16 projection GEMM with a fused residual add, for GB300 (sm_103a).

    Y[M,N] = bf16( A[M,K] . W[N,K]^T  (FP32 accumulate)  +  R[M,N] )

and its low-bit weight variant (FP8 E4M3 codes Wq with a per-column scale):

    Y[M,N] = bf16( scale[N] * A[M,K] . e4m3(Wq[N,K])^T  +  R[M,N] )

The work runs in hand-written CUDA kernels behind the C ABI declared in
include/skinny_gemm_residual.h; this package is a ctypes binding with the
same function names (see ``binding``), the build step (``build``) and the
seeded synthetic input generators (``inputs``).  The library is loaded on
first use; there is no CPU fallback.
"""
from .binding import (  # noqa: F401
    ABI_VERSION,
    SGR_ERR_ALIAS,
    SGR_ERR_ALIGN,
    SGR_ERR_DEVICE,
    SGR_ERR_LAUNCH,
    SGR_ERR_NULL,
    SGR_ERR_SHAPE,
    SGR_ERR_UNSUPPORTED,
    SGR_FLAG_NO_PDL,
    SGR_OK,
    SGR_PATH_AUTO,
    SGR_PATH_SIMT,
    SGR_PATH_TC,
    SGR_PATH_TC_ROWS,
    SGR_PATH_TILE,
    SGR_PATH_W8,
    SGR_PATH_PAIR,
    SGR_PATH_W8S,
    SgrError,
    load,
    make_config,
    sgr_abi_version,
    sgr_config,
    sgr_default_config,
    sgr_device_error,
    sgr_init,
    sgr_kernel_resources,
    sgr_select_path,
    sgr_status_string,
    sgr_validate_ptr,
    skinny_gemm_residual,
    skinny_gemm_residual_config,
    skinny_gemm_residual_config_ptr,
    skinny_gemm_residual_ex,
    skinny_gemm_residual_ex_ptr,
    skinny_gemm_residual_noalloc,
    skinny_gemm_residual_grouped,
    skinny_gemm_residual_grouped_ptr,
    sgr_group,
    skinny_gemm_residual_noalloc_ptr,
    skinny_gemm_residual_ptr,
    skinny_gemm_residual_w8,
    skinny_gemm_residual_w8_ptr,
    sgr_validate_w8_ptr,
    skinny_gemm_residual_w4,
    skinny_gemm_residual_w4_ptr,
    sgr_validate_w4_ptr,
    sgr_selftest_wait_timeout,
    sgr_selftest_streamk_abort,
)
