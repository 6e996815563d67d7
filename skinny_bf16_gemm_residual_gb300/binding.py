"""ctypes binding of the C ABI in include/skinny_gemm_residual.h.

Argument marshalling only: every step of the operation runs in the CUDA
library.  Functions carry the C names.  Tensor arguments are torch CUDA
tensors of dtype bfloat16 (2-D, unit inner stride); raw-pointer forms
(``*_ptr``) take integers.  There is no CPU fallback: if the library is not
built or does not load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

ABI_VERSION = 9  # must equal SGR_ABI_VERSION of the loaded library

SGR_OK = 0
SGR_ERR_NULL = 1
SGR_ERR_SHAPE = 2
SGR_ERR_ALIGN = 3
SGR_ERR_ALIAS = 4
SGR_ERR_UNSUPPORTED = 5
SGR_ERR_LAUNCH = 6
SGR_ERR_DEVICE = 7

SGR_FLAG_NO_PDL = 0x1

SGR_PATH_AUTO = 0
SGR_PATH_SIMT = 1
SGR_PATH_TC = 2
SGR_PATH_TC_ROWS = 3
SGR_PATH_TILE = 4
SGR_PATH_W8 = 5
SGR_PATH_PAIR = 6
SGR_PATH_W8S = 7


class sgr_group(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("W", ctypes.c_void_p),
                ("R", ctypes.c_void_p), ("ldr", ctypes.c_int64), ("Y", ctypes.c_void_p),
                ("ldy", ctypes.c_int64), ("M", ctypes.c_int), ("reserved", ctypes.c_int)]


class SgrError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({sgr_status_string(status)})")


class sgr_config(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("stages", ctypes.c_int), ("rows_per_stage", ctypes.c_int),
                ("k_blocks_per_stage", ctypes.c_int), ("token_tile", ctypes.c_int),
                ("prefetch_stages", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("k_split", ctypes.c_int),
                ("reserved", ctypes.c_int * 2)]

    def as_dict(self) -> dict:
        return {"path": self.path, "ctas_per_sm": self.ctas_per_sm, "stages": self.stages,
                "rows_per_stage": self.rows_per_stage,
                "k_blocks_per_stage": self.k_blocks_per_stage, "token_tile": self.token_tile,
                "prefetch_stages": self.prefetch_stages, "tile_n": self.tile_n, "k_split": self.k_split}


_lock = threading.Lock()
_lib = None

# Entry points declared in include/skinny_gemm_residual.h.
EXPORTS = (
    "skinny_gemm_residual",
    "skinny_gemm_residual_ex",
    "skinny_gemm_residual_config",
    "sgr_validate",
    "sgr_select_path",
    "sgr_default_config",
    "sgr_init",
    "sgr_device_error",
    "sgr_kernel_resources",
    "sgr_status_string",
    "sgr_abi_version",
    "skinny_gemm_residual_noalloc",
    "skinny_gemm_residual_grouped",
    "skinny_gemm_residual_w8",
    "sgr_validate_w8",
    "skinny_gemm_residual_w4",
    "sgr_validate_w4",
    "sgr_selftest_wait_timeout",
    "sgr_selftest_streamk_abort",
)


def library_path() -> str:
    return os.environ.get("SGR_LIBRARY", _build.LIB_PATH)


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library; raise if impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if build_if_missing and path == _build.LIB_PATH and _build.is_stale(path):
            _build.build_library()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not found at {path}; run the build step")
        lib = ctypes.CDLL(path)
        vp, i64, I, U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint
        ip = ctypes.POINTER(ctypes.c_int)
        lib.skinny_gemm_residual.argtypes = [vp, vp, vp, vp, I, I, I, vp]
        lib.skinny_gemm_residual_ex.argtypes = [vp, i64, vp, vp, i64, vp, i64, I, I, I, U, vp]
        lib.skinny_gemm_residual_config.argtypes = [vp, i64, vp, vp, i64, vp, i64, I, I, I,
                                                    ctypes.POINTER(sgr_config), U, vp]
        lib.sgr_validate.argtypes = [vp, i64, vp, vp, i64, vp, i64, I, I, I]
        lib.sgr_select_path.argtypes = [I, I, I]
        lib.sgr_default_config.argtypes = [I, I, I, I, I, ctypes.POINTER(sgr_config)]
        lib.sgr_init.argtypes = [I]
        lib.sgr_device_error.argtypes = [I, ctypes.POINTER(ctypes.c_uint), I]
        lib.sgr_kernel_resources.argtypes = [I, I, I, I, I, ip, ip, ip, ip]
        lib.sgr_status_string.argtypes = [I]
        lib.sgr_status_string.restype = ctypes.c_char_p
        lib.sgr_abi_version.argtypes = []
        lib.skinny_gemm_residual_noalloc.argtypes = [vp, i64, vp, vp, i64, vp, i64, I, I, I, U, vp]
        lib.skinny_gemm_residual_grouped.argtypes = [ctypes.POINTER(sgr_group), I, I, I,
                                                     ctypes.POINTER(sgr_config), U, vp]
        fp = ctypes.POINTER(ctypes.c_float)
        lib.skinny_gemm_residual_w8.argtypes = [vp, i64, vp, i64, fp, vp, i64, vp, i64, I, I, I,
                                                ctypes.POINTER(sgr_config), U, vp]
        lib.sgr_validate_w8.argtypes = [vp, i64, vp, i64, fp, vp, i64, vp, i64, I, I, I]
        lib.skinny_gemm_residual_w4.argtypes = [vp, i64, vp, i64, vp, i64, ctypes.c_float, vp, i64, vp, i64,
                                                I, I, I, ctypes.POINTER(sgr_config), U, vp]
        lib.sgr_validate_w4.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, I, I, I]
        lib.sgr_selftest_wait_timeout.argtypes = [U, ctypes.POINTER(ctypes.c_uint)]
        lib.sgr_selftest_streamk_abort.argtypes = [vp, vp, vp, vp, I, I, I, I, ctypes.POINTER(ctypes.c_uint)]
        for name in EXPORTS:
            if name != "sgr_status_string":
                getattr(lib, name).restype = ctypes.c_int
        v = lib.sgr_abi_version()
        if v != ABI_VERSION:
            raise RuntimeError(f"library ABI version {v} != binding ABI version {ABI_VERSION}; rebuild")
        _lib = lib
        return lib


# ---------------------------------------------------------------- host-only
def sgr_status_string(status: int) -> str:
    return load().sgr_status_string(int(status)).decode()


def sgr_abi_version() -> int:
    return load().sgr_abi_version()


def sgr_validate_ptr(A: int, lda: int, W: int, R: int, ldr: int, Y: int, ldy: int,
                     M: int, N: int, K: int) -> int:
    """Host-only argument check on raw addresses; returns the status."""
    return load().sgr_validate(A, lda, W, R, ldr, Y, ldy, M, N, K)


def sgr_select_path(M: int, N: int, K: int) -> int:
    return load().sgr_select_path(M, N, K)


def sgr_default_config(M: int, N: int, K: int, path: int = SGR_PATH_AUTO, device: int | None = None) -> sgr_config:
    import torch

    dev = torch.cuda.current_device() if device is None else device
    c = sgr_config()
    rc = load().sgr_default_config(dev, M, N, K, path, ctypes.byref(c))
    if rc != SGR_OK:
        raise SgrError(rc, "sgr_default_config")
    return c


def sgr_init(device: int | None = None) -> None:
    import torch

    dev = torch.cuda.current_device() if device is None else device
    rc = load().sgr_init(dev)
    if rc != SGR_OK:
        raise SgrError(rc, "sgr_init")


def sgr_device_error(device: int | None = None, clear: bool = True) -> int:
    import torch

    dev = torch.cuda.current_device() if device is None else device
    code = ctypes.c_uint(0)
    rc = load().sgr_device_error(dev, ctypes.byref(code), 1 if clear else 0)
    if rc != SGR_OK:
        raise SgrError(rc, "sgr_device_error")
    return code.value


def sgr_kernel_resources(M: int, N: int, K: int, path: int = SGR_PATH_AUTO,
                         device: int | None = None) -> dict:
    import torch

    dev = torch.cuda.current_device() if device is None else device
    vals = [ctypes.c_int(0) for _ in range(4)]
    rc = load().sgr_kernel_resources(dev, path, M, N, K, *(ctypes.byref(v) for v in vals))
    if rc != SGR_OK:
        raise SgrError(rc, "sgr_kernel_resources")
    return dict(zip(("registers_per_thread", "spill_bytes", "smem_bytes", "threads"),
                    (v.value for v in vals)))


# ---------------------------------------------------------------- launches
def _common_device(tensors):
    """The one device every tensor lives on.  The library launches on the
    calling thread's current CUDA device, so the tensor-level calls make that
    device current for the call; tensors on different devices are refused
    (their addresses would reach a kernel on a device that does not own them)."""
    dev = tensors[0].device
    for t in tensors[1:]:
        if t.device != dev:
            raise ValueError(f"all tensors must be on one CUDA device, got {dev} and {t.device}")
    return dev


def _stream_handle(stream, device=None) -> int:
    import torch

    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    if device is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device}, tensors on {device}")
    return stream.cuda_stream


def _check_tensor(t, name: str):
    import torch

    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be torch.bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit inner stride")


def _ld(t) -> int:
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def skinny_gemm_residual_ptr(A: int, W: int, R: int, Y: int, M: int, N: int, K: int, stream: int) -> int:
    return load().skinny_gemm_residual(A, W, R, Y, M, N, K, stream)


def skinny_gemm_residual_ex_ptr(A: int, lda: int, W: int, R: int, ldr: int, Y: int, ldy: int,
                                M: int, N: int, K: int, flags: int, stream: int) -> int:
    return load().skinny_gemm_residual_ex(A, lda, W, R, ldr, Y, ldy, M, N, K, flags, stream)


def skinny_gemm_residual_config_ptr(A: int, lda: int, W: int, R: int, ldr: int, Y: int, ldy: int,
                                    M: int, N: int, K: int, cfg: sgr_config | None, flags: int,
                                    stream: int) -> int:
    return load().skinny_gemm_residual_config(A, lda, W, R, ldr, Y, ldy, M, N, K,
                                              ctypes.byref(cfg) if cfg is not None else None,
                                              flags, stream)


def skinny_gemm_residual(A, W, R, Y=None, stream=None):
    """Y = bf16(A . W^T + R) for contiguous CUDA bf16 tensors; returns Y."""
    import torch

    for t, n in ((A, "A"), (W, "W"), (R, "R")):
        _check_tensor(t, n)
    if Y is None:
        Y = torch.empty_like(R, memory_format=torch.contiguous_format)
    _check_tensor(Y, "Y")
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(R.shape) != (M, N) or tuple(Y.shape) != (M, N):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} W{tuple(W.shape)} R{tuple(R.shape)} Y{tuple(Y.shape)}")
    if not (A.is_contiguous() and W.is_contiguous() and R.is_contiguous() and Y.is_contiguous()):
        raise ValueError("skinny_gemm_residual takes contiguous tensors; use skinny_gemm_residual_ex")
    dev = _common_device((A, W, R, Y))
    with torch.cuda.device(dev):
        rc = load().skinny_gemm_residual(A.data_ptr(), W.data_ptr(), R.data_ptr(), Y.data_ptr(),
                                         M, N, K, _stream_handle(stream, dev))
    if rc != SGR_OK:
        raise SgrError(rc, "skinny_gemm_residual")
    return Y


def skinny_gemm_residual_ex(A, W, R, Y=None, flags: int = 0, stream=None, config: sgr_config | None = None):
    """Row-strided form: A, R, Y may be row slices/column slices with unit inner stride."""
    import torch

    for t, n in ((A, "A"), (W, "W"), (R, "R")):
        _check_tensor(t, n)
    if Y is None:
        Y = torch.empty(R.shape, dtype=R.dtype, device=R.device)
    _check_tensor(Y, "Y")
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(R.shape) != (M, N) or tuple(Y.shape) != (M, N):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} W{tuple(W.shape)} R{tuple(R.shape)} Y{tuple(Y.shape)}")
    if not W.is_contiguous():
        raise ValueError("W must be contiguous [N, K]")
    dev = _common_device((A, W, R, Y))
    with torch.cuda.device(dev):
        if config is None:
            rc = load().skinny_gemm_residual_ex(A.data_ptr(), _ld(A), W.data_ptr(), R.data_ptr(), _ld(R),
                                                Y.data_ptr(), _ld(Y), M, N, K, flags, _stream_handle(stream, dev))
            what = "skinny_gemm_residual_ex"
        else:
            rc = skinny_gemm_residual_config_ptr(A.data_ptr(), _ld(A), W.data_ptr(), R.data_ptr(), _ld(R),
                                                 Y.data_ptr(), _ld(Y), M, N, K, config, flags,
                                                 _stream_handle(stream, dev))
            what = "skinny_gemm_residual_config"
    if rc != SGR_OK:
        raise SgrError(rc, what)
    return Y


def skinny_gemm_residual_config(A, W, R, Y=None, config: sgr_config | None = None, flags: int = 0, stream=None):
    """Explicit launch configuration (sweeps, tests)."""
    return skinny_gemm_residual_ex(A, W, R, Y, flags=flags, stream=stream,
                                   config=config if config is not None else sgr_config())


def sgr_selftest_wait_timeout(limit_us: int = 1000) -> int:
    """Run the bounded-wait failure self-test on the current device; returns
    the error code the timed-out wait recorded (1 expected)."""
    code = ctypes.c_uint(0)
    rc = load().sgr_selftest_wait_timeout(int(limit_us), ctypes.byref(code))
    if rc != SGR_OK:
        raise SgrError(rc, "sgr_selftest_wait_timeout")
    return code.value


def sgr_selftest_streamk_abort(A, W, R, Y, cta: int) -> int:
    """One stream-K launch on the current device's default stream in which CTA
    `cta` acts as if its first accumulator wait ran out; returns the code the
    kernel recorded (3 expected).  Contiguous CUDA tensors; Y is overwritten
    with unspecified values."""
    import torch

    for t in (A, W, R, Y):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError("sgr_selftest_streamk_abort takes contiguous CUDA bfloat16 tensors")
    M, K = A.shape
    N = W.shape[0]
    code = ctypes.c_uint(0)
    rc = load().sgr_selftest_streamk_abort(A.data_ptr(), W.data_ptr(), R.data_ptr(), Y.data_ptr(), M, N, K,
                                           int(cta), ctypes.byref(code))
    if rc != SGR_OK:
        raise SgrError(rc, "sgr_selftest_streamk_abort")
    return code.value


def _fptr(addr: int):
    return ctypes.cast(ctypes.c_void_p(addr), ctypes.POINTER(ctypes.c_float)) if addr else None


def sgr_validate_w8_ptr(A: int, lda: int, Wq: int, ldw: int, scale: int, R: int, ldr: int, Y: int, ldy: int,
                        M: int, N: int, K: int) -> int:
    """Host-only argument check of the FP8-weight entry point (no GPU needed)."""
    return load().sgr_validate_w8(A, lda, Wq, ldw, _fptr(scale), R, ldr, Y, ldy, M, N, K)


def skinny_gemm_residual_w8_ptr(A: int, lda: int, Wq: int, ldw: int, scale: int, R: int, ldr: int, Y: int,
                                ldy: int, M: int, N: int, K: int, cfg: sgr_config | None, flags: int,
                                stream: int) -> int:
    """FP8-weight entry point on raw device addresses; returns the status."""
    return load().skinny_gemm_residual_w8(A, lda, Wq, ldw, _fptr(scale), R, ldr, Y, ldy, M, N, K,
                                          ctypes.byref(cfg) if cfg is not None else None, flags, stream)


def skinny_gemm_residual_w8(A, Wq, scale, R, Y=None, flags: int = 0, stream=None,
                            config: sgr_config | None = None):
    """Y = bf16(scale[n] * A . e4m3(Wq)^T + R).

    A [M,K], R and Y [M,N]: CUDA bf16 with unit inner stride (row strides
    allowed).  Wq [N,K]: CUDA torch.uint8 or torch.float8_e4m3fn codes with
    unit inner stride and a row stride that is a multiple of 16 bytes.
    scale [N]: contiguous CUDA float32.  Returns Y."""
    import torch

    for t, n in ((A, "A"), (R, "R")):
        _check_tensor(t, n)
    if Wq.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"Wq must be torch.uint8 or torch.float8_e4m3fn, got {Wq.dtype}")
    if not Wq.is_cuda or Wq.dim() != 2 or (Wq.shape[1] > 1 and Wq.stride(1) != 1):
        raise ValueError("Wq must be a 2-D CUDA tensor with unit inner stride")
    if scale.dtype != torch.float32 or not scale.is_cuda or scale.dim() != 1 or not scale.is_contiguous():
        raise ValueError("scale must be a contiguous 1-D CUDA float32 tensor")
    if Y is None:
        Y = torch.empty(R.shape, dtype=R.dtype, device=R.device)
    _check_tensor(Y, "Y")
    M, K = A.shape
    N = Wq.shape[0]
    if Wq.shape[1] != K or tuple(R.shape) != (M, N) or tuple(Y.shape) != (M, N) or scale.shape[0] != N:
        raise ValueError(f"shape mismatch A{tuple(A.shape)} Wq{tuple(Wq.shape)} scale{tuple(scale.shape)} "
                         f"R{tuple(R.shape)} Y{tuple(Y.shape)}")
    dev = _common_device((A, Wq, scale, R, Y))
    with torch.cuda.device(dev):
        rc = skinny_gemm_residual_w8_ptr(A.data_ptr(), _ld(A), Wq.data_ptr(), _ld(Wq), scale.data_ptr(),
                                         R.data_ptr(), _ld(R), Y.data_ptr(), _ld(Y), M, N, K, config, flags,
                                         _stream_handle(stream, dev))
    if rc != SGR_OK:
        raise SgrError(rc, "skinny_gemm_residual_w8")
    return Y


def sgr_validate_w4_ptr(A: int, lda: int, Wq4: int, ldw: int, bs: int, ldbs: int, R: int, ldr: int, Y: int,
                        ldy: int, M: int, N: int, K: int) -> int:
    """Host-only argument check of the NVFP4-weight entry point (no GPU needed)."""
    return load().sgr_validate_w4(A, lda, Wq4, ldw, bs, ldbs, R, ldr, Y, ldy, M, N, K)


def skinny_gemm_residual_w4_ptr(A: int, lda: int, Wq4: int, ldw: int, bs: int, ldbs: int, gs: float, R: int,
                                ldr: int, Y: int, ldy: int, M: int, N: int, K: int, cfg: sgr_config | None,
                                flags: int, stream: int) -> int:
    """NVFP4-weight entry point on raw device addresses; returns the status."""
    return load().skinny_gemm_residual_w4(A, lda, Wq4, ldw, bs, ldbs, float(gs), R, ldr, Y, ldy, M, N, K,
                                          ctypes.byref(cfg) if cfg is not None else None, flags, stream)


def skinny_gemm_residual_w4(A, Wq4, bs, gs: float, R, Y=None, flags: int = 0, stream=None,
                            config: sgr_config | None = None):
    """Y = bf16(gs * A . (e2m1(Wq4) * e4m3(bs))^T + R).

    A [M,K], R and Y [M,N]: CUDA bf16 with unit inner stride (row strides
    allowed).  Wq4 [N,K/2]: CUDA torch.uint8, two E2M1 codes per byte
    (element 2i in the low nibble), unit inner stride, row stride a multiple
    of 16 bytes.  bs [N,ceil(K/16)]: CUDA torch.uint8 or float8_e4m3fn block
    scales, unit inner stride, row stride a multiple of 16 bytes and at least
    ceil(K/16) rounded up to 16 (rows are read in 16-byte units).  gs: the
    tensor's scale (a float).  Returns Y."""
    import torch

    for t, n in ((A, "A"), (R, "R")):
        _check_tensor(t, n)
    if Wq4.dtype != torch.uint8:
        raise TypeError(f"Wq4 must be torch.uint8, got {Wq4.dtype}")
    if bs.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"bs must be torch.uint8 or torch.float8_e4m3fn, got {bs.dtype}")
    for t, n in ((Wq4, "Wq4"), (bs, "bs")):
        if not t.is_cuda or t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError(f"{n} must be a 2-D CUDA tensor with unit inner stride")
    if Y is None:
        Y = torch.empty(R.shape, dtype=R.dtype, device=R.device)
    _check_tensor(Y, "Y")
    M, K = A.shape
    N = Wq4.shape[0]
    if (K % 2 or Wq4.shape[1] != K // 2 or tuple(bs.shape) != (N, (K + 15) // 16) or tuple(R.shape) != (M, N)
            or tuple(Y.shape) != (M, N)):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} Wq4{tuple(Wq4.shape)} bs{tuple(bs.shape)} "
                         f"R{tuple(R.shape)} Y{tuple(Y.shape)}")
    padded = ((K + 15) // 16 + 15) // 16 * 16
    ldbs = bs.stride(0) if N > 1 else padded
    if K > 0 and N > 0 and bs.untyped_storage().nbytes() - bs.storage_offset() < (N - 1) * ldbs + padded:
        raise ValueError("bs rows are read in 16-byte units: the buffer must hold the padding of the last row")
    dev = _common_device((A, Wq4, bs, R, Y))
    with torch.cuda.device(dev):
        rc = skinny_gemm_residual_w4_ptr(A.data_ptr(), _ld(A), Wq4.data_ptr(), _ld(Wq4), bs.data_ptr(), ldbs,
                                         float(gs), R.data_ptr(), _ld(R), Y.data_ptr(), _ld(Y), M, N, K, config,
                                         flags, _stream_handle(stream, dev))
    if rc != SGR_OK:
        raise SgrError(rc, "skinny_gemm_residual_w4")
    return Y


def skinny_gemm_residual_noalloc_ptr(A: int, lda: int, W: int, R: int, ldr: int, Y: int, ldy: int,
                                    M: int, N: int, K: int, flags: int, stream: int) -> int:
    """Allocation-free entry point on raw device addresses; returns the status."""
    return load().skinny_gemm_residual_noalloc(A, lda, W, R, ldr, Y, ldy, M, N, K, flags, stream)


def skinny_gemm_residual_noalloc(A, W, R, Y, flags: int = 0, stream=None):
    """Y = bf16(A . W^T + R) without any device allocation (fixed scratch
    inside the library; see include/skinny_gemm_residual.h).  Y is required:
    this call allocates nothing, not even its output."""
    import torch

    for t, n in ((A, "A"), (W, "W"), (R, "R"), (Y, "Y")):
        _check_tensor(t, n)
    M, K = A.shape
    N = W.shape[0]
    if W.shape[1] != K or tuple(R.shape) != (M, N) or tuple(Y.shape) != (M, N):
        raise ValueError(f"shape mismatch A{tuple(A.shape)} W{tuple(W.shape)} R{tuple(R.shape)} Y{tuple(Y.shape)}")
    if not W.is_contiguous():
        raise ValueError("W must be contiguous [N, K]")
    dev = _common_device((A, W, R, Y))
    with torch.cuda.device(dev):
        rc = skinny_gemm_residual_noalloc_ptr(A.data_ptr(), _ld(A), W.data_ptr(), R.data_ptr(), _ld(R),
                                              Y.data_ptr(), _ld(Y), M, N, K, flags, _stream_handle(stream, dev))
    if rc != SGR_OK:
        raise SgrError(rc, "skinny_gemm_residual_noalloc")
    return Y


def skinny_gemm_residual_grouped_ptr(groups, N: int, K: int, config: sgr_config | None = None,
                                     flags: int = 0, stream: int = 0) -> int:
    """Grouped entry point on an array of sgr_group (raw device addresses);
    returns the status."""
    arr = (sgr_group * max(1, len(groups)))(*groups)
    cfg = ctypes.byref(config) if config is not None else None
    return load().skinny_gemm_residual_grouped(arr, len(groups), N, K, cfg, flags, stream)


def skinny_gemm_residual_grouped(problems, flags: int = 0, stream=None, config: sgr_config | None = None):
    """Y_g = bf16(A_g . W_g^T + R_g) for every (A, W, R, Y) in `problems`
    (the experts of a mixture-of-experts layer: same N and K, own weights and
    token counts; an A with zero rows skips that expert), in one launch.
    Y may be None (allocated).  Returns the list of Y."""
    import torch

    groups, outs, tensors = [], [], []
    N = K = None
    for A, W, R, Y in problems:
        for t, n in ((A, "A"), (W, "W"), (R, "R")):
            _check_tensor(t, n)
        M, k = A.shape
        n_out = W.shape[0]
        if N is None:
            N, K = n_out, k
        if (n_out, W.shape[1], k) != (N, K, K) or tuple(R.shape) != (M, N):
            raise ValueError("every group needs W [N, K], A [M, K], R [M, N] with one N and K")
        if not W.is_contiguous():
            raise ValueError("W must be contiguous [N, K]")
        if Y is None:
            Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
        _check_tensor(Y, "Y")
        if tuple(Y.shape) != (M, N):
            raise ValueError("Y must be [M, N]")
        groups.append(sgr_group(A.data_ptr(), _ld(A), W.data_ptr(), R.data_ptr(), _ld(R), Y.data_ptr(), _ld(Y), M, 0))
        outs.append(Y)
        tensors += [A, W, R, Y]
    if not groups:
        return outs
    dev = _common_device(tensors)
    with torch.cuda.device(dev):
        rc = skinny_gemm_residual_grouped_ptr(groups, N, K, config, flags, _stream_handle(stream, dev))
    if rc != SGR_OK:
        raise SgrError(rc, "skinny_gemm_residual_grouped")
    return outs


def make_config(path: int = SGR_PATH_AUTO, ctas_per_sm: int = 0, stages: int = 0,
                rows_per_stage: int = 0, k_blocks_per_stage: int = 0, token_tile: int = 0,
                prefetch_stages: int = 0, tile_n: int = 0, k_split: int = 0) -> sgr_config:
    c = sgr_config()
    c.path, c.ctas_per_sm, c.stages = path, ctas_per_sm, stages
    c.rows_per_stage, c.k_blocks_per_stage, c.token_tile = rows_per_stage, k_blocks_per_stage, token_tile
    c.prefetch_stages, c.tile_n, c.k_split = prefetch_stages, tile_n, k_split
    return c
