"""CPU oracle for Y = bf16(A . W^T + R) and its low-bit weight variants
Y = bf16(scale . A . e4m3(Wq)^T + R) (FP8) and
Y = bf16(gs . A . (e2m1(Wq4) . e4m3(bs))^T + R) (NVFP4)  --  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never calls it and shares no code with it.

The arithmetic lives in ``skinny_ref.c`` (plain C, FP64 accumulation, one
round-to-nearest-even to BF16; see the header of that file for the passages it
follows).  This module compiles it with gcc and wraps it with ctypes.  BF16
arrays travel as numpy uint16 bit patterns, FP8 E4M3 weights as uint8 codes,
NVFP4 weights as uint8 bytes holding two E2M1 codes (element 2i in the low
nibble) plus uint8 E4M3 block scales (one per 16 elements of a row); torch
tensors are accepted and converted with ``to_bits`` / ``to_codes``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "skinny_ref.c")
BUILD_DIR = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_cache: dict[str, "Oracle"] = {}

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-Wall"]


def build(mutant: int = 0, out_dir: str | None = None) -> str:
    """Compile the oracle (optionally with a planted mistake) and return the .so path."""
    out_dir = out_dir or BUILD_DIR
    os.makedirs(out_dir, exist_ok=True)
    name = "libskinny_ref.so" if mutant == 0 else f"libskinny_ref_mutant{mutant}.so"
    out = os.path.join(out_dir, name)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SOURCE):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DSGR_REF_MUTANT={int(mutant)}", SOURCE, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def to_bits(x) -> np.ndarray:
    """torch.bfloat16 tensor (any device) or uint16 array -> numpy uint16 bits."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("expected uint16 BF16 bit patterns")
        return x
    import torch

    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected torch.bfloat16, got {x.dtype}")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _to_numpy(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return x
    return x.detach().cpu().contiguous().numpy()


def to_codes(x) -> np.ndarray:
    """FP8 E4M3 codes: uint8 array, or a torch uint8 / float8_e4m3fn tensor -> numpy uint8."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint8:
            raise TypeError("expected uint8 E4M3 codes")
        return x
    import torch

    if x.dtype == torch.float8_e4m3fn:
        x = x.view(torch.uint8)
    if x.dtype != torch.uint8:
        raise TypeError(f"expected torch.uint8 or float8_e4m3fn, got {x.dtype}")
    return x.detach().cpu().contiguous().numpy()


def from_bits(bits: np.ndarray):
    """numpy uint16 bits -> torch.bfloat16 CPU tensor."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _rows(a: np.ndarray) -> tuple[np.ndarray, int]:
    """Return (array, row stride in elements); inner stride must be one element."""
    if a.ndim != 2:
        raise ValueError("expected a 2-D array")
    if a.strides[1] != a.itemsize or a.strides[0] % a.itemsize or a.strides[0] < 0:
        a = np.ascontiguousarray(a)
    ld = a.strides[0] // a.itemsize if a.shape[0] > 1 else a.shape[1]
    return a, max(ld, a.shape[1])


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        L, I = ctypes.c_long, ctypes.c_int
        lib.sgr_ref_round_bf16.restype = ctypes.c_uint16
        lib.sgr_ref_round_bf16.argtypes = [ctypes.c_double]
        lib.sgr_ref_round_bf16_array.restype = None
        lib.sgr_ref_round_bf16_array.argtypes = [dp, u16p, L]
        lib.sgr_ref_bf16_to_double.restype = ctypes.c_double
        lib.sgr_ref_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.sgr_ref_gemm_residual.restype = I
        lib.sgr_ref_gemm_residual.argtypes = [u16p, L, u16p, L, u16p, L, u16p, L, L, L, L, I]
        lib.sgr_ref_gemm_residual_f64.restype = I
        lib.sgr_ref_gemm_residual_f64.argtypes = [u16p, L, u16p, L, u16p, L, dp, L, L, L, L, I]
        lib.sgr_ref_sample.restype = I
        lib.sgr_ref_sample.argtypes = [u16p, L, u16p, L, u16p, L, L, L, L, lp, lp, L, u16p]
        u8p = ctypes.POINTER(ctypes.c_uint8)
        fp = ctypes.POINTER(ctypes.c_float)
        lib.sgr_ref_gemm_residual_w8.restype = I
        lib.sgr_ref_gemm_residual_w8.argtypes = [u16p, L, u8p, L, fp, u16p, L, u16p, L, L, L, L, I]
        lib.sgr_ref_sample_w8.restype = I
        lib.sgr_ref_sample_w8.argtypes = [u16p, L, u8p, L, fp, u16p, L, L, L, L, lp, lp, L, u16p]
        lib.sgr_ref_e4m3_to_double.restype = ctypes.c_double
        lib.sgr_ref_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.sgr_ref_gemm_residual_w4.restype = I
        lib.sgr_ref_gemm_residual_w4.argtypes = [u16p, L, u8p, L, u8p, L, ctypes.c_float, u16p, L, u16p, L,
                                                 L, L, L, I]
        lib.sgr_ref_sample_w4.restype = I
        lib.sgr_ref_sample_w4.argtypes = [u16p, L, u8p, L, u8p, L, ctypes.c_float, u16p, L, L, L, L, lp, lp, L,
                                          u16p]
        lib.sgr_ref_e2m1_to_double.restype = ctypes.c_double
        lib.sgr_ref_e2m1_to_double.argtypes = [ctypes.c_uint8]
        lib.sgr_ref_mutant.restype = I
        lib.sgr_ref_mutant.argtypes = []
        self.lib = lib
        self.mutant = lib.sgr_ref_mutant()

    @staticmethod
    def _p(a: np.ndarray, ctype):
        return a.ctypes.data_as(ctypes.POINTER(ctype))

    def _operands(self, A, W, R):
        A, lda = _rows(to_bits(A))
        W, ldw = _rows(to_bits(W))
        R, ldr = _rows(to_bits(R))
        M, K = A.shape
        N = W.shape[0]
        if W.shape[1] != K or R.shape != (M, N):
            raise ValueError(f"shape mismatch: A{A.shape} W{W.shape} R{R.shape}")
        return A, lda, W, ldw, R, ldr, M, N, K

    def gemm_residual(self, A, W, R, threads: int | None = None) -> np.ndarray:
        """Y = bf16_rne(A . W^T + R) as a uint16 [M,N] array (every element)."""
        A, lda, W, ldw, R, ldr, M, N, K = self._operands(A, W, R)
        Y = np.empty((M, N), dtype=np.uint16)
        threads = threads or os.cpu_count() or 1
        rc = self.lib.sgr_ref_gemm_residual(
            self._p(A, ctypes.c_uint16), lda, self._p(W, ctypes.c_uint16), ldw,
            self._p(R, ctypes.c_uint16), ldr, self._p(Y, ctypes.c_uint16), N,
            M, N, K, int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle failed with status {rc}")
        return Y

    def gemm_residual_f64(self, A, W, R, threads: int | None = None) -> np.ndarray:
        """The unrounded FP64 value A . W^T + R as a float64 [M,N] array."""
        A, lda, W, ldw, R, ldr, M, N, K = self._operands(A, W, R)
        T = np.empty((M, N), dtype=np.float64)
        threads = threads or os.cpu_count() or 1
        rc = self.lib.sgr_ref_gemm_residual_f64(
            self._p(A, ctypes.c_uint16), lda, self._p(W, ctypes.c_uint16), ldw,
            self._p(R, ctypes.c_uint16), ldr, self._p(T, ctypes.c_double), N,
            M, N, K, int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle failed with status {rc}")
        return T

    def sample(self, A, W, R, ms, ns) -> np.ndarray:
        """Y[ms[i], ns[i]] for each i, as uint16."""
        A, lda, W, ldw, R, ldr, M, N, K = self._operands(A, W, R)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        if ms.shape != ns.shape or ms.ndim != 1:
            raise ValueError("ms and ns must be 1-D and of equal length")
        out = np.empty(ms.shape, dtype=np.uint16)
        rc = self.lib.sgr_ref_sample(
            self._p(A, ctypes.c_uint16), lda, self._p(W, ctypes.c_uint16), ldw,
            self._p(R, ctypes.c_uint16), ldr, M, N, K,
            self._p(ms, ctypes.c_long), self._p(ns, ctypes.c_long), len(ms),
            self._p(out, ctypes.c_uint16))
        if rc != 0:
            raise RuntimeError(f"oracle failed with status {rc}")
        return out

    def _operands_w8(self, A, Wq, scale, R):
        A, lda = _rows(to_bits(A))
        Wq, ldw = _rows(to_codes(Wq))
        R, ldr = _rows(to_bits(R))
        scale = np.ascontiguousarray(_to_numpy(scale), dtype=np.float32)
        M, K = A.shape
        N = Wq.shape[0]
        if Wq.shape[1] != K or R.shape != (M, N) or scale.shape != (N,):
            raise ValueError(f"shape mismatch: A{A.shape} Wq{Wq.shape} scale{scale.shape} R{R.shape}")
        return A, lda, Wq, ldw, scale, R, ldr, M, N, K

    def gemm_residual_w8(self, A, Wq, scale, R, threads: int | None = None) -> np.ndarray:
        """Y = bf16_rne(scale[n] * A . e4m3(Wq)^T + R) as uint16 [M,N] (every element).

        Wq: [N,K] E4M3 codes (uint8 array or torch uint8 / float8_e4m3fn
        tensor); scale: [N] float32."""
        A, lda, Wq, ldw, scale, R, ldr, M, N, K = self._operands_w8(A, Wq, scale, R)
        Y = np.empty((M, N), dtype=np.uint16)
        threads = threads or os.cpu_count() or 1
        rc = self.lib.sgr_ref_gemm_residual_w8(
            self._p(A, ctypes.c_uint16), lda, self._p(Wq, ctypes.c_uint8), ldw,
            self._p(scale, ctypes.c_float), self._p(R, ctypes.c_uint16), ldr,
            self._p(Y, ctypes.c_uint16), N, M, N, K, int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle failed with status {rc}")
        return Y

    def sample_w8(self, A, Wq, scale, R, ms, ns) -> np.ndarray:
        """Y[ms[i], ns[i]] of the low-bit variant, as uint16."""
        A, lda, Wq, ldw, scale, R, ldr, M, N, K = self._operands_w8(A, Wq, scale, R)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        if ms.shape != ns.shape or ms.ndim != 1:
            raise ValueError("ms and ns must be 1-D and of equal length")
        out = np.empty(ms.shape, dtype=np.uint16)
        rc = self.lib.sgr_ref_sample_w8(
            self._p(A, ctypes.c_uint16), lda, self._p(Wq, ctypes.c_uint8), ldw,
            self._p(scale, ctypes.c_float), self._p(R, ctypes.c_uint16), ldr, M, N, K,
            self._p(ms, ctypes.c_long), self._p(ns, ctypes.c_long), len(ms),
            self._p(out, ctypes.c_uint16))
        if rc != 0:
            raise RuntimeError(f"oracle failed with status {rc}")
        return out

    def _operands_w4(self, A, Wq4, bs, R):
        A, lda = _rows(to_bits(A))
        Wq4, ldw = _rows(to_codes(Wq4))
        bs, ldbs = _rows(to_codes(bs))
        R, ldr = _rows(to_bits(R))
        M, K = A.shape
        N = Wq4.shape[0]
        if K % 2 or Wq4.shape[1] != K // 2 or bs.shape != (N, (K + 15) // 16) or R.shape != (M, N):
            raise ValueError(f"shape mismatch: A{A.shape} Wq4{Wq4.shape} bs{bs.shape} R{R.shape}")
        return A, lda, Wq4, ldw, bs, ldbs, R, ldr, M, N, K

    def gemm_residual_w4(self, A, Wq4, bs, gs: float, R, threads: int | None = None) -> np.ndarray:
        """Y = bf16_rne(gs * A . (e2m1(Wq4) * e4m3(bs))^T + R) as uint16 [M,N] (every element).

        Wq4: [N, K/2] bytes of two E2M1 codes (element 2i in the low nibble);
        bs: [N, ceil(K/16)] E4M3 block scales; gs: the tensor's float32 scale."""
        A, lda, Wq4, ldw, bs, ldbs, R, ldr, M, N, K = self._operands_w4(A, Wq4, bs, R)
        Y = np.empty((M, N), dtype=np.uint16)
        threads = threads or os.cpu_count() or 1
        rc = self.lib.sgr_ref_gemm_residual_w4(
            self._p(A, ctypes.c_uint16), lda, self._p(Wq4, ctypes.c_uint8), ldw, self._p(bs, ctypes.c_uint8),
            ldbs, float(np.float32(gs)), self._p(R, ctypes.c_uint16), ldr, self._p(Y, ctypes.c_uint16), N, M, N,
            K, int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle failed with status {rc}")
        return Y

    def sample_w4(self, A, Wq4, bs, gs: float, R, ms, ns) -> np.ndarray:
        """Y[ms[i], ns[i]] of the NVFP4 variant, as uint16."""
        A, lda, Wq4, ldw, bs, ldbs, R, ldr, M, N, K = self._operands_w4(A, Wq4, bs, R)
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        if ms.shape != ns.shape or ms.ndim != 1:
            raise ValueError("ms and ns must be 1-D and of equal length")
        out = np.empty(ms.shape, dtype=np.uint16)
        rc = self.lib.sgr_ref_sample_w4(
            self._p(A, ctypes.c_uint16), lda, self._p(Wq4, ctypes.c_uint8), ldw, self._p(bs, ctypes.c_uint8),
            ldbs, float(np.float32(gs)), self._p(R, ctypes.c_uint16), ldr, M, N, K, self._p(ms, ctypes.c_long),
            self._p(ns, ctypes.c_long), len(ms), self._p(out, ctypes.c_uint16))
        if rc != 0:
            raise RuntimeError(f"oracle failed with status {rc}")
        return out

    def e2m1_to_double(self, codes) -> np.ndarray:
        """Values of 4-bit E2M1 codes (the low nibble of each uint8)."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        return np.array([self.lib.sgr_ref_e2m1_to_double(int(b)) for b in codes.ravel()]
                        ).reshape(codes.shape)

    def e4m3_to_double(self, codes) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        return np.array([self.lib.sgr_ref_e4m3_to_double(int(b)) for b in codes.ravel()]
                        ).reshape(codes.shape)

    def round_bf16(self, t) -> np.ndarray:
        t = np.ascontiguousarray(t, dtype=np.float64)
        out = np.empty(t.shape, dtype=np.uint16)
        self.lib.sgr_ref_round_bf16_array(self._p(t, ctypes.c_double),
                                          self._p(out, ctypes.c_uint16), t.size)
        return out

    def bf16_to_double(self, bits: np.ndarray) -> np.ndarray:
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        return np.array([self.lib.sgr_ref_bf16_to_double(int(b)) for b in bits.ravel()]
                        ).reshape(bits.shape)


def load(mutant: int = 0, out_dir: str | None = None) -> Oracle:
    """Build if needed and load the oracle library (cached per path)."""
    with _lock:
        path = build(mutant, out_dir)
        if path not in _cache:
            _cache[path] = Oracle(path)
        return _cache[path]


def gemm_residual(A, W, R, threads: int | None = None) -> np.ndarray:
    return load().gemm_residual(A, W, R, threads)


def gemm_residual_w8(A, Wq, scale, R, threads: int | None = None) -> np.ndarray:
    return load().gemm_residual_w8(A, Wq, scale, R, threads)


def gemm_residual_w4(A, Wq4, bs, gs: float, R, threads: int | None = None) -> np.ndarray:
    return load().gemm_residual_w4(A, Wq4, bs, gs, R, threads)
