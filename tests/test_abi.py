"""The C-ABI library builds, loads and exports every symbol the public header
declares; host-only argument checks (no GPU needed, nothing is launched)."""
import ctypes
import glob
import os
import re

import pytest

import skinny_bf16_gemm_residual_gb300 as sgr
from skinny_bf16_gemm_residual_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    assert "skinny_gemm_residual" in names
    assert set(binding.EXPORTS) <= set(names), set(binding.EXPORTS) - set(names)


def test_library_exports_every_declared_symbol():
    lib = sgr.load()
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)


def _header_text():
    text = "".join(open(h).read() for h in glob.glob(os.path.join(ROOT, "include", "*.h")))
    return re.sub(r"/\*.*?\*/", "", text, flags=re.S)


def test_header_constants_match_binding():
    """Every SGR_ constant of the header (ABI version, status codes, flags,
    paths) has the same value in the Python binding."""
    text = _header_text()
    consts = {m.group(1): int(m.group(2), 0) for m in re.finditer(r"#define\s+(SGR_\w+)\s+(0x[0-9a-fA-F]+|\d+)u?", text)}
    consts.update({m.group(1): int(m.group(2)) for m in re.finditer(r"\b(SGR_\w+)\s*=\s*(\d+)", text)})
    assert len(consts) >= 15, consts
    for name, value in consts.items():
        key = "ABI_VERSION" if name == "SGR_ABI_VERSION" else name
        assert getattr(binding, key) == value, (name, value, getattr(binding, key, None))


def _struct_fields(text, name):
    body = re.search(r"typedef struct\s*\{([^{}]*)\}\s*" + name + r"\s*;", text).group(1)
    return [m.group(1) for m in re.finditer(r"(\w+)\s*(?:\[\s*\d+\s*\])?\s*;", body)]


def test_header_structs_match_binding():
    """The ctypes structures list the C structures' fields in the same order
    with the same sizes (a stale layout would pass garbage to the library)."""
    text = _header_text()
    assert _struct_fields(text, "sgr_config") == [f[0] for f in binding.sgr_config._fields_]
    assert _struct_fields(text, "sgr_group") == [f[0] for f in binding.sgr_group._fields_]
    assert ctypes.sizeof(binding.sgr_config) == 11 * 4
    assert ctypes.sizeof(binding.sgr_group) == 7 * 8 + 2 * 4


def test_binding_argument_counts_match_header():
    """Each function's ctypes argument list is as long as its C parameter list."""
    text = _header_text()
    lib = sgr.load()
    seen = 0
    for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(([^()]*)\)\s*;", text, flags=re.M):
        name, params = m.group(1), m.group(2).strip()
        if name not in binding.EXPORTS:
            continue
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(getattr(lib, name).argtypes) == n, (name, n, getattr(lib, name).argtypes)
        seen += 1
    assert seen == len(binding.EXPORTS)


def test_abi_version_and_status_strings():
    assert sgr.sgr_abi_version() == sgr.ABI_VERSION
    for s in range(0, 8):
        assert sgr.sgr_status_string(s)
    assert sgr.sgr_status_string(99) == "unknown status"


# Fake, never-dereferenced addresses for the host-only validator.
BASE = 1 << 40
A_, W_, R_, Y_ = BASE, BASE + (1 << 32), BASE + (2 << 32), BASE + (3 << 32)


def v(A=A_, lda=3584, W=W_, R=R_, ldr=7168, Y=Y_, ldy=7168, M=4, N=7168, K=3584):
    return sgr.sgr_validate_ptr(A, lda, W, R, ldr, Y, ldy, M, N, K)


def test_validate_accepts_good_arguments():
    assert v() == sgr.SGR_OK
    assert v(M=1) == sgr.SGR_OK
    assert v(M=1024) == sgr.SGR_OK
    assert v(lda=7168, ldr=7168 * 2, ldy=7168 * 3) == sgr.SGR_OK


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), sgr.SGR_ERR_SHAPE),
    (dict(N=-8), sgr.SGR_ERR_SHAPE),
    (dict(K=-8), sgr.SGR_ERR_SHAPE),
    (dict(N=7170, ldr=7176, ldy=7176), sgr.SGR_ERR_SHAPE),
    (dict(K=3585, lda=3592), sgr.SGR_ERR_SHAPE),
    (dict(A=0), sgr.SGR_ERR_NULL),
    (dict(W=0), sgr.SGR_ERR_NULL),
    (dict(R=0), sgr.SGR_ERR_NULL),
    (dict(Y=0), sgr.SGR_ERR_NULL),
    (dict(lda=3576), sgr.SGR_ERR_SHAPE),
    (dict(ldr=7160), sgr.SGR_ERR_SHAPE),
    (dict(ldy=7000), sgr.SGR_ERR_SHAPE),
    (dict(lda=3588), sgr.SGR_ERR_ALIGN),
    (dict(ldy=7172), sgr.SGR_ERR_ALIGN),
    (dict(A=A_ + 2), sgr.SGR_ERR_ALIGN),
    (dict(W=W_ + 8), sgr.SGR_ERR_ALIGN),
    (dict(R=R_ + 4), sgr.SGR_ERR_ALIGN),
    (dict(Y=Y_ + 2), sgr.SGR_ERR_ALIGN),
    (dict(Y=A_), sgr.SGR_ERR_ALIAS),
    (dict(Y=W_ + 4096), sgr.SGR_ERR_ALIAS),
    (dict(Y=R_ + 16), sgr.SGR_ERR_ALIAS),
    (dict(Y=R_, ldy=7176), sgr.SGR_ERR_ALIAS),
    (dict(M=(1 << 20) + 1), sgr.SGR_ERR_UNSUPPORTED),
    (dict(lda=(1 << 36) + 8), sgr.SGR_ERR_UNSUPPORTED),  # strides beyond 2^36 elements
    (dict(ldr=(1 << 36) + 8), sgr.SGR_ERR_UNSUPPORTED),
    (dict(ldy=1 << 62), sgr.SGR_ERR_UNSUPPORTED),        # would overflow the overlap arithmetic
])
def test_validate_rejects(kw, status):
    assert v(**kw) == status


def test_validate_largest_stride():
    big = dict(A=1 << 44, R=2 << 44, Y=3 << 44, ldr=1 << 36, ldy=1 << 36, M=2)  # regions 16 TiB apart
    assert v(W=4 << 44, lda=1 << 36, **big) == sgr.SGR_OK
    assert v8(Wq=4 << 44, scale=5 << 44, lda=1 << 36, ldw=1 << 36, **big) == sgr.SGR_OK


def test_validate_in_place_and_empty():
    assert v(Y=R_) == sgr.SGR_OK                       # Y == R exactly: in-place residual
    # M = 0 is a deliberate no-op (an expert with no tokens), not an error;
    # negative sizes are errors.
    assert v(M=0, A=0, W=0, R=0, Y=0) == sgr.SGR_OK    # empty problem
    assert v(M=-1) == sgr.SGR_ERR_SHAPE
    lib = sgr.load()
    assert lib.skinny_gemm_residual(None, None, None, None, 0, 7168, 3584, None) == sgr.SGR_OK
    assert lib.skinny_gemm_residual(None, None, None, None, -1, 7168, 3584, None) == sgr.SGR_ERR_SHAPE
    assert v(N=0, A=0, W=0, R=0, Y=0) == sgr.SGR_OK
    assert v(K=0, A=0, W=0) == sgr.SGR_OK              # empty sum: Y = R


def test_select_path():
    paths = (sgr.SGR_PATH_SIMT, sgr.SGR_PATH_TC, sgr.SGR_PATH_TC_ROWS, sgr.SGR_PATH_TILE, sgr.SGR_PATH_PAIR)
    for M in (1, 2, 3, 4, 8, 16, 32, 100, 256, 257, 1024, 5000):
        assert sgr.sgr_select_path(M, 7168, 3584) in paths
    for M in (1, 7, 300):  # shapes outside the measured table use the fallback rules
        assert sgr.sgr_select_path(M, 1024, 512) in paths
    assert sgr.sgr_select_path(257, 7168, 3584) in (sgr.SGR_PATH_TC, sgr.SGR_PATH_TILE, sgr.SGR_PATH_PAIR)  # row slab holds <= 256 tokens
    assert sgr.sgr_select_path(5000, 1024, 512) == sgr.SGR_PATH_TILE  # large M off the table: tile GEMM
    assert sgr.sgr_select_path(0, 7168, 3584) < 0
    assert sgr.sgr_select_path(4, 7170, 3584) < 0


def test_automatic_choice_never_takes_the_shared_workspace_path():
    """The stream-K kernel shares the library's per-device workspace, so only
    an explicit configuration may select it (the header says so)."""
    for N in (8, 152, 1024, 3584, 7168, 7176, 1 << 17):
        for K in (8, 64, 520, 3584, 7168, 65536):
            for M in (1, 2, 3, 16, 17, 64, 65, 128, 256, 257, 1024, 5000):
                path = sgr.sgr_select_path(M, N, K)
                assert path > 0 and path != sgr.SGR_PATH_TC, (M, N, K, path)


def test_table_header_is_sorted_and_covers_the_latent_moe_shape():
    """The generated per-M table lists entries by increasing M per (N, K)."""
    import re
    text = open(os.path.join(ROOT, "skinny_bf16_gemm_residual_gb300", "csrc", "sgr_table.h")).read()
    rows = [tuple(int(x) for x in m.groups()) for m in
            re.finditer(r"\{(\d+), (\d+), (\d+), (\d+),", text)]
    assert rows, "empty table"
    shapes = {}
    for n, k, m, path in rows:
        shapes.setdefault((n, k), []).append(m)
        assert path in (1, 2, 3, 4, 6)
    for ms in shapes.values():
        assert ms == sorted(ms)
    assert (7168, 3584) in shapes and shapes[(7168, 3584)][0] == 1


def test_table_header_is_generated_from_the_committed_tuning_rows():
    """sgr_table.h holds exactly what gen_table.py writes from the committed
    sweep rows (the comment block above the code aside)."""
    import glob
    import json

    from skinny_bf16_gemm_residual_gb300 import gen_table

    pkg = os.path.join(ROOT, "skinny_bf16_gemm_residual_gb300")
    rows = []
    for path in sorted(glob.glob(os.path.join(pkg, "tuning", "*.jsonl"))):
        with open(path) as f:
            rows += [json.loads(line) for line in f if line.strip()]
    want = gen_table.render(gen_table.best_rows(rows), "tuning")
    have = open(os.path.join(pkg, "csrc", "sgr_table.h")).read()
    code = lambda text: text[text.index("#pragma once"):]  # noqa: E731
    assert code(have) == code(want)


# ------------------------------------------------------------ grouped call (host-side checks only)
def grp(i, M=4, **kw):
    """Group i with fake addresses spaced 16 GiB apart (never dereferenced)."""
    off = i << 34
    f = dict(A=A_ + off, lda=3584, W=W_ + off, R=R_ + off, ldr=7168, Y=Y_ + off, ldy=7168, M=M)
    f.update(kw)
    return binding.sgr_group(f["A"], f["lda"], f["W"], f["R"], f["ldr"], f["Y"], f["ldy"], f["M"], 0)


def g_call(groups, N=7168, K=3584, n=None):
    return binding.skinny_gemm_residual_grouped_ptr(groups if n is None else groups[:n], N, K)


def test_grouped_rejects_before_launch():
    assert g_call([grp(0), grp(1, M=257)]) == sgr.SGR_ERR_UNSUPPORTED     # an expert batch above 256 tokens
    assert g_call([grp(0), grp(1, lda=3588)]) == sgr.SGR_ERR_ALIGN         # one bad group rejects the call
    assert g_call([grp(0), grp(1, R=0)]) == sgr.SGR_ERR_NULL
    # group 1 writes into group 0's residual / weights / output
    assert g_call([grp(0), grp(1, Y=R_)]) == sgr.SGR_ERR_ALIAS
    assert g_call([grp(0), grp(1, Y=W_)]) == sgr.SGR_ERR_ALIAS
    assert g_call([grp(0), grp(1, Y=Y_)]) == sgr.SGR_ERR_ALIAS
    bad = grp(0)
    bad.reserved = 1
    assert g_call([bad]) == sgr.SGR_ERR_UNSUPPORTED
    lib = sgr.load()
    assert lib.skinny_gemm_residual_grouped(None, 2, 7168, 3584, None, 0, None) == sgr.SGR_ERR_NULL
    assert lib.skinny_gemm_residual_grouped(None, -1, 7168, 3584, None, 0, None) == sgr.SGR_ERR_UNSUPPORTED


def test_grouped_nothing_to_do_needs_no_device():
    assert g_call([]) == sgr.SGR_OK
    assert g_call([grp(0, M=0), grp(1, M=0)]) == sgr.SGR_OK   # no expert received a token


# ------------------------------------------------------------ FP8-weight entry point (host-side checks only)
S_ = BASE + (4 << 32)


def v8(A=A_, lda=3584, Wq=W_, ldw=3584, scale=S_, R=R_, ldr=7168, Y=Y_, ldy=7168, M=4, N=7168, K=3584):
    return sgr.sgr_validate_w8_ptr(A, lda, Wq, ldw, scale, R, ldr, Y, ldy, M, N, K)


def test_validate_w8_accepts_good_arguments():
    assert v8() == sgr.SGR_OK
    assert v8(M=256, ldw=3600) == sgr.SGR_OK            # padded code rows (multiple of 16 bytes)
    assert v8(Y=R_) == sgr.SGR_OK                       # in-place residual
    assert v8(M=0, A=0, Wq=0, scale=0, R=0, Y=0) == sgr.SGR_OK
    assert v8(K=0, A=0, Wq=0, scale=0) == sgr.SGR_OK    # empty sum: Y = R
    assert v8(scale=S_ + 4) == sgr.SGR_OK               # scales need only float alignment


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), sgr.SGR_ERR_SHAPE),
    (dict(K=3580, lda=3584, ldw=3584), sgr.SGR_ERR_SHAPE),
    (dict(Wq=0), sgr.SGR_ERR_NULL),
    (dict(scale=0), sgr.SGR_ERR_NULL),
    (dict(ldw=3576), sgr.SGR_ERR_SHAPE),
    (dict(ldw=3592), sgr.SGR_ERR_ALIGN),                # row stride not a multiple of 16 bytes
    (dict(Wq=W_ + 8), sgr.SGR_ERR_ALIGN),
    (dict(scale=S_ + 2), sgr.SGR_ERR_ALIGN),
    (dict(Y=W_ + 4096), sgr.SGR_ERR_ALIAS),              # Y inside the codes
    (dict(Y=S_ - 4096), sgr.SGR_ERR_ALIAS),              # Y runs into the scales
    (dict(Y=A_), sgr.SGR_ERR_ALIAS),
    (dict(Y=R_ + 16), sgr.SGR_ERR_ALIAS),
    (dict(ldw=(1 << 36) + 16), sgr.SGR_ERR_UNSUPPORTED),
    (dict(ldr=1 << 62), sgr.SGR_ERR_UNSUPPORTED),
])
def test_validate_w8_rejects(kw, status):
    assert v8(**kw) == status


def test_w8_config_rejections_need_no_device():
    """A path other than AUTO / W8, or tile-only fields, are refused before any launch."""
    lib = sgr.load()
    cfg = sgr.make_config(path=sgr.SGR_PATH_TILE)
    rc = binding.skinny_gemm_residual_w8_ptr(A_, 3584, W_, 3584, S_, R_, 7168, Y_, 7168, 0, 7168, 3584,
                                             cfg, 0, 0)
    assert rc == sgr.SGR_OK  # M = 0: nothing to do, nothing checked further
    assert lib.sgr_validate_w8(None, 3584, None, 3584, None, None, 7168, None, 7168, 4, 7168, 3584) == sgr.SGR_ERR_NULL


# ------------------------------------------------------------ NVFP4-weight entry point (host-side checks only)
B_ = BASE + (5 << 32)


def v4(A=A_, lda=3584, Wq4=W_, ldw=1792, bs=B_, ldbs=224, R=R_, ldr=7168, Y=Y_, ldy=7168, M=4, N=7168, K=3584):
    return sgr.sgr_validate_w4_ptr(A, lda, Wq4, ldw, bs, ldbs, R, ldr, Y, ldy, M, N, K)


def test_validate_w4_accepts_good_arguments():
    assert v4() == sgr.SGR_OK
    assert v4(M=256, ldw=1808, ldbs=240) == sgr.SGR_OK   # padded code and scale rows (multiples of 16 bytes)
    assert v4(Y=R_) == sgr.SGR_OK                         # in-place residual
    assert v4(M=0, A=0, Wq4=0, bs=0, R=0, Y=0) == sgr.SGR_OK
    assert v4(K=0, A=0, Wq4=0, bs=0) == sgr.SGR_OK        # empty sum: Y = R
    assert v4(K=1056, lda=1056, ldw=528, ldbs=80) == sgr.SGR_OK  # 66 scales per row, read as 80 bytes
    assert v4(K=3592, lda=3592, ldw=1808, ldbs=240) == sgr.SGR_OK  # K not a multiple of 32: tensor-core kernel


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), sgr.SGR_ERR_SHAPE),
    (dict(K=3580, lda=3584), sgr.SGR_ERR_SHAPE),          # K not a multiple of 8
    (dict(Wq4=0), sgr.SGR_ERR_NULL),
    (dict(bs=0), sgr.SGR_ERR_NULL),
    (dict(ldw=1776), sgr.SGR_ERR_SHAPE),                  # fewer than K/2 bytes per code row
    (dict(K=1056, lda=1056, ldw=528, ldbs=66), sgr.SGR_ERR_SHAPE),  # scale rows not padded to 16 bytes
    (dict(ldw=1800), sgr.SGR_ERR_ALIGN),                  # row stride not a multiple of 16 bytes
    (dict(ldbs=232), sgr.SGR_ERR_ALIGN),
    (dict(Wq4=W_ + 8), sgr.SGR_ERR_ALIGN),
    (dict(bs=B_ + 4), sgr.SGR_ERR_ALIGN),
    (dict(Y=W_ + 4096), sgr.SGR_ERR_ALIAS),               # Y inside the codes
    (dict(Y=B_ + 4096), sgr.SGR_ERR_ALIAS),               # Y inside the scales
    (dict(Y=A_), sgr.SGR_ERR_ALIAS),
    (dict(Y=R_ + 16), sgr.SGR_ERR_ALIAS),
    (dict(ldbs=(1 << 36) + 16), sgr.SGR_ERR_UNSUPPORTED),
])
def test_validate_w4_rejects(kw, status):
    assert v4(**kw) == status


def test_w4_config_and_size_rejections_need_no_device():
    """A tile path, tile-only fields, M above 256, or a K the CUDA-core kernel
    cannot take on that path are refused before any launch (M = 0 is a no-op
    whatever the configuration)."""
    lib = sgr.load()
    cfg = sgr.make_config(path=sgr.SGR_PATH_TILE)
    assert binding.skinny_gemm_residual_w4_ptr(A_, 3584, W_, 1792, B_, 224, 1.0, R_, 7168, Y_, 7168, 0, 7168, 3584,
                                               cfg, 0, 0) == sgr.SGR_OK
    assert lib.sgr_validate_w4(None, 3584, None, 1792, None, 224, None, 7168, None, 7168, 4, 7168, 3584) == \
        sgr.SGR_ERR_NULL
    call = lambda M, K, c: binding.skinny_gemm_residual_w4_ptr(A_, K, W_, (K // 2 + 15) // 16 * 16, B_,
                                                                ((K + 15) // 16 + 15) // 16 * 16, 1.0, R_, 7168, Y_,
                                                                7168, M, 7168, K, c, 0, 0)
    assert call(4, 3584, cfg) == sgr.SGR_ERR_UNSUPPORTED                          # tile path
    assert call(4, 3584, sgr.make_config(k_split=2)) == sgr.SGR_ERR_UNSUPPORTED   # tile-only field
    assert call(257, 3584, None) == sgr.SGR_ERR_UNSUPPORTED                       # more than 256 tokens
    simt = sgr.make_config(path=sgr.SGR_PATH_SIMT)
    assert call(1, 7200, simt) == sgr.SGR_ERR_UNSUPPORTED                         # CUDA-core kernel: K <= 7168
    assert call(1, 3592, simt) == sgr.SGR_ERR_UNSUPPORTED                         # and whole 32-code vectors
