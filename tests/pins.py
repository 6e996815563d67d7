"""Pins for the CPU oracle: checks that tie it to the definition of the
operation and to the mathematics, not to itself.

Each ``check_*`` takes a loaded oracle (``oracle.Oracle``) and raises
AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` runs them on builds with one planted
mistake each and expects at least one to fail.

Independent formulations used here:
  * exact rational arithmetic (fractions.Fraction) and a rounding to BF16 by
    bisection over the ordered BF16 grid (no frexp/ldexp, unlike the oracle);
  * hand-worked fixtures under tests/golden/;
  * special cases whose answer is a library rounding (torch float32 -> bf16,
    IEEE round-to-nearest-even) or an exact integer (numpy int64 matmul).
"""
from __future__ import annotations

import os
import struct
from fractions import Fraction

import numpy as np
import torch

from skinny_bf16_gemm_residual_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers
def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_value(pattern: int) -> Fraction:
    """Exact value of a finite BF16 bit pattern."""
    f = struct.unpack("<f", struct.pack("<I", (pattern & 0xFFFF) << 16))[0]
    return Fraction(f)


_POS_MAX = 0x7F7F


def rne_bf16_exact(x: Fraction) -> int:
    """Round an exact rational to BF16 (ties to even) by bisection on the grid.

    Positive finite patterns 0x0000..0x7F7F are ordered by value, so the two
    neighbours of |x| are found by binary search; the nearer wins, and a tie
    goes to the pattern with a zero last bit.  Above the largest finite value,
    the next grid point is 2^128 (infinity)."""
    if x == 0:
        return 0x0000
    sign = 0x8000 if x < 0 else 0x0000
    ax = abs(x)
    top = bf16_value(_POS_MAX)
    if ax >= top:
        nxt = Fraction(2) ** 128
        if ax - top < nxt - ax:
            return sign | _POS_MAX
        return sign | 0x7F80  # tie or above: the even neighbour is infinity
    lo, hi = 0, _POS_MAX  # invariant: value(lo) <= ax < value(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if bf16_value(mid) <= ax:
            lo = mid
        else:
            hi = mid
    dlo, dhi = ax - bf16_value(lo), bf16_value(hi) - ax
    if dlo < dhi:
        p = lo
    elif dhi < dlo:
        p = hi
    else:
        p = lo if lo % 2 == 0 else hi
    return sign | p


def exact_reference(A: np.ndarray, W: np.ndarray, R: np.ndarray) -> np.ndarray:
    """Brute force: Y[m,n] = rne(sum_k A[m,k] W[n,k] + R[m,n]) in exact rationals."""
    M, K = A.shape
    N = W.shape[0]
    a = [[bf16_value(int(v)) for v in row] for row in A]
    w = [[bf16_value(int(v)) for v in row] for row in W]
    out = np.empty((M, N), dtype=np.uint16)
    for m in range(M):
        for n in range(N):
            s = sum((a[m][k] * w[n][k] for k in range(K)), Fraction(0))
            out[m, n] = rne_bf16_exact(s + bf16_value(int(R[m, n])))
    return out


def load_rounding_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            x, y = line.split()
            rows.append((float.fromhex(x), int(y, 16)))
    return rows


def load_crafted_fixture():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "crafted_gemm.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                cur = {"name": line[5:].split(":", 1)[0]}
                cases.append(cur)
            elif ":" not in line:
                cur["M"], cur["N"], cur["K"] = (int(v) for v in line.split())
            else:
                key, vals = line.split(":", 1)
                vals = vals.split()
                if key == "Y":
                    cur["Y"] = np.array([int(v, 16) for v in vals], dtype=np.uint16)
                else:
                    f32 = np.array([float.fromhex(v) for v in vals], dtype=np.float32)
                    cur[key] = bits(torch.from_numpy(f32).to(torch.bfloat16))
    for c in cases:
        c["A"] = c["A"].reshape(c["M"], c["K"])
        c["W"] = c["W"].reshape(c["N"], c["K"])
        c["R"] = c["R"].reshape(c["M"], c["N"])
        c["Y"] = c["Y"].reshape(c["M"], c["N"])
    return cases


def _eq(got: np.ndarray, want: np.ndarray, what: str):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: "
                             f"got 0x{int(got[i]):04X} want 0x{int(want[i]):04X}")


def _library_round_f32(x: np.ndarray) -> np.ndarray:
    """float64 values that are exact in float32 -> BF16 via torch's float32
    conversion (IEEE round-to-nearest-even)."""
    f32 = x.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), x), "value not exact in float32"
    return bits(torch.from_numpy(f32).to(torch.bfloat16))


def _f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- pins
def check_rounding_fixture(orc):
    rows = load_rounding_fixture()
    got = orc.round_bf16(np.array([x for x, _ in rows]))
    want = np.array([y for _, y in rows], dtype=np.uint16)
    _eq(got, want, "BF16 round-to-nearest-even fixture")


def check_rounding_vs_exact_bisection(orc):
    """Random doubles near grid points and midpoints, checked against the
    bisection rounding on exact rationals."""
    rng = np.random.default_rng(1234)
    base = rng.integers(0x0001, 0x7F7F, 400)
    vals = []
    for p in base:
        v = float(bf16_value(int(p)))
        nxt = float(bf16_value(int(p) + 1))
        mid = (v + nxt) / 2
        for x in (v, mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf), (v + mid) / 2):
            vals.append(x)
            vals.append(-x)
    vals = np.array(vals, dtype=np.float64)
    got = orc.round_bf16(vals)
    want = np.array([rne_bf16_exact(Fraction(float(x))) for x in vals], dtype=np.uint16)
    _eq(got, want, "rounding vs exact bisection")


def check_crafted_fixture(orc):
    for c in load_crafted_fixture():
        _eq(orc.gemm_residual(c["A"], c["W"], c["R"], threads=1), c["Y"], f"crafted case {c['name']}")


def check_brute_force_exact(orc):
    """4x8x16 and a few other tiny shapes: oracle == exact rational brute force."""
    for (M, N, K, seed) in ((4, 8, 16, 1), (3, 5, 7, 2), (1, 1, 1, 3), (2, 9, 33, 4), (5, 3, 64, 5)):
        A = bits(inputs.random_bf16_bits((M, K), seed))
        W = bits(inputs.random_bf16_bits((N, K), seed + 100))
        R = bits(inputs.random_bf16_bits((M, N), seed + 200))
        _eq(orc.gemm_residual(A, W, R, threads=2), exact_reference(A, W, R),
            f"brute force {M}x{N}x{K}")


def check_unrounded_sum_vs_exact(orc):
    """The oracle's unrounded FP64 value of A . W^T + R against exact rationals.
    FP64 summation of K + 1 terms in order is within (K + 1) * 2^-53 of the
    sum of magnitudes (each product of two BF16 values is exact in FP64), far
    inside half a BF16 ulp, so a value that was already rounded to BF16, or
    one that drops or mis-signs a term, falls outside the bound.  With integer
    operands every step is exact and the values must be equal."""
    for (M, N, K, seed) in ((4, 8, 16, 61), (3, 5, 33, 62), (2, 7, 64, 63)):
        A = bits(inputs.random_bf16_bits((M, K), seed))
        W = bits(inputs.random_bf16_bits((N, K), seed + 100))
        R = bits(inputs.random_bf16_bits((M, N), seed + 200))
        t = orc.gemm_residual_f64(A, W, R, threads=2)
        a = [[bf16_value(int(v)) for v in row] for row in A]
        w = [[bf16_value(int(v)) for v in row] for row in W]
        far = 0
        for m in range(M):
            for n in range(N):
                terms = [a[m][k] * w[n][k] for k in range(K)] + [bf16_value(int(R[m, n]))]
                exact = sum(terms, Fraction(0))
                bound = Fraction(K + 1, 2 ** 53) * sum((abs(x) for x in terms), Fraction(0))
                assert abs(Fraction(float(t[m, n])) - exact) <= bound, \
                    f"unrounded sum {M}x{N}x{K} at ({m},{n}): {t[m, n]!r} vs {float(exact)!r}"
                far += abs(exact - bf16_value(rne_bf16_exact(exact))) > bound
        assert far > 0, "no element of the case separates rounded from unrounded values"
    Ai = inputs.integer_bf16((5, 24), -3, 3, 64)
    Wi = inputs.integer_bf16((6, 24), -3, 3, 65)
    Ri = inputs.integer_bf16((5, 6), -8, 8, 66)
    want = (Ai.to(torch.int64) @ Wi.to(torch.int64).T + Ri.to(torch.int64)).numpy().astype(np.float64)
    t = orc.gemm_residual_f64(bits(Ai), bits(Wi), bits(Ri))
    assert np.array_equal(t, want), "unrounded sum of integer operands is not exact"


def check_identity_weight(orc):
    """N = K and W = I: Y = bf16(A + R), a single library rounding."""
    K = 24
    A = bits(inputs.random_bf16_bits((5, K), 11, lo_exp=-4, hi_exp=4))
    R = bits(inputs.random_bf16_bits((5, K), 12, lo_exp=-4, hi_exp=4))
    W = bits(torch.eye(K, dtype=torch.bfloat16))
    want = _library_round_f32(_f64(A) + _f64(R))
    _eq(orc.gemm_residual(A, W, R), want, "identity W")


def check_one_hot_activation(orc):
    """A[m,:] = e_j(m): Y[m,n] = bf16(W[n, j(m)] + R[m,n])."""
    M, N, K = 6, 10, 12
    W = bits(inputs.random_bf16_bits((N, K), 21, lo_exp=-4, hi_exp=4))
    R = bits(inputs.random_bf16_bits((M, N), 22, lo_exp=-4, hi_exp=4))
    js = [(3 * m + 1) % K for m in range(M)]
    A_t = torch.zeros((M, K), dtype=torch.bfloat16)
    for m, j in enumerate(js):
        A_t[m, j] = 1.0
    A = bits(A_t)
    want = _library_round_f32(_f64(W)[:, js].T + _f64(R))
    _eq(orc.gemm_residual(A, W, R), want, "one-hot A")


def check_zero_operands(orc):
    """W = 0 or A = 0 leaves Y == R (R has no zeros, so no -0 question);
    R = 0 with integer A, W gives the exact integer product."""
    M, N, K = 3, 7, 9
    A = bits(inputs.random_bf16_bits((M, K), 31))
    W = bits(inputs.random_bf16_bits((N, K), 32))
    R = bits(inputs.random_bf16_bits((M, N), 33))
    zA = np.zeros_like(A)
    zW = np.zeros_like(W)
    _eq(orc.gemm_residual(A, zW, R), R, "W = 0")
    _eq(orc.gemm_residual(zA, W, R), R, "A = 0")
    Ai = inputs.integer_bf16((M, K), -3, 3, 34)
    Wi = inputs.integer_bf16((N, K), -3, 3, 35)
    prod = Ai.to(torch.int64) @ Wi.to(torch.int64).T
    want = bits(prod.to(torch.bfloat16))  # |prod| <= 81: exact
    _eq(orc.gemm_residual(bits(Ai), bits(Wi), np.zeros((M, N), np.uint16)), want, "R = 0")


def check_integer_exact(orc):
    """A, W in [-2,2], R in [-8,8], K <= 32: |y| <= 136, every step exact."""
    for (M, N, K, s) in ((16, 40, 32, 41), (1, 128, 32, 42), (7, 9, 5, 43)):
        Ai = inputs.integer_bf16((M, K), -2, 2, s)
        Wi = inputs.integer_bf16((N, K), -2, 2, s + 1)
        Ri = inputs.integer_bf16((M, N), -8, 8, s + 2)
        y = Ai.to(torch.int64) @ Wi.to(torch.int64).T + Ri.to(torch.int64)
        _eq(orc.gemm_residual(bits(Ai), bits(Wi), bits(Ri)), bits(y.to(torch.bfloat16)),
            f"integer-valued {M}x{N}x{K}")


def check_transpose_symmetry(orc):
    """With R = 0, swapping the roles of A and W transposes Y."""
    M, N, K = 4, 6, 20
    A = bits(inputs.random_bf16_bits((M, K), 51))
    W = bits(inputs.random_bf16_bits((N, K), 52))
    y1 = orc.gemm_residual(A, W, np.zeros((M, N), np.uint16))
    y2 = orc.gemm_residual(W, A, np.zeros((N, M), np.uint16))
    _eq(y1, np.ascontiguousarray(y2.T), "transpose symmetry")


def check_strided_rows(orc):
    """Row strides larger than the row width give the same result as a
    contiguous copy (the operand view is what is multiplied)."""
    M, N, K = 3, 5, 8
    A = bits(inputs.random_bf16_bits((M, 2 * K), 61))
    W = bits(inputs.random_bf16_bits((N, K), 62))
    R = bits(inputs.random_bf16_bits((M, 3 * N), 63))
    a_view, r_view = A[:, K:], R[:, N:2 * N]
    want = exact_reference(np.ascontiguousarray(a_view), W, np.ascontiguousarray(r_view))
    _eq(orc.gemm_residual(a_view, W, r_view), want, "strided operands")


# ------------------------------------------------------ low-bit weight pins
def e4m3_value(code: int) -> Fraction | None:
    """Exact value of an FP8 E4M3 code from its fields (None for NaN)."""
    s, e, f = code >> 7, (code >> 3) & 15, code & 7
    if e == 15 and f == 7:
        return None
    mag = Fraction(f, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(f, 8)) * Fraction(2) ** (e - 7)
    return -mag if s else mag


def load_e4m3_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            c, v = line.split()
            rows.append((int(c, 16), float("nan") if v == "nan" else float.fromhex(v)))
    return rows


def exact_reference_w8(A: np.ndarray, Wq: np.ndarray, scale: np.ndarray, R: np.ndarray) -> np.ndarray:
    """Brute force: Y[m,n] = rne(scale[n] * sum_k A[m,k] e4m3(Wq[n,k]) + R[m,n]) in exact rationals."""
    M, K = A.shape
    N = Wq.shape[0]
    out = np.empty((M, N), dtype=np.uint16)
    for m in range(M):
        for n in range(N):
            s = sum((bf16_value(int(A[m, k])) * e4m3_value(int(Wq[n, k])) for k in range(K)), Fraction(0))
            out[m, n] = rne_bf16_exact(Fraction(float(scale[n])) * s + bf16_value(int(R[m, n])))
    return out


def _same_float(got: np.ndarray, want: np.ndarray) -> bool:
    """Equal values, NaN matching NaN, and the sign of zero compared too."""
    both_nan = np.isnan(got) & np.isnan(want)
    same = (got == want) & (np.signbit(got) == np.signbit(want))
    return bool(np.all(both_nan | same))


def load_crafted_w8_fixture():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "crafted_w8.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                cur = {"name": line[5:].split(":", 1)[0]}
                cases.append(cur)
            elif ":" not in line:
                cur["M"], cur["N"], cur["K"] = (int(v) for v in line.split())
            else:
                key, vals = line.split(":", 1)
                vals = vals.split()
                if key == "Y":
                    cur["Y"] = np.array([int(v, 16) for v in vals], dtype=np.uint16)
                elif key == "Wq":
                    cur["Wq"] = np.array([int(v, 16) for v in vals], dtype=np.uint8)
                elif key == "scale":
                    cur["scale"] = np.array([float.fromhex(v) for v in vals], dtype=np.float32)
                else:
                    f32 = np.array([float.fromhex(v) for v in vals], dtype=np.float32)
                    cur[key] = bits(torch.from_numpy(f32).to(torch.bfloat16))
    for c in cases:
        c["A"] = c["A"].reshape(c["M"], c["K"])
        c["Wq"] = c["Wq"].reshape(c["N"], c["K"])
        c["R"] = c["R"].reshape(c["M"], c["N"])
        c["Y"] = c["Y"].reshape(c["M"], c["N"])
    return cases


def check_w8_crafted_fixture(orc):
    for c in load_crafted_w8_fixture():
        _eq(orc.gemm_residual_w8(c["A"], c["Wq"], c["scale"], c["R"], threads=1), c["Y"],
            f"crafted w8 case {c['name']}")
        _eq(exact_reference_w8(c["A"], c["Wq"], c["scale"], c["R"]), c["Y"],
            f"crafted w8 case {c['name']} (exact rationals)")


def check_e4m3_fixture(orc):
    rows = load_e4m3_fixture()
    got = orc.e4m3_to_double(np.array([c for c, _ in rows], dtype=np.uint8))
    want = np.array([v for _, v in rows])
    if not _same_float(got, want):
        bad = [(hex(c), g, w) for (c, w), g in zip(rows, got) if not _same_float(np.array([g]), np.array([w]))]
        raise AssertionError(f"E4M3 fixture mismatches (code, got, want): {bad[:4]}")


def check_e4m3_all_codes_vs_library(orc):
    """All 256 codes against torch's float8_e4m3fn -> float64 conversion and
    against the field formula above (signed zero included)."""
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_double(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if not _same_float(got, lib):
        raise AssertionError("E4M3 decode differs from torch.float8_e4m3fn")
    field = []
    for c in codes:
        v = e4m3_value(int(c))
        field.append(np.nan if v is None else np.copysign(float(abs(v)), -1.0 if c >= 128 else 1.0))
    if not _same_float(got, np.array(field)):
        raise AssertionError("E4M3 decode differs from the field formula")


def check_w8_brute_force_exact(orc):
    """Tiny shapes with every kind of code (zero, subnormal, normal, both
    signs) and random non-power-of-two scales: oracle == exact rationals."""
    for (M, N, K, seed) in ((3, 5, 8, 1), (1, 1, 1, 2), (2, 7, 19, 3), (4, 3, 32, 4)):
        A = bits(inputs.random_bf16_bits((M, K), seed + 300, lo_exp=-6, hi_exp=4))
        Wq = inputs.random_e4m3_codes((N, K), seed + 400).numpy()
        sc = inputs.random_scales(N, seed + 500).numpy()
        R = bits(inputs.random_bf16_bits((M, N), seed + 600, lo_exp=-6, hi_exp=6))
        _eq(orc.gemm_residual_w8(A, Wq, sc, R, threads=2), exact_reference_w8(A, Wq, sc, R),
            f"w8 brute force {M}x{N}x{K}")


def check_w8_subnormal_codes_exact(orc):
    """Only zero, subnormal and smallest-binade codes (exponent field 0 or 1),
    where the subnormal decoding decides the result."""
    M, N, K = 2, 6, 24
    A = bits(inputs.random_bf16_bits((M, K), 351, lo_exp=-2, hi_exp=2))
    Wq = (inputs.random_e4m3_codes((N, K), 352) & 0x8F).numpy()
    sc = inputs.random_scales(N, 353, lo_exp=4, hi_exp=8).numpy()
    R = bits(inputs.random_bf16_bits((M, N), 354, lo_exp=-4, hi_exp=0))
    _eq(orc.gemm_residual_w8(A, Wq, sc, R), exact_reference_w8(A, Wq, sc, R), "w8 subnormal codes")


def check_w8_unit_scale_is_bf16_gemm(orc):
    """scale = 1: every E4M3 value is a BF16 value (4 significant bits, exponent
    in range), so the low-bit variant equals the BF16 operation on the
    library-decoded weights."""
    M, N, K = 4, 33, 200
    A = bits(inputs.random_bf16_bits((M, K), 71, lo_exp=-4, hi_exp=4))
    R = bits(inputs.random_bf16_bits((M, N), 72, lo_exp=-2, hi_exp=6))
    Wq = inputs.random_e4m3_codes((N, K), 73)
    Wb = bits(Wq.view(torch.float8_e4m3fn).to(torch.bfloat16))
    ones = np.ones(N, dtype=np.float32)
    _eq(orc.gemm_residual_w8(A, Wq.numpy(), ones, R), orc.gemm_residual(A, Wb, R), "w8 unit scale")


def check_w8_power_of_two_scales(orc):
    """scale[n] = 2^j[n]: equals the BF16 operation on weights e4m3 * 2^j,
    which are still exact BF16 values."""
    M, N, K = 3, 16, 96
    A = bits(inputs.random_bf16_bits((M, K), 81, lo_exp=-4, hi_exp=4))
    R = bits(inputs.random_bf16_bits((M, N), 82))
    Wq = inputs.random_e4m3_codes((N, K), 83)
    j = np.arange(N) % 9 - 6
    sc = np.ldexp(np.ones(N), j).astype(np.float32)
    Wf = Wq.view(torch.float8_e4m3fn).to(torch.float64) * torch.from_numpy(np.ldexp(np.ones(N), j))[:, None]
    Wb = bits(Wf.to(torch.float32).to(torch.bfloat16))
    assert np.array_equal(_f64(Wb), Wf.numpy()), "scaled weights not exact in BF16"
    _eq(orc.gemm_residual_w8(A, Wq.numpy(), sc, R), orc.gemm_residual(A, Wb, R), "w8 power-of-two scales")


def check_w8_strided_rows(orc):
    M, N, K = 2, 4, 16
    A = bits(inputs.random_bf16_bits((M, 2 * K), 91))
    Wq = inputs.random_e4m3_codes((N, 3 * K), 92).numpy()
    sc = inputs.random_scales(N, 93).numpy()
    R = bits(inputs.random_bf16_bits((M, 2 * N), 94))
    a_v, w_v, r_v = A[:, K:], Wq[:, K:2 * K], R[:, N:]
    want = exact_reference_w8(np.ascontiguousarray(a_v), np.ascontiguousarray(w_v), sc, np.ascontiguousarray(r_v))
    _eq(orc.gemm_residual_w8(a_v, w_v, sc, r_v), want, "w8 strided operands")


def check_w8_sample_matches_full(orc):
    p = inputs.make_problem_w8(3, N=40, K=64, seed=95)
    full = orc.gemm_residual_w8(p.A, p.Wq, p.scale, p.R)
    ms = np.array([0, 2, 1, 2, 0])
    ns = np.array([0, 39, 17, 3, 21])
    _eq(orc.sample_w8(p.A, p.Wq, p.scale, p.R, ms, ns), full[ms, ns], "w8 sample")


# ------------------------------------------------------------ NVFP4 pins
def e2m1_value(code: int) -> Fraction:
    """Exact value of a 4-bit E2M1 code from its fields (OCP MX v1.0 FP4)."""
    s, e, f = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = Fraction(f, 2) if e == 0 else (1 + Fraction(f, 2)) * Fraction(2) ** (e - 1)
    return -mag if s else mag


def load_e2m1_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "e2m1_codes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float.fromhex(v)))
    return rows


def w4_codes(Wq4: np.ndarray) -> np.ndarray:
    """[N, K/2] packed bytes -> [N, K] 4-bit codes (element 2i = low nibble)."""
    out = np.empty((Wq4.shape[0], 2 * Wq4.shape[1]), dtype=np.uint8)
    out[:, 0::2] = Wq4 & 15
    out[:, 1::2] = Wq4 >> 4
    return out


def exact_reference_w4(A: np.ndarray, Wq4: np.ndarray, bs: np.ndarray, gs: float, R: np.ndarray) -> np.ndarray:
    """Brute force in exact rationals:
    Y[m,n] = rne(gs * sum_k A[m,k] e2m1(code[n,k]) e4m3(bs[n,k//16]) + R[m,n])."""
    M, K = A.shape
    N = Wq4.shape[0]
    codes = w4_codes(Wq4)
    out = np.empty((M, N), dtype=np.uint16)
    g = Fraction(float(np.float32(gs)))
    for m in range(M):
        for n in range(N):
            s = sum((bf16_value(int(A[m, k])) * e2m1_value(int(codes[n, k])) * e4m3_value(int(bs[n, k // 16]))
                     for k in range(K)), Fraction(0))
            out[m, n] = rne_bf16_exact(g * s + bf16_value(int(R[m, n])))
    return out


def load_crafted_w4_fixture():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "crafted_w4.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                cur = {"name": line[5:].split(":", 1)[0]}
                cases.append(cur)
            elif ":" not in line:
                cur["M"], cur["N"], cur["K"] = (int(v) for v in line.split())
            else:
                key, vals = line.split(":", 1)
                vals = vals.split()
                if key == "Y":
                    cur["Y"] = np.array([int(v, 16) for v in vals], dtype=np.uint16)
                elif key in ("Wq4", "bs"):
                    cur[key] = np.array([int(v, 16) for v in vals], dtype=np.uint8)
                elif key == "gs":
                    cur["gs"] = float(np.float32(float.fromhex(vals[0])))
                else:
                    f32 = np.array([float.fromhex(v) for v in vals], dtype=np.float32)
                    cur[key] = bits(torch.from_numpy(f32).to(torch.bfloat16))
    for c in cases:
        c["A"] = c["A"].reshape(c["M"], c["K"])
        c["Wq4"] = c["Wq4"].reshape(c["N"], c["K"] // 2)
        c["bs"] = c["bs"].reshape(c["N"], (c["K"] + 15) // 16)
        c["R"] = c["R"].reshape(c["M"], c["N"])
        c["Y"] = c["Y"].reshape(c["M"], c["N"])
    return cases


def check_e2m1_fixture(orc):
    rows = load_e2m1_fixture()
    assert [c for c, _ in rows] == list(range(16)), "the fixture lists every 4-bit code"
    got = orc.e2m1_to_double(np.array([c for c, _ in rows], dtype=np.uint8))
    want = np.array([v for _, v in rows])
    if not _same_float(got, want):
        raise AssertionError(f"E2M1 fixture mismatch: {list(zip(got, want))}")
    field = np.array([np.copysign(float(abs(e2m1_value(c))), -1.0 if c & 8 else 1.0) for c in range(16)])
    if not _same_float(got, field):
        raise AssertionError("E2M1 decode differs from the field formula")


def check_w4_crafted_fixture(orc):
    for c in load_crafted_w4_fixture():
        _eq(orc.gemm_residual_w4(c["A"], c["Wq4"], c["bs"], c["gs"], c["R"], threads=1), c["Y"],
            f"crafted w4 case {c['name']}")
        _eq(exact_reference_w4(c["A"], c["Wq4"], c["bs"], c["gs"], c["R"]), c["Y"],
            f"crafted w4 case {c['name']} (exact rationals)")


def check_w4_brute_force_exact(orc):
    """Tiny shapes with every code, random non-NaN block scales of both signs,
    a random tensor scale, and K not a multiple of 16 (a partial last block):
    oracle == exact rationals."""
    for (M, N, K, seed) in ((2, 3, 32, 1), (1, 2, 48, 2), (3, 2, 16, 3), (2, 4, 2, 4), (1, 3, 38, 5)):
        A = bits(inputs.random_bf16_bits((M, K), seed + 700, lo_exp=-6, hi_exp=4))
        Wq4 = inputs.random_e2m1_bytes((N, K // 2), seed + 710).numpy()
        bs = inputs.random_e4m3_codes((N, (K + 15) // 16), seed + 720).numpy()
        gs = float(inputs.random_scales(1, seed + 730, lo_exp=-4, hi_exp=4)[0])
        R = bits(inputs.random_bf16_bits((M, N), seed + 740, lo_exp=-6, hi_exp=6))
        _eq(orc.gemm_residual_w4(A, Wq4, bs, gs, R, threads=2), exact_reference_w4(A, Wq4, bs, gs, R),
            f"w4 brute force {M}x{N}x{K}")


def _w4_decoded_bf16(Wq4: np.ndarray, bs: np.ndarray, gs: float) -> np.ndarray:
    """e2m1(code) * e4m3(block scale) * gs as BF16 bits, built with torch's
    float8_e4m3fn conversion and a table of the 16 E2M1 values; the caller
    picks scales that keep every product exact in BF16."""
    table = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0],
                         dtype=torch.float64)
    codes = torch.from_numpy(w4_codes(Wq4).astype(np.int64))
    K = codes.shape[1]
    sc = torch.from_numpy(bs).view(torch.float8_e4m3fn).to(torch.float64)
    sc_k = sc.repeat_interleave(16, dim=1)[:, :K]
    Wf = table[codes] * sc_k * float(gs)
    Wb = Wf.to(torch.float32).to(torch.bfloat16)
    assert torch.equal(Wb.to(torch.float64), Wf), "decoded weights not exact in BF16"
    return bits(Wb)


def check_w4_unit_scales_is_bf16_gemm(orc):
    """All block scales 1 and gs = 1: every E2M1 value is a BF16 value, so the
    NVFP4 variant equals the pinned BF16 operation on the decoded weights."""
    M, N, K = 4, 21, 160
    A = bits(inputs.random_bf16_bits((M, K), 761, lo_exp=-4, hi_exp=4))
    R = bits(inputs.random_bf16_bits((M, N), 762, lo_exp=-2, hi_exp=6))
    Wq4 = inputs.random_e2m1_bytes((N, K // 2), 763).numpy()
    bs = np.full((N, K // 16), 0x38, dtype=np.uint8)
    _eq(orc.gemm_residual_w4(A, Wq4, bs, 1.0, R), orc.gemm_residual(A, _w4_decoded_bf16(Wq4, bs, 1.0), R),
        "w4 unit scales")


def check_w4_block_scales_as_bf16_gemm(orc):
    """Power-of-two block scales (different per block and row) and a
    power-of-two gs: equals the BF16 operation on e2m1 * scale * gs, which
    pins the block indexing (k // 16) and the nibble order independently."""
    M, N, K = 3, 12, 96
    A = bits(inputs.random_bf16_bits((M, K), 771, lo_exp=-4, hi_exp=4))
    R = bits(inputs.random_bf16_bits((M, N), 772))
    Wq4 = inputs.random_e2m1_bytes((N, K // 2), 773).numpy()
    g = torch.Generator().manual_seed(774)
    e = torch.randint(-6, 7, (N, K // 16), generator=g)
    bs = torch.pow(2.0, e.to(torch.float64)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    gs = 0.25
    _eq(orc.gemm_residual_w4(A, Wq4, bs, gs, R), orc.gemm_residual(A, _w4_decoded_bf16(Wq4, bs, gs), R),
        "w4 block scales")


def check_w4_strided_rows(orc):
    M, N, K = 2, 3, 32
    A = bits(inputs.random_bf16_bits((M, 2 * K), 781))
    Wq4 = inputs.random_e2m1_bytes((N, K), 782).numpy()            # row stride K bytes, codes in the second half
    bs = inputs.random_e4m3_codes((N, 4), 783).numpy()             # row stride 4, scales in columns 2-3
    R = bits(inputs.random_bf16_bits((M, 2 * N), 784))
    a_v, w_v, b_v, r_v = A[:, K:], Wq4[:, K // 2:], bs[:, 2:], R[:, N:]
    want = exact_reference_w4(np.ascontiguousarray(a_v), np.ascontiguousarray(w_v), np.ascontiguousarray(b_v),
                              1.5, np.ascontiguousarray(r_v))
    _eq(orc.gemm_residual_w4(a_v, w_v, b_v, 1.5, r_v), want, "w4 strided operands")


def check_w4_sample_matches_full(orc):
    p = inputs.make_problem_w4(3, N=40, K=64, seed=95)
    full = orc.gemm_residual_w4(p.A, p.Wq4, p.bs, p.gs, p.R)
    ms = np.array([0, 2, 1, 2, 0])
    ns = np.array([0, 39, 17, 3, 21])
    _eq(orc.sample_w4(p.A, p.Wq4, p.bs, p.gs, p.R, ms, ns), full[ms, ns], "w4 sample")


ALL_CHECKS = [
    check_rounding_fixture,
    check_rounding_vs_exact_bisection,
    check_crafted_fixture,
    check_brute_force_exact,
    check_unrounded_sum_vs_exact,
    check_identity_weight,
    check_one_hot_activation,
    check_zero_operands,
    check_integer_exact,
    check_transpose_symmetry,
    check_strided_rows,
    check_e4m3_fixture,
    check_e4m3_all_codes_vs_library,
    check_w8_crafted_fixture,
    check_w8_brute_force_exact,
    check_w8_subnormal_codes_exact,
    check_w8_unit_scale_is_bf16_gemm,
    check_w8_power_of_two_scales,
    check_w8_strided_rows,
    check_w8_sample_matches_full,
    check_e2m1_fixture,
    check_w4_crafted_fixture,
    check_w4_brute_force_exact,
    check_w4_unit_scales_is_bf16_gemm,
    check_w4_block_scales_as_bf16_gemm,
    check_w4_strided_rows,
    check_w4_sample_matches_full,
]
