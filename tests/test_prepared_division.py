"""CPU check of the prepared exact division behind float16 and bfloat16
BatchNormalization and BiasPReluBN.

For a divisor shared by a row the engine forms r = RN(1/d) once and, per
element, q0 = RN(t r) followed by two corrections q <- RN(q + RN(t - q d) r)
(P. Markstein's final-correction scheme, twice); the argument beside the
kernels shows q2 == RN(t / d) for significands up to 2^24 - 5 within the
stated ranges.  A C restatement (tests/prepared_division.c) is checked here
against the IEEE quotient on random operands, on quotients built to lie next
to rounding midpoints (some within a few units of 2^-25 ulp), and on the
largest significands; a scheme without the corrections must be caught.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "prepared_division.c")


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("pd") / "libpd.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", SRC, "-o", so, "-lm"])
    L = ctypes.CDLL(so)
    p = ctypes.c_void_p
    L.pd_check.argtypes = [p, p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, p, p]
    L.pd_check.restype = None
    return L


def check(L, t, d, corrections=2, tlow=2.0 ** -100):
    t = np.ascontiguousarray(t, np.float32)
    d = np.ascontiguousarray(d, np.float32)
    counts = np.zeros(3, np.int64)
    bad = np.zeros(1, np.int64)
    L.pd_check(t.ctypes.data, d.ctypes.data, t.size, corrections, tlow, counts.ctypes.data,
               bad.ctypes.data)
    return counts, int(bad[0])


def floats(rng, n, emin, emax, sig=None):
    """Random binary32 values with exponents in [emin, emax] and random signs;
    sig: fixed significand fields (23 bits), else uniform."""
    e = rng.integers(emin, emax + 1, n) + 127
    m = rng.integers(0, 1 << 23, n) if sig is None else np.resize(np.asarray(sig), n)
    s = rng.integers(0, 2, n) << 31
    return (s | (e << 23) | m).astype(np.uint32).view(np.float32)


def near_midpoints(rng, n, d):
    """t such that t / d lies within a fraction of an ulp of a rounding midpoint
    of binary32: t = the float nearest to (q + ulp/2) d, and its neighbours."""
    q = np.abs(floats(rng, n, -30, 30))
    ulp = np.spacing(q).astype(np.float64)
    m = q.astype(np.float64) + ulp / 2
    base = (m * np.abs(d).astype(np.float64)).astype(np.float32)
    out = [base]
    for k in (1, 2):
        out.append(np.nextafter(base, np.float32(np.inf)))
        out.append(np.nextafter(base, np.float32(0)))
        base = out[-2]
    return np.concatenate(out), np.tile(d, 1 + 2 * 2)


def hardest_midpoints(rng, n):
    """(t, d) whose quotient lies within |e| / (2D) ulp of a rounding midpoint,
    e in {+-1, +-3, +-5}: for odd significands D, the odd 25-bit midpoint
    numerator M = e D^-1 mod 2^k makes M D = T 2^k + e with T a 24-bit integer,
    so t = T (scaled) and d = D (scaled) give a quotient e / D units of the
    midpoint numerator M away from the midpoint M / 2 (in ulps: e / (2D))."""
    ts, ds = [], []
    while len(ts) < n:
        D = int(rng.integers(1 << 22, 1 << 23)) * 2 + 1            # odd, in [2^23, 2^24)
        e = int(rng.choice([-5, -3, -1, 1, 3, 5]))
        for k in (24, 25):
            M = (e * pow(D, -1, 1 << k)) % (1 << k)
            if k == 24:
                M += 1 << 24
            if not (1 << 24) <= M < (1 << 25) or M % 2 == 0:
                continue
            P = M * D
            if (P - e) % (1 << k):
                continue
            T = (P - e) >> k
            if not (1 << 23) <= T < (1 << 24):
                continue
            sd, st = int(rng.integers(-20, 20)), int(rng.integers(-40, 40))
            ds.append(np.ldexp(np.float64(D), sd - 23))
            ts.append(np.ldexp(np.float64(T), st - 23) * (1 if rng.random() < 0.5 else -1))
    return np.array(ts[:n], np.float32), np.array(ds[:n], np.float32)


def test_random_quotients(lib):
    rng = np.random.default_rng(7)
    n = 4_000_000
    d = np.abs(floats(rng, n, -22, 22))
    t = floats(rng, n, -126, 127)
    counts, bad = check(lib, t, d)
    assert counts[2] == 0, ("kept a wrong quotient", counts, t[bad], d[bad])
    assert counts[0] > 0.5 * n, counts


def test_quotients_next_to_midpoints(lib):
    rng = np.random.default_rng(8)
    d = np.abs(floats(rng, 400_000, -20, 20))
    t, dd = near_midpoints(rng, d.size, d)
    counts, bad = check(lib, t, dd)
    assert counts[2] == 0, ("kept a wrong quotient", counts, t[bad], dd[bad])
    assert counts[0] > 0.9 * t.size, counts


def test_largest_significands(lib):
    """2^24 - 5 (the largest admitted) and its neighbours; larger ones are refused."""
    rng = np.random.default_rng(9)
    fields = np.arange((1 << 23) - 16, 1 << 23)                 # D = 2^24 - 16 .. 2^24 - 1
    d = np.abs(floats(rng, 200_000, -20, 20, sig=fields))
    for t, dd in (near_midpoints(rng, d.size, d), (floats(rng, d.size, -60, 60), d)):
        counts, bad = check(lib, t, dd)
        assert counts[2] == 0, ("kept a wrong quotient", counts, t[bad], dd[bad])
    big = np.abs(floats(rng, 1000, -20, 20, sig=np.arange((1 << 23) - 4, 1 << 23)))
    counts, _ = check(lib, floats(rng, 1000, -10, 10), big)
    assert counts[0] == 0 and counts[1] == 1000, counts


def test_zeros_and_extremes_are_refused(lib):
    t = np.array([0.0, -0.0, 1e-38, 3e38, np.inf, -np.inf, np.nan, 1.0], np.float32)
    d = np.array([1.5, 1.5, 1e5, 1e-5, 2.0, 2.0, 2.0, 2.0 ** 21], np.float32)
    counts, _ = check(lib, t, d)
    assert counts[0] == 0 and counts[1] == t.size, counts


def test_rows_whose_t_is_plus_zero_or_not_tiny(lib):
    """tlow = 0: +0 divides to +0 exactly; infinities and NaNs are still refused."""
    rng = np.random.default_rng(13)
    d = np.abs(floats(rng, 200_000, -20, 20))
    t = floats(rng, d.size, -99, 110)
    t[::7] = 0.0
    counts, bad = check(lib, t, d, tlow=0.0)
    assert counts[2] == 0, ("kept a wrong quotient", counts, t[bad], d[bad])
    zeros = np.zeros(1000, np.float32)
    dz = np.abs(floats(rng, 1000, -20, 19, sig=np.arange(0, (1 << 23) - 4, 8191)))
    counts, _ = check(lib, zeros, dz, tlow=0.0)
    assert counts[0] == 1000 and counts[2] == 0, counts
    counts, _ = check(lib, np.array([np.inf, -np.inf, np.nan], np.float32),
                      np.full(3, 1.5, np.float32), tlow=0.0)
    assert counts[0] == 0, counts


def test_quotients_within_a_few_units_of_a_midpoint(lib):
    t, d = hardest_midpoints(np.random.default_rng(11), 200_000)
    counts, bad = check(lib, t, d)
    assert counts[2] == 0, ("kept a wrong quotient", counts, t[bad], d[bad])
    assert counts[0] == t.size, counts


def test_a_missing_correction_is_caught(lib):
    """Planted mistake: keeping q0 = RN(t r) uncorrected gives wrong quotients
    next to midpoints.  (One correction is within (1/2 + 2^-22) ulp, which the
    argument does not take to the correct rounding; the engine makes two.)"""
    t, d = hardest_midpoints(np.random.default_rng(12), 200_000)
    counts, _ = check(lib, t, d, corrections=0)
    assert counts[2] > 0, counts
