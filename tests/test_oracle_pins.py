"""Pins of the oracle against things other than itself (CPU only).

Each test checks the oracle against a library routine that does not share the
oracle's code (numpy / torch ufuncs, Python integers, exact rational
arithmetic with ``fractions``, arbitrary precision ``mpmath``), a closed form
or worked table under ``tests/golden/`` (each with its citation), an identity,
or brute force over tiny shapes.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import datagen
import oracle
from conftest import assert_bits_equal, ulp_distance

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def f32(*v):
    return np.array(v, dtype=np.float32)


def bf16_bits(x_f32):
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def bf16_to_f32(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .float().numpy()


SPECIALS = f32(0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 1.17549435e-38,
               3.4028235e38, -3.4028235e38, 65504.0, 65520.0, 6.1035156e-05, 5.9604645e-08,
               2.9802322e-08, 0.5, 3.0, -7.0, 1e30, 1e-30)


def float_corpus(n, seed):
    """Random float32 bit patterns (all exponents) plus values of moderate size and specials."""
    bits = datagen.raw_u32(seed, 0, n).view(np.float32)
    mid = datagen.normal(seed, 1, n) * np.float32(100.0)
    return np.concatenate([bits, mid, SPECIALS])


# --------------------------------------------------------------------------- conversions

def stratified_f32_bits():
    """All 2^16 upper halves times low halves that sit on and around every rounding boundary."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x3000, 0x7FFF,
                     0x8000, 0x8001, 0xC000, 0xE000, 0xF000, 0xFFFF, 0x5A5A], dtype=np.uint32)
    rnd = datagen.raw_u32(7, 0, 16) & 0xFFFF
    lows = np.concatenate([lows, rnd.astype(np.uint32)])
    return (hi[:, None] | lows[None, :]).reshape(-1).view(np.float32)


def test_half_widening_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.f16_bits_to_f32(bits)
    want = bits.view(np.float16).astype(np.float32)
    assert_bits_equal(got, want, "float32", "half->float")


def test_bf16_widening_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.bf16_bits_to_f32(bits)
    want = bf16_to_f32(bits)
    assert_bits_equal(got, want, "float32", "bf16->float")


def test_half_narrowing_matches_numpy():
    x = stratified_f32_bits()
    got = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert_bits_equal(got.view(np.float16), want.view(np.float16), "float16", "float->half")


def test_bf16_narrowing_matches_torch():
    x = stratified_f32_bits()
    got = oracle.f32_to_bf16_bits(x)
    want = bf16_bits(x)
    assert_bits_equal(got, want, "bfloat16", "float->bf16")


# --------------------------------------------------------------------------- broadcasting

def all_small_shapes():
    shapes = [()]
    for r in (1, 2, 3):
        for flat in range(4 ** r):
            shapes.append(tuple((flat // 4 ** k) % 4 for k in range(r))[::-1])
    return shapes


def test_broadcast_shape_brute_force():
    shapes = all_small_shapes()
    assert len(shapes) == 85
    for sa in shapes:
        for sb in shapes:
            try:
                want = np.broadcast_shapes(sa, sb)
            except ValueError:
                want = None
            try:
                got = oracle.output_shape("Add", sa, sb)
            except ValueError as e:
                assert str(e) == "incompatible_shapes"
                got = None
            assert got == want, (sa, sb, got, want)


def test_broadcast_values_brute_force():
    """Every compatible pair of tiny shapes: oracle Add/Sub == numpy broadcasting, bit for bit."""
    shapes = all_small_shapes()
    for sa in shapes:
        for sb in shapes:
            try:
                np.broadcast_shapes(sa, sb)
            except ValueError:
                continue
            a = datagen.make("uniform", "float32", sa, 0, 0)
            b = datagen.make("uniform", "float32", sb, 0, 1)
            for op, fn in (("Add", np.add), ("Sub", np.subtract)):
                got, st = oracle.run(op, a, b, "float32")
                assert st == 0
                assert_bits_equal(got, fn(a, b), "float32", "%s %s %s" % (op, sa, sb))


def test_offsets_match_numpy_index_mapping():
    sa, sb = (2, 1, 4, 1), (3, 1, 5)
    out_shape = np.broadcast_shapes(sa, sb)
    n = int(np.prod(out_shape))
    ia = np.broadcast_to(np.arange(np.prod(sa)).reshape(sa), out_shape).reshape(-1)
    ib = np.broadcast_to(np.arange(np.prod(sb)).reshape(sb), out_shape).reshape(-1)
    oa, ob = oracle.offsets(sa, sb, np.arange(n))
    assert (oa == ia).all() and (ob == ib).all()


def test_empty_dims_do_no_work():
    """numel 0: no element is read (NULL inputs are fine) and the output is untouched."""
    lib = oracle._load()
    sa = np.array([0, 3], np.int64)
    sb = np.array([3], np.int64)
    st = np.zeros(1, np.uint32)
    rc = lib.oracle_eval(oracle.OPS.index("Div"), oracle.DTYPES.index("int32"), 0, 0, 0.0, 1, 1,
                         sa.ctypes.data, 2, sb.ctypes.data, 1, None, None, None, None, 0,
                         st.ctypes.data)
    assert rc == 0 and st[0] == 0
    out, st2 = oracle.run("Add", np.zeros((2, 0, 3), np.float32), np.zeros((1, 3), np.float32),
                          "float32")
    assert out.shape == (2, 0, 3) and st2 == 0


def test_coalescing_and_unit_dims_do_not_change_results():
    x = datagen.make("normal", "bfloat16", (8, 4, 16, 16), 2, 0)
    b = datagen.make("uniform", "bfloat16", (4, 1, 1), 2, 1, lo=-0.5, hi=0.5)
    full, _ = oracle.run("Add", x, b, "bfloat16")
    merged, _ = oracle.run("Add", x.reshape(8, 4, 256), b.reshape(4, 1), "bfloat16")
    unit, _ = oracle.run("Add", x.reshape(1, 8, 4, 1, 16, 16), b.reshape(1, 4, 1, 1, 1),
                         "bfloat16")
    assert full.tobytes() == merged.tobytes() == unit.tobytes()


# --------------------------------------------------------------------------- float arithmetic

@pytest.mark.parametrize("op,fn", [("Add", np.add), ("Sub", np.subtract), ("Mul", np.multiply),
                                   ("Div", np.divide)])
def test_f32_arith_matches_numpy(op, fn):
    a = float_corpus(20000, 11)
    b = float_corpus(20000, 12)
    b = np.roll(b, 7)
    got, st = oracle.run(op, a, b, "float32")
    with np.errstate(all="ignore"):
        want = fn(a, b)
    assert st == 0
    assert_bits_equal(got, want, "float32", op)


@pytest.mark.parametrize("op,fn", [("Add", np.add), ("Sub", np.subtract), ("Mul", np.multiply),
                                   ("Div", np.divide), ("Mod", np.remainder)])
def test_f16_arith_matches_numpy_half(op, fn):
    """numpy float16 ufuncs widen to float, operate and round once: the same semantics."""
    a = np.concatenate([datagen.raw_u32(13, 0, 30000).astype(np.uint16).view(np.float16),
                        datagen.make("normal", "float16", (30000,), 13, 1)])
    b = np.concatenate([datagen.raw_u32(13, 2, 30000).astype(np.uint16).view(np.float16),
                        datagen.make("normal", "float16", (30000,), 13, 3)])
    got, st = oracle.run(op, a, b, "float16")
    with np.errstate(all="ignore"):
        want = fn(a, b)
    assert_bits_equal(got, want, "float16", op)


@pytest.mark.parametrize("op,fn", [("Add", torch.add), ("Sub", torch.sub), ("Mul", torch.mul),
                                   ("Div", torch.div)])
def test_bf16_arith_matches_torch(op, fn):
    a = np.concatenate([datagen.raw_u32(14, 0, 30000).astype(np.uint16),
                        datagen.make("normal", "bfloat16", (30000,), 14, 1)])
    b = np.concatenate([datagen.raw_u32(14, 2, 30000).astype(np.uint16),
                        datagen.make("normal", "bfloat16", (30000,), 14, 3)])
    got, _ = oracle.run(op, a, b, "bfloat16")
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    want = fn(ta, tb).view(torch.int16).numpy().view(np.uint16)
    assert_bits_equal(got, want, "bfloat16", op)


def test_f32_identities():
    a = float_corpus(5000, 15)
    b = np.roll(float_corpus(5000, 16), 3)
    run = lambda op, x, y: oracle.run(op, x, y, "float32")[0]
    negzero = f32(-0.0).reshape(())
    one = f32(1.0).reshape(())
    assert_bits_equal(run("Add", a, negzero), a, "float32", "A + (-0) == A")
    assert_bits_equal(run("Mul", a, one), a, "float32", "A * 1 == A")
    assert_bits_equal(run("Div", a, one), a, "float32", "A / 1 == A")
    assert_bits_equal(run("Add", a, b), run("Add", b, a), "float32", "Add commutes")
    assert_bits_equal(run("Mul", a, b), run("Mul", b, a), "float32", "Mul commutes")
    assert_bits_equal(run("Sub", a, b), run("Add", a, -b), "float32", "A - B == A + (-B)")
    # A + (+0) is not an identity: -0 + +0 = +0
    assert run("Add", f32(-0.0), f32(0.0)).view(np.uint32)[0] == 0


# --------------------------------------------------------------------------- Mod

def rn32(x: Fraction) -> float:
    """Round an exact rational to binary32, nearest, ties to even (subnormals, overflow)."""
    if x == 0:
        return 0.0
    sign = -1.0 if x < 0 else 1.0
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 23)
    m = x / quantum
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * quantum
    if val >= Fraction(2) ** 128:
        return sign * math.inf
    return sign * float(val)


def exact_mod(a: float, b: float, fmod_flag: int) -> float:
    """Mod from exact rationals: truncated remainder, then the floor rule of opset 28."""
    fa, fb = Fraction(a), Fraction(b)
    q = fa / fb
    t = q.numerator // q.denominator if q >= 0 else -((-q.numerator) // q.denominator)
    r = fa - t * fb
    if fmod_flag:
        return math.copysign(0.0, a) if r == 0 else float(r)
    if r == 0:
        return math.copysign(0.0, b)
    if (r < 0) != (fb < 0):
        return rn32(r + fb)
    return float(r)


def mod_inputs(n, seed):
    a = np.concatenate([datagen.uniform_zeros(seed, 0, n, -100, 100, 0.01),
                        datagen.raw_u32(seed, 2, n).view(np.float32)])
    b = np.concatenate([datagen.uniform_reject(seed, 1, n, -7, 7, 0.01),
                        datagen.raw_u32(seed, 3, n).view(np.float32)])
    ok = np.isfinite(a) & np.isfinite(b) & (b != 0)
    return a[ok], b[ok]


@pytest.mark.parametrize("fmod_flag", [0, 1])
def test_f32_mod_exact_rational(fmod_flag):
    a, b = mod_inputs(3000, 21)
    got, st = oracle.run("Mod", a, b, "float32", fmod=fmod_flag)
    want = np.array([exact_mod(float(x), float(y), fmod_flag) for x, y in zip(a, b)], np.float32)
    assert st == 0
    assert_bits_equal(got, want, "float32", "Mod fmod=%d" % fmod_flag)


def test_f32_mod_matches_numpy_remainder():
    """numpy.remainder is the floor remainder with a divisor-signed zero (fmod=0)."""
    a = float_corpus(20000, 22)
    b = np.roll(float_corpus(20000, 23), 5)
    got, _ = oracle.run("Mod", a, b, "float32", fmod=0)
    with np.errstate(all="ignore"):
        want = np.remainder(a, b)
    assert_bits_equal(got, want, "float32", "Mod fmod=0 vs numpy.remainder")


def test_mod_sign_table():
    for dtype, a, b, fm, want in read_golden("mod_sign_rules.txt"):
        fm = int(fm)
        if dtype in ("float32", "float16", "bfloat16"):
            av, bv = f32(float(a)), f32(float(b))
            if dtype == "float16":
                av, bv = av.astype(np.float16), bv.astype(np.float16)
            elif dtype == "bfloat16":
                av, bv = bf16_bits(av), bf16_bits(bv)
            got, _ = oracle.run("Mod", av, bv, dtype, fmod=fm)
            g = got.astype(np.float32) if dtype == "float16" else \
                bf16_to_f32(got) if dtype == "bfloat16" else got
            w = float(want)
            assert g[0] == w and math.copysign(1, g[0]) == math.copysign(1, w), \
                (dtype, a, b, fm, g[0], w)
        else:
            st = datagen.STORAGE[dtype]
            got, _ = oracle.run("Mod", np.array([int(a)]).astype(st), np.array([int(b)]).astype(st),
                                dtype, fmod=fm)
            assert int(got[0]) == int(want), (dtype, a, b, fm, got[0])


def test_mod_specials():
    nan, inf = np.nan, np.inf
    a = f32(nan, inf, -inf, 5.0, 5.0, 5.0, -5.0, 5.0, -0.0)
    b = f32(2.0, 2.0, 2.0, 0.0, -0.0, nan, inf, -inf, inf)
    g0, _ = oracle.run("Mod", a, b, "float32", fmod=0)
    g1, _ = oracle.run("Mod", a, b, "float32", fmod=1)
    assert np.isnan(g0[:6]).all() and np.isnan(g1[:6]).all()
    # fmod(a, +-inf) = a; the floor rule then moves a sign mismatch to the divisor
    assert g1[6] == -5.0 and g1[7] == 5.0
    assert g0[6] == inf and g0[7] == -inf
    assert g0[8] == 0.0 and not math.copysign(1, g0[8]) < 0
    assert g1[8] == 0.0 and math.copysign(1, g1[8]) < 0


# --------------------------------------------------------------------------- integers

INT_LIMITS = {"int32": (-(1 << 31), (1 << 31) - 1), "int64": (-(1 << 63), (1 << 63) - 1),
              "uint8": (0, 255), "uint32": (0, (1 << 32) - 1),
              "int8": (-128, 127), "int16": (-(1 << 15), (1 << 15) - 1),
              "uint16": (0, (1 << 16) - 1), "uint64": (0, (1 << 64) - 1)}
ALL_INTS = ["int32", "int64", "uint8", "uint32", "int8", "int16", "uint16", "uint64"]


def wrap(v, dtype):
    lo, hi = INT_LIMITS[dtype]
    m = hi - lo + 1
    return (v - lo) % m + lo


def int_pairs(dtype):
    lo, hi = INT_LIMITS[dtype]
    small = list(range(max(lo, -40), min(hi, 40) + 1))
    edges = [lo, lo + 1, hi, hi - 1, 0, 1, 2, 3, 7, 255, 256]
    edges += [lo // 2, hi // 3] if dtype != "uint8" else [128, 129]
    vals = sorted(set(v for v in small + edges if lo <= v <= hi))
    a, b = np.meshgrid(np.array(vals, dtype=object), np.array(vals, dtype=object))
    return a.reshape(-1), b.reshape(-1)


def trunc_div(a, b):
    q = abs(a) // abs(b)
    return q if (a >= 0) == (b >= 0) else -q


@pytest.mark.parametrize("dtype", ALL_INTS)
def test_int_arith_matches_python_integers(dtype):
    a, b = int_pairs(dtype)
    st_t = datagen.STORAGE[dtype]
    A = np.array([int(x) for x in a], dtype=object).astype(st_t)
    B = np.array([int(x) for x in b], dtype=object).astype(st_t)
    nz = b != 0
    for op in ("Add", "Sub", "Mul", "Div", "Mod", "BitwiseAnd", "BitwiseOr", "BitwiseXor"):
        fmods = (0, 1) if op == "Mod" else (0,)
        for fm in fmods:
            got, st = oracle.run(op, A, B, dtype, fmod=fm)
            want = []
            for x, y in zip(a, b):
                x, y = int(x), int(y)
                if op == "Add": v = x + y
                elif op == "Sub": v = x - y
                elif op == "Mul": v = x * y
                elif op == "Div": v = trunc_div(x, y) if y else 0
                elif op == "Mod":
                    if y == 0: v = 0
                    elif fm: v = x - trunc_div(x, y) * y
                    else: v = x % y
                elif op == "BitwiseAnd": v = (x & y)
                elif op == "BitwiseOr": v = (x | y)
                else: v = (x ^ y)
                want.append(wrap(v, dtype))
            want = np.array(want, dtype=object).astype(st_t)
            assert (got == want).all(), (op, fm, dtype)
            if op in ("Div", "Mod"):
                assert st == (0 if nz.all() else oracle.STATUS_DIV_BY_ZERO)


# --------------------------------------------------------------------------- ncnn binaryop extras
# ncnn operators.md, binaryop: operation types 4 = MAX, 5 = MIN, 7 = RSUB, 8 = RDIV.

def _no_zero_pairs(a, b):
    """Drop pairs where both are zeros: numpy's maximum/minimum do not order -0 and +0."""
    keep = ~((a == 0) & (b == 0))
    return a[keep], b[keep]


@pytest.mark.parametrize("dtype", ["float32", "float16"])
def test_max_min_match_numpy(dtype):
    """numpy.maximum / numpy.minimum also return NaN for a NaN operand."""
    if dtype == "float32":
        a, b = float_corpus(20000, 21), np.roll(float_corpus(20000, 22), 5)
    else:
        a = np.concatenate([datagen.raw_u32(23, 0, 30000).astype(np.uint16).view(np.float16),
                            datagen.make("normal", "float16", (30000,), 23, 1)])
        b = np.concatenate([datagen.raw_u32(23, 2, 30000).astype(np.uint16).view(np.float16),
                            datagen.make("normal", "float16", (30000,), 23, 3)])
    b[::11] = a[::11]                                        # equal pairs
    a, b = _no_zero_pairs(a, b)
    for op, fn in (("Max", np.maximum), ("Min", np.minimum)):
        got, st = oracle.run(op, a, b, dtype)
        assert st == 0
        assert_bits_equal(got, fn(a, b), dtype, op)


def test_max_min_match_torch_bf16():
    a = np.concatenate([datagen.raw_u32(24, 0, 30000).astype(np.uint16),
                        datagen.make("normal", "bfloat16", (30000,), 24, 1)])
    b = np.concatenate([datagen.raw_u32(24, 2, 30000).astype(np.uint16),
                        datagen.make("normal", "bfloat16", (30000,), 24, 3)])
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    keep = (~((ta == 0) & (tb == 0))).numpy()
    a, b, ta, tb = a[keep], b[keep], ta[keep], tb[keep]
    for op, fn in (("Max", torch.maximum), ("Min", torch.minimum)):
        got, _ = oracle.run(op, a, b, "bfloat16")
        want = fn(ta, tb).view(torch.int16).numpy().view(np.uint16)
        assert_bits_equal(got, want, "bfloat16", op)


def test_max_min_signed_zero_and_nan():
    """Closed forms of the reading (IEEE 754-2019 maximum / minimum): +0 counts as
    larger than -0, and a NaN operand on either side gives NaN."""
    a = f32(0.0, -0.0, -0.0, 0.0, np.nan, 1.0, -np.inf, np.inf, 3.0)
    b = f32(-0.0, 0.0, -0.0, 0.0, 1.0, np.nan, 5.0, 5.0, 3.0)
    got, _ = oracle.run("Max", a, b, "float32")
    assert_bits_equal(got, f32(0.0, 0.0, -0.0, 0.0, np.nan, np.nan, 5.0, np.inf, 3.0), "float32")
    got, _ = oracle.run("Min", a, b, "float32")
    assert_bits_equal(got, f32(-0.0, -0.0, -0.0, 0.0, np.nan, np.nan, -np.inf, 5.0, 3.0),
                      "float32")


@pytest.mark.parametrize("dtype", ALL_INTS)
def test_int_max_min_rsub_rdiv_match_python_integers(dtype):
    a, b = int_pairs(dtype)
    st_t = datagen.STORAGE[dtype]
    A = np.array([int(x) for x in a], dtype=object).astype(st_t)
    B = np.array([int(x) for x in b], dtype=object).astype(st_t)
    for op in ("Max", "Min", "RSub", "RDiv"):
        got, st = oracle.run(op, A, B, dtype)
        want = []
        for x, y in zip(a, b):
            x, y = int(x), int(y)
            if op == "Max": v = max(x, y)
            elif op == "Min": v = min(x, y)
            elif op == "RSub": v = y - x
            else: v = trunc_div(y, x) if x else 0
            want.append(wrap(v, dtype))
        want = np.array(want, dtype=object).astype(st_t)
        assert (got == want).all(), (op, dtype)
        if op == "RDiv":
            assert st == (oracle.STATUS_DIV_BY_ZERO if (a == 0).any() else 0)
        else:
            assert st == 0


@pytest.mark.parametrize("op,fn", [("RSub", np.subtract), ("RDiv", np.divide)])
@pytest.mark.parametrize("dtype", ["float32", "float16"])
def test_rsub_rdiv_are_numpy_with_operands_reversed(op, fn, dtype):
    if dtype == "float32":
        a, b = float_corpus(20000, 25), np.roll(float_corpus(20000, 26), 3)
    else:
        a = datagen.raw_u32(27, 0, 30000).astype(np.uint16).view(np.float16)
        b = datagen.raw_u32(27, 1, 30000).astype(np.uint16).view(np.float16)
    got, st = oracle.run(op, a, b, dtype)
    with np.errstate(all="ignore"):
        want = fn(b, a)
    assert st == 0
    assert_bits_equal(got, want, dtype, op)


def test_int_division_by_zero_sets_status():
    a = np.array([5, 7, -9], np.int32)
    _, st = oracle.run("Div", a, np.array([1, 0, 2], np.int32), "int32")
    assert st == oracle.STATUS_DIV_BY_ZERO
    _, st = oracle.run("Mod", a, np.array([1, 3, 2], np.int32), "int32")
    assert st == 0


@pytest.mark.parametrize("dtype", ["uint8", "uint16", "uint32", "uint64"])
def test_bitshift_matches_numpy(dtype):
    w = 8 * np.dtype(datagen.STORAGE[dtype]).itemsize
    a = datagen.make("bits", dtype, (4096,), 5, 0)
    for s in range(w):
        b = np.full(a.shape, s, datagen.STORAGE[dtype])
        gl, st_l = oracle.run("BitShift", a, b, dtype, direction=0)
        gr, st_r = oracle.run("BitShift", a, b, dtype, direction=1)
        assert st_l == 0 and st_r == 0
        assert (gl == np.left_shift(a, b)).all() and (gr == np.right_shift(a, b)).all()
    _, st = oracle.run("BitShift", a, np.full(a.shape, w, datagen.STORAGE[dtype]), dtype,
                       direction=1)
    assert st == oracle.STATUS_SHIFT_RANGE
    _, st = oracle.run("BitShift", a, np.full(a.shape, w - 1, datagen.STORAGE[dtype]), dtype)
    assert st == 0


@pytest.mark.parametrize("dtype", ["int32", "int64"])
def test_int_pow_matches_python(dtype):
    st_t = datagen.STORAGE[dtype]
    bases = list(range(-12, 13)) + [INT_LIMITS[dtype][0], INT_LIMITS[dtype][1], 3 ** 19]
    exps = list(range(0, 70))
    a = np.array([x for x in bases for _ in exps], dtype=object)
    b = np.array([y for _ in bases for y in exps], dtype=object)
    got, st = oracle.run("Pow", a.astype(st_t), b.astype(st_t), dtype)
    want = np.array([wrap(pow(int(x), int(y)), dtype) for x, y in zip(a, b)],
                    dtype=object).astype(st_t)
    assert st == 0 and (got == want).all()


@pytest.mark.parametrize("dtype", ["int32", "int64"])
def test_int_pow_negative_exponent_against_exact_rationals(dtype):
    """The negative-exponent reading (the pages leave it open) is the exact
    power truncated toward zero, as integer Div truncates: checked by brute
    force against Python's exact rationals, trunc(Fraction(base) ** e), for
    every base in [-40, 40] and the type's limits, every exponent in [-70, -1]
    and the most negative one; a zero base flags division by zero and writes 0."""
    st_t = datagen.STORAGE[dtype]
    lo, hi = INT_LIMITS[dtype]
    bases = [x for x in list(range(-40, 41)) + [lo, lo + 1, hi, hi - 1] if x != 0]
    exps = list(range(-70, 0)) + [lo]
    pairs = [(x, y) for x in bases for y in exps if abs(x) == 1 or y >= -70]
    a = np.array([x for x, _ in pairs], dtype=object).astype(st_t)
    b = np.array([y for _, y in pairs], dtype=object).astype(st_t)
    got, st = oracle.run("Pow", a, b, dtype)
    want = [math.trunc(Fraction(x) ** y) for x, y in pairs]
    assert st == 0 and [int(v) for v in got] == want
    z = np.zeros(len(exps), st_t)
    got, st = oracle.run("Pow", z, np.array(exps, dtype=object).astype(st_t), dtype)
    assert st == oracle.STATUS_DIV_BY_ZERO and not got.any()


def test_int_pow_negative_exponent_reading():
    """The negative-exponent reading on named cases: trunc(1 / base^|e|), base 0
    flags division by zero."""
    a = np.array([1, -1, -1, 2, -3, 7], np.int32)
    b = np.array([-5, -3, -4, -1, -2, -1], np.int32)
    got, st = oracle.run("Pow", a, b, "int32")
    assert list(got) == [1, -1, 1, 0, 0, 0] and st == 0
    _, st = oracle.run("Pow", np.array([0], np.int32), np.array([-1], np.int32), "int32")
    assert st == oracle.STATUS_DIV_BY_ZERO


# --------------------------------------------------------------------------- Pow (float)

def test_f32_pow_within_half_ulp_of_mpmath():
    import mpmath
    mpmath.mp.prec = 200
    n = 1500
    base = np.concatenate([datagen.uniform(31, 0, n, 1e-3, 50.0),
                           -np.floor(datagen.uniform(31, 1, n, 1.0, 20.0))])
    expo = np.concatenate([datagen.uniform(31, 2, n, -12.0, 12.0),
                           np.floor(datagen.uniform(31, 3, n, -9.0, 10.0))]).astype(np.float32)
    base = base.astype(np.float32)
    got, _ = oracle.run("Pow", base, expo, "float32")
    want = []
    for x, y in zip(base, expo):
        v = mpmath.power(mpmath.mpf(float(x)), mpmath.mpf(float(y)))
        sign, man, exp, _ = mpmath.mpf(v)._mpf_
        want.append(rn32((-1) ** sign * Fraction(int(man)) * Fraction(2) ** int(exp)))
    want = np.array(want, np.float32)
    d = ulp_distance(got, want, "float32")
    assert d.max() <= 1, d.max()
    assert (d == 0).mean() > 0.999


# --------------------------------------------------------------------------- mixed-type Pow
MIXED_EXP = ["float32", "float16", "bfloat16", "int32", "int64", "uint8", "uint32", "int8",
             "int16", "uint16", "uint64"]


def _exponents(dtype, n, seed):
    if dtype in ("float32", "float16", "bfloat16"):
        e = datagen.uniform(seed, 0, n, -4.0, 4.0)
        e[::3] = np.round(e[::3])
        return datagen.float_to(e.astype(np.float32), dtype)
    lo = 0 if dtype.startswith("u") else -3
    return datagen.make("int_range", dtype, (n,), seed, 1, lo=lo, hi=9)


def _as_f64(x, dtype):
    if dtype == "bfloat16":
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


@pytest.mark.parametrize("ta", ["float32", "float16", "bfloat16"])
@pytest.mark.parametrize("tb", MIXED_EXP)
def test_pow_mixed_float_base_matches_numpy_float64(ta, tb):
    """ONNX Pow base T / exponent T1 (typed scalar adapters): a floating base
    takes pow in binary64 on the exponent's exact value, rounded to binary32,
    then to the base type."""
    if ta == tb:
        pytest.skip("same type")
    n = 4000
    a = datagen.float_to(datagen.uniform(61, 0, n, 0.0, 6.0).astype(np.float32), ta)
    b = _exponents(tb, n, 62)
    got, st = oracle.run_pow_mixed(a, b, ta, tb)
    with np.errstate(all="ignore"):
        y = np.power(_as_f64(a, ta), _as_f64(b, tb)).astype(np.float32)
    want = datagen.float_to(y, ta) if ta != "float32" else y
    assert st == 0
    assert_bits_equal(got, want, ta, "Pow %s^%s" % (ta, tb))


@pytest.mark.parametrize("ta", ["int32", "int64"])
@pytest.mark.parametrize("tb", ["int32", "int64", "uint8", "uint32", "int8", "int16", "uint16",
                                "uint64"])
def test_pow_mixed_int_base_int_exponent_matches_python(ta, tb):
    if ta == tb:
        pytest.skip("same type")
    a = np.array([v for v in range(-5, 6) for _ in range(12)], datagen.STORAGE[ta])
    lo = 0 if tb.startswith("u") else -3
    b = np.array(list(range(lo, lo + 12)) * 11, datagen.STORAGE[tb])
    got, st = oracle.run_pow_mixed(a, b, ta, tb)
    want = []
    for x, e in zip(a.tolist(), b.tolist()):
        if e >= 0:
            want.append(wrap(x ** e, ta))
        else:                                    # the same-type reading: 1/x^|e| truncated
            want.append(1 if x == 1 else (1 if e % 2 == 0 else -1) if x == -1 else 0)
    assert (got == np.array(want, dtype=object).astype(datagen.STORAGE[ta])).all()
    assert st == (oracle.STATUS_DIV_BY_ZERO if ((a == 0) & (b < 0)).any() else 0)


@pytest.mark.parametrize("ta", ["int32", "int64"])
@pytest.mark.parametrize("tb", ["float32", "float16", "bfloat16"])
def test_pow_mixed_int_base_float_exponent(ta, tb):
    """pow in binary64, truncated toward zero, saturated at the type's bounds,
    NaN to 0, no status."""
    n = 3000
    a = datagen.make("int_range", ta, (n,), 63, 0, lo=-20, hi=40)
    b = _exponents(tb, n, 64)
    a[:6] = [2, -8, 0, 10, 7, 3]
    b[:6] = datagen.float_to(np.array([0.5, 1 / 3, -1.0, 20.0, np.nan, 2.0], np.float32), tb)
    got, st = oracle.run_pow_mixed(a, b, ta, tb)
    info = np.iinfo(datagen.STORAGE[ta])
    with np.errstate(all="ignore"):
        y = np.power(a.astype(np.float64), _as_f64(b, tb))
    want = []
    for v in y.tolist():
        if math.isnan(v):
            want.append(0)
        elif v >= info.max:
            want.append(info.max)
        elif v <= info.min:
            want.append(info.min)
        else:
            want.append(int(math.trunc(v)))
    assert (got == np.array(want, dtype=object).astype(datagen.STORAGE[ta])).all()
    assert list(got[:6]) == [1, 0, info.max, info.max, 0, 9]    # 10^20 saturates both
    assert st == 0


def test_pow_special_values():
    for x, y, want in read_golden("pow_special_values.txt"):
        got, _ = oracle.run("Pow", f32(float(x)), f32(float(y)), "float32")
        g = float(got[0])
        if want == "nan":
            assert math.isnan(g), (x, y, g)
        else:
            w = float(want)
            assert g == w and math.copysign(1, g) == math.copysign(1, w), (x, y, g, w)


# --------------------------------------------------------------------------- comparisons/logic

CMP = [("Equal", np.equal), ("Less", np.less), ("Greater", np.greater),
       ("LessOrEqual", np.less_equal), ("GreaterOrEqual", np.greater_equal)]


@pytest.mark.parametrize("op,fn", CMP)
def test_comparisons_match_numpy(op, fn):
    a = float_corpus(5000, 41)
    b = np.concatenate([np.roll(a[:-len(SPECIALS)], 1), SPECIALS[::-1]])
    b[::3] = a[::3]                                # many equal pairs
    got, _ = oracle.run(op, a, b, "float32")
    assert got.dtype == np.uint8 and (got == fn(a, b).astype(np.uint8)).all()
    h_a, h_b = a.astype(np.float16), b.astype(np.float16)
    got, _ = oracle.run(op, h_a, h_b, "float16")
    assert (got == fn(h_a, h_b).astype(np.uint8)).all()
    bf_a, bf_b = bf16_bits(a), bf16_bits(b)
    got, _ = oracle.run(op, bf_a, bf_b, "bfloat16")
    assert (got == fn(bf16_to_f32(bf_a), bf16_to_f32(bf_b)).astype(np.uint8)).all()
    for dtype in ALL_INTS:
        ia = datagen.make("bits", dtype, (3000,), 42, 0)
        ib = datagen.make("bits", dtype, (3000,), 42, 1)
        ib[::4] = ia[::4]
        got, _ = oracle.run(op, ia, ib, dtype)
        assert (got == fn(ia, ib).astype(np.uint8)).all()


def test_comparisons_nan_and_signed_zero():
    a = f32(np.nan, np.nan, 0.0, -0.0)
    b = f32(np.nan, 1.0, -0.0, 0.0)
    for op, _ in CMP:
        got, _ = oracle.run(op, a, b, "float32")
        assert got[0] == 0 and got[1] == 0
    eq, _ = oracle.run("Equal", a, b, "float32")
    assert eq[2] == 1 and eq[3] == 1


@pytest.mark.parametrize("op,fn", [("And", np.logical_and), ("Or", np.logical_or),
                                   ("Xor", np.logical_xor)])
def test_logical_matches_numpy(op, fn):
    a = datagen.make("bool", "bool", (5000,), 43, 0)
    b = datagen.make("bool", "bool", (5000,), 43, 1)
    got, _ = oracle.run(op, a, b, "bool")
    assert (got == fn(a, b).astype(np.uint8)).all()
    x, _ = oracle.run("Xor", a, a, "bool")
    assert not x.any()


def test_less_is_mirrored_greater():
    a = float_corpus(4000, 44)
    b = np.roll(a, 11)
    lt, _ = oracle.run("Less", a, b, "float32")
    gt, _ = oracle.run("Greater", b, a, "float32")
    le, _ = oracle.run("LessOrEqual", a, b, "float32")
    eq, _ = oracle.run("Equal", a, b, "float32")
    assert (lt == gt).all()
    ok = ~(np.isnan(a) | np.isnan(b))
    assert (le[ok] == (lt | eq)[ok]).all()


# --------------------------------------------------------------------------- PRelu / BN / Clip

def test_prelu_closed_forms():
    for row in read_golden("prelu_clip_closed_form.txt"):
        op, x, p1, p2, want = row
        if op == "prelu":
            got, _ = oracle.run("PRelu", f32(float(x)), f32(float(p1)), "float32")
        else:
            got, _ = oracle.run("Clip", f32(float(x)), f32(float(p1), float(p2)), "float32")
        g, w = float(got[0]), float(want)
        assert g == w and math.copysign(1, g) == math.copysign(1, w), row


@pytest.mark.parametrize("dtype", ["float32", "float16"])
def test_prelu_matches_numpy_where(dtype):
    x = datagen.make("normal", dtype, (64, 3, 5), 45, 0)
    s = datagen.make("uniform", dtype, (3, 1), 45, 1, lo=0.0, hi=0.3)
    got, _ = oracle.run("PRelu", x, s, dtype)
    want = np.where(x >= 0, x, np.broadcast_to(s, x.shape) * x)
    assert_bits_equal(got, want, dtype, "PRelu")
    one, _ = oracle.run("PRelu", x, np.ones((3, 1), datagen.STORAGE[dtype]), dtype)
    assert_bits_equal(one, x, dtype, "PRelu slope 1 is the identity")


def test_prelu_one_dimensional_slope_is_per_channel():
    """A 1-D slope [C] multiplies channel c (axis 1) of the data, whatever the
    last extent is (0verkilll/onnx ops, PReluOp: per-channel slope forms)."""
    for shape, slope, x, want, note in read_golden("prelu_per_channel_slope.txt"):
        xs = f32(*[float(v) for v in x.split(",")]).reshape([int(v) for v in shape.split(",")])
        sl = f32(*[float(v) for v in slope.split(",")])
        if want == "refused":
            with pytest.raises(ValueError, match="incompatible_shapes"):
                oracle.run("PRelu", xs, sl, "float32")
            continue
        got, st = oracle.run("PRelu", xs, sl, "float32")
        w = f32(*[float(v) for v in want.split(",")]).reshape(xs.shape)
        assert st == 0 and got.shape == xs.shape, note
        assert_bits_equal(got, w, "float32", note)


def test_prelu_one_dimensional_slope_equals_its_channel_shaped_form():
    """[C] and [C,1,...,1] / [1,C,1,...,1] are the same per-channel slope."""
    for shape in ((3, 5, 4, 5), (2, 5, 5), (1, 5, 7, 2, 3)):
        x = datagen.make("normal", "float32", shape, 47, 0)
        s = datagen.make("uniform", "float32", (5,), 47, 1, lo=0.0, hi=0.3)
        flat, _ = oracle.run("PRelu", x, s, "float32")
        tail = (1,) * (len(shape) - 2)
        for form in ((5,) + tail, (1, 5) + tail):
            shaped, _ = oracle.run("PRelu", x, s.reshape(form), "float32")
            assert_bits_equal(flat, shaped, "float32", "%s vs %s" % (shape, form))
        want = np.where(x >= 0, x, s.reshape((1, 5) + tail) * x)
        assert_bits_equal(flat, want, "float32", "numpy per-channel where %s" % (shape,))


def test_prelu_is_unidirectional():
    with pytest.raises(ValueError, match="incompatible_shapes"):
        oracle.run("PRelu", np.zeros((3, 1), np.float32), np.zeros((3, 4), np.float32), "float32")


def test_batchnorm_closed_forms():
    for x, mean, var, eps, scale, bias, want in read_golden("batchnorm_closed_form.txt"):
        xs = f32(float(x)).reshape(1, 1)
        params = f32(float(scale), float(bias), float(mean), float(var)).reshape(4, 1)
        got, _ = oracle.run("BatchNormalization", xs, params, "float32", eps=float(eps))
        g, w = float(got[0, 0]), float(want)
        assert g == w and math.copysign(1, g) == math.copysign(1, w), (x, g, w)


def test_batchnorm_identity_and_channel_axis():
    x = datagen.make("normal", "float32", (2, 3, 4, 5), 46, 0)
    ident = np.zeros((4, 3), np.float32)
    ident[0] = 1.0
    ident[1] = -0.0
    ident[3] = 1.0
    got, _ = oracle.run("BatchNormalization", x, ident, "float32", eps=0.0)
    assert_bits_equal(got, x, "float32", "BN identity")
    # only channel 1 gets a shift: everything else stays bit-identical
    p = ident.copy()
    p[1, 1] = 10.0
    got, _ = oracle.run("BatchNormalization", x, p, "float32", eps=0.0)
    assert_bits_equal(got[:, [0, 2]], x[:, [0, 2]], "float32", "BN other channels")
    assert_bits_equal(got[:, 1], x[:, 1] + np.float32(10.0), "float32", "BN channel 1")


def test_batchnorm_within_float64_bound():
    """Five correctly rounded binary32 steps stay within a few ulp of the exact value."""
    x = datagen.make("normal", "float32", (4, 8, 33), 47, 0)
    p = np.stack([datagen.normal(47, 1, 8), datagen.normal(47, 2, 8), datagen.normal(47, 3, 8),
                  datagen.uniform(47, 4, 8, 0.1, 2.0)]).astype(np.float32)
    got, _ = oracle.run("BatchNormalization", x, p, "float32", eps=1e-5)
    sc, bi, mu, va = (p[i].astype(np.float64)[None, :, None] for i in range(4))
    exact = (x.astype(np.float64) - mu) / np.sqrt(va + np.float64(np.float32(1e-5))) * sc + bi
    err = np.abs(got.astype(np.float64) - exact)
    scale = np.abs(exact) + np.abs(bi) + np.abs(sc) * np.abs(x.astype(np.float64) - mu)
    assert (err <= 8 * 2.0 ** -24 * scale + 1e-30).all()


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_bias_prelu_matches_float32_numpy_chain(dtype):
    """BiasPRelu (0verkilll/onnx ops, ConvPReluOp: per-channel bias add then
    per-channel PReLU in one pass): t = x + bias[c], y = t >= 0 ? t : slope[c]*t,
    each step a binary32 operation, rounded once to x's type."""
    C = 6
    x = datagen.make("normal", dtype, (3, C, 5, 7), 31, 0)
    x.reshape(-1)[:SPECIALS.size] = datagen.float_to(SPECIALS, dtype)
    params = np.concatenate([datagen.normal(31, 1, C), datagen.uniform(31, 2, C, -0.5, 0.5)])
    B = datagen.float_to(params.astype(np.float32), dtype).reshape(2, C)
    got, st = oracle.run("BiasPRelu", x, B, dtype)
    assert st == 0
    if dtype == "bfloat16":
        to32 = lambda v: torch.from_numpy(v.view(np.int16).copy()).view(torch.bfloat16).float()
        xf, bf = to32(x), to32(B)
        t = xf + bf[0].view(1, C, 1, 1)
        y = torch.where(t >= 0, t, bf[1].view(1, C, 1, 1) * t)
        want = y.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        xf, bf = x.astype(np.float32), B.astype(np.float32)
        with np.errstate(all="ignore"):
            t = xf + bf[0].reshape(1, C, 1, 1)
            y = np.where(t >= 0, t, bf[1].reshape(1, C, 1, 1) * t).astype(np.float32)
        want = y.astype(x.dtype)
    assert_bits_equal(got, want, dtype, "BiasPRelu")


def test_bias_prelu_shapes():
    x = np.zeros((2, 3, 4), np.float32)
    assert oracle.run("BiasPRelu", x, np.zeros((2, 3), np.float32), "float32")[0].shape == x.shape
    for bad in [(2, 4), (3, 3), (4, 3), (3,)]:
        with pytest.raises(Exception):
            oracle.run("BiasPRelu", x, np.zeros(bad, np.float32), "float32")


# --------------------------------------------------------------------------- BiasPReluBN
def test_bias_prelu_bn_closed_forms():
    for row in read_golden("bias_prelu_bn_closed_form.txt"):
        x, bias, slope, mean, var, eps, scale, bnb, want = (float(v) for v in row)
        xs = f32(x).reshape(1, 1)
        params = f32(bias, slope, scale, bnb, mean, var).reshape(6, 1)
        got, _ = oracle.run("BiasPReluBN", xs, params, "float32", eps=eps)
        g = float(got[0, 0])
        assert g == want and math.copysign(1, g) == math.copysign(1, want), (row, g)


def _chain_params(dtype, C, seed):
    p = np.concatenate([datagen.normal(seed, 1, C), datagen.uniform(seed, 2, C, -0.5, 0.5),
                        datagen.normal(seed, 3, C), datagen.normal(seed, 4, C),
                        datagen.normal(seed, 5, C), datagen.uniform(seed, 6, C, 0.1, 2.0)])
    return datagen.float_to(p.astype(np.float32), dtype).reshape(6, C)


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_bias_prelu_bn_matches_float32_numpy_chain(dtype):
    """BiasPReluBN: bias add, PReLU and inference BatchNormalization of one
    channel in one pass, every step a binary32 operation in the order written,
    rounded once to x's type (torch rounds float32 to bfloat16)."""
    C = 6
    x = datagen.make("normal", dtype, (3, C, 5, 7), 33, 0)
    x.reshape(-1)[:SPECIALS.size] = datagen.float_to(SPECIALS, dtype)
    B = _chain_params(dtype, C, 33)
    eps = np.float32(1e-5)
    got, st = oracle.run("BiasPReluBN", x, B, dtype, eps=float(eps))
    assert st == 0
    if dtype == "bfloat16":
        to32 = lambda v: torch.from_numpy(v.view(np.int16).copy()).view(torch.bfloat16).float()
        xf, bf = to32(x), to32(B)
        col = lambda i: bf[i].view(1, C, 1, 1)
        t = xf + col(0)
        t = torch.where(t >= 0, t, col(1) * t)
        y = (t - col(4)) / torch.sqrt(col(5) + torch.tensor(eps)) * col(2) + col(3)
        want = y.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        xf, bf = x.astype(np.float32), B.astype(np.float32)
        col = lambda i: bf[i].reshape(1, C, 1, 1)
        with np.errstate(all="ignore"):
            t = xf + col(0)
            t = np.where(t >= 0, t, col(1) * t).astype(np.float32)
            y = ((t - col(4)) / np.sqrt(col(5) + eps) * col(2) + col(3)).astype(np.float32)
        want = y.astype(x.dtype)
    assert_bits_equal(got, want, dtype, "BiasPReluBN")


def test_bias_prelu_bn_float32_is_the_unfused_chain():
    """In binary32 the fused pass equals BiasPRelu followed by
    BatchNormalization, each rounded to float32; channel by channel."""
    C = 5
    x = datagen.make("normal", "float32", (4, C, 9), 34, 0)
    B = _chain_params("float32", C, 34)
    got, _ = oracle.run("BiasPReluBN", x, B, "float32", eps=1e-3)
    t, _ = oracle.run("BiasPRelu", x, B[:2].copy(), "float32")
    want, _ = oracle.run("BatchNormalization", t, B[2:].copy(), "float32", eps=1e-3)
    assert_bits_equal(got, want, "float32", "fused vs unfused")


def test_bias_prelu_bn_float64_chain():
    C = 4
    x = datagen.make("normal", "float64", (2, C, 6), 35, 0)
    B = _chain_params("float64", C, 35)
    got, _ = oracle.run("BiasPReluBN", x, B, "float64", eps=1e-5)
    col = lambda i: B[i].reshape(1, C, 1)
    t = x + col(0)
    t = np.where(t >= 0, t, col(1) * t)
    want = (t - col(4)) / np.sqrt(col(5) + np.float64(np.float32(1e-5))) * col(2) + col(3)
    assert_bits_equal(got, want, "float64", "BiasPReluBN float64")


def test_bias_prelu_bn_shapes():
    x = np.zeros((2, 3, 4), np.float32)
    assert oracle.run("BiasPReluBN", x, np.zeros((6, 3), np.float32), "float32")[0].shape == x.shape
    for bad in [(6, 4), (4, 3), (2, 3), (6,)]:
        with pytest.raises(Exception):
            oracle.run("BiasPReluBN", x, np.zeros(bad, np.float32), "float32")


# ------------------------------------------------------- float32 parameter blocks
# The BatchNormalization block is "in x's dtype or fp32"; BiasPRelu and
# BiasPReluBN take the same choice.  With fp32 parameters beside fp16/bf16 x,
# each parameter enters the binary32 chain as it is (not rounded to x's type).

PARAM_ROWS = {"BatchNormalization": 4, "BiasPRelu": 2, "BiasPReluBN": 6}


def _f32_params(op, C, seed):
    rows = [datagen.normal(seed, i + 1, C) for i in range(PARAM_ROWS[op])]
    rows[-1] = datagen.uniform(seed, 9, C, 0.1, 2.0)     # var (BN rows) stays positive
    if op == "BiasPRelu":
        rows[1] = datagen.uniform(seed, 8, C, -0.5, 0.5)
    if op == "BiasPReluBN":
        rows[1] = datagen.uniform(seed, 8, C, -0.5, 0.5)
    return np.stack(rows).astype(np.float32)


def _torch_chain(op, xf, P, eps):
    """The operator's binary32 steps on torch float32 tensors, in the order
    written; each torch op rounds on its own."""
    C = P.shape[1]
    col = lambda i: P[i].view(1, C, *([1] * (xf.dim() - 2)))
    if op == "BatchNormalization":
        return (xf - col(2)) / torch.sqrt(col(3) + torch.tensor(eps)) * col(0) + col(1)
    t = xf + col(0)
    t = torch.where(t >= 0, t, col(1) * t)
    if op == "BiasPRelu":
        return t
    return (t - col(4)) / torch.sqrt(col(5) + torch.tensor(eps)) * col(2) + col(3)


@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
@pytest.mark.parametrize("op", ["BatchNormalization", "BiasPRelu", "BiasPReluBN"])
def test_float32_parameters_match_the_torch_chain(op, dtype):
    """16-bit x, binary32 parameters: the torch float32 chain on x widened and
    the parameters as given, rounded once to x's type (torch rounds to
    nearest even)."""
    C = 7
    x = datagen.make("normal", dtype, (3, C, 5, 6), 36, 0)
    x.reshape(-1)[:SPECIALS.size] = datagen.float_to(SPECIALS, dtype)
    P = _f32_params(op, C, 36)
    eps = np.float32(1e-5)
    got = oracle.run_params(op, x, P, dtype, "float32", eps=float(eps))
    tx = torch.from_numpy(x.view(np.int16).copy()).view(
        torch.bfloat16 if dtype == "bfloat16" else torch.float16).float()
    y = _torch_chain(op, tx, torch.from_numpy(P), eps)
    if dtype == "bfloat16":
        want = y.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        want = y.to(torch.float16).numpy()
    assert_bits_equal(got, want, dtype, "%s fp32 parameters" % op)
    # the parameters are not first rounded to x's type: the 16-bit block differs
    same, _ = oracle.run(op, x, datagen.float_to(P, dtype), dtype, eps=float(eps))
    assert (got.view(np.uint16) != same.view(np.uint16)).any()


@pytest.mark.parametrize("op", ["BatchNormalization", "BiasPRelu", "BiasPReluBN"])
def test_float32_parameters_beside_float64(op):
    """float64 x, binary32 parameters widened exactly: the numpy float64 chain."""
    C = 5
    x = datagen.make("normal", "float64", (2, C, 9), 37, 0)
    P = _f32_params(op, C, 37)
    got = oracle.run_params(op, x, P, "float64", "float32", eps=1e-5)
    y = _torch_chain(op, torch.from_numpy(x), torch.from_numpy(P.astype(np.float64)),
                     float(np.float32(1e-5))).numpy()
    assert_bits_equal(got, y, "float64", "%s fp32 parameters, float64 x" % op)


@pytest.mark.parametrize("op", ["BatchNormalization", "BiasPRelu", "BiasPReluBN"])
def test_float32_parameters_exact_in_x_type_equal_the_same_type_block(op):
    """Parameters that x's type holds exactly give the same-type operator's
    result, bit for bit; and a block of x's own type is that operator."""
    C = 6
    for dtype in ("float16", "bfloat16"):
        x = datagen.make("normal", dtype, (4, C, 11), 38, 0)
        Bx = datagen.float_to(_f32_params(op, C, 38), dtype)
        P = (Bx.astype(np.float32) if dtype == "float16" else bf16_to_f32(Bx)).astype(np.float32)
        want, _ = oracle.run(op, x, Bx, dtype)
        assert_bits_equal(oracle.run_params(op, x, P, dtype, "float32"), want, dtype, op)
        assert_bits_equal(oracle.run_params(op, x, Bx, dtype, dtype), want, dtype, op)


def test_float32_parameters_refusals():
    x16 = np.zeros((2, 3, 4), np.float16)
    P = np.zeros((4, 3), np.float32)
    with pytest.raises(ValueError, match="type"):
        oracle.run_params("Add", x16, np.zeros((4,), np.float32), "float16", "float32")
    with pytest.raises(ValueError, match="type"):      # fp16 parameters beside fp32 x
        oracle.run_params("BatchNormalization", np.zeros((2, 3, 4), np.float32),
                          P.astype(np.float16), "float32", "float16")
    with pytest.raises(ValueError, match="shapes"):
        oracle.run_params("BatchNormalization", x16, np.zeros((4, 2), np.float32), "float16",
                          "float32")


# --------------------------------------------------------------------------- MulAdd
# 0verkilll/onnx ops, MulAddOp: y = (a * b) + c, shapes as the unfused Mul + Add.

def _muladd_inputs(dtype, shapes, seed):
    return [datagen.make("normal" if dtype in ("float32", "float16", "bfloat16") else "bits",
                         dtype, sh, seed, k) for k, sh in enumerate(shapes)]


@pytest.mark.parametrize("shapes", [((4, 8, 5, 6), (1, 8, 1, 1), (4, 8, 5, 6)),
                                    ((1,), (3, 7, 11), (3, 7, 11)),
                                    ((2, 1, 5), (1, 4, 1), (4, 5))])
@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_muladd_matches_float32_chain(dtype, shapes):
    a, b, c = _muladd_inputs(dtype, shapes, 41)
    for x in (a, b, c):
        x.reshape(-1)[: min(x.size, 5)] = datagen.float_to(SPECIALS[:5], dtype)[: min(x.size, 5)]
    got = oracle.run3("MulAdd", a, b, c, dtype)
    if dtype == "bfloat16":
        t = [torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).float() for x in (a, b, c)]
        want = (t[0] * t[1] + t[2]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        f = [x.astype(np.float32) for x in (a, b, c)]
        with np.errstate(all="ignore"):
            prod = np.multiply(f[0], f[1], dtype=np.float32)       # rounded product
            want = np.add(prod, f[2], dtype=np.float32).astype(a.dtype)
    assert got.shape == np.broadcast_shapes(*shapes)
    assert_bits_equal(got, want, dtype, "MulAdd")


@pytest.mark.parametrize("dtype", ALL_INTS)
def test_muladd_int_wraps_like_python_integers(dtype):
    a, b, c = _muladd_inputs(dtype, [(3, 1, 40), (1, 5, 40), (40,)], 42)
    got = oracle.run3("MulAdd", a, b, c, dtype)
    lo, hi = INT_LIMITS[dtype]
    A, B, C = np.broadcast_arrays(a.astype(object), b.astype(object), c.astype(object))
    want = np.vectorize(lambda x, y, z: wrap(int(x) * int(y) + int(z), dtype), otypes=[object])(
        A, B, C).astype(datagen.STORAGE[dtype])
    assert (got == want).all()


def test_muladd_broadcast_brute_force():
    """Index mapping of three-way broadcasting against numpy's, with small integer
    values so that every result is exact."""
    rng = np.random.default_rng(43)
    dims = [()] + [s for r in (1, 2, 3) for s in itertools.product((1, 2, 3), repeat=r)]
    for _ in range(1500):
        sh = [dims[i] for i in rng.integers(0, len(dims), 3)]
        try:
            want_shape = np.broadcast_shapes(*sh)
        except ValueError:
            with pytest.raises(ValueError):
                oracle.run3("MulAdd", *[np.zeros(s, np.float32) for s in sh], "float32")
            continue
        a, b, c = [rng.integers(-8, 9, s).astype(np.float32) for s in sh]
        got = oracle.run3("MulAdd", a, b, c, "float32")
        assert got.shape == want_shape
        assert (got == a * b + c).all(), sh


# --------------------------------------------------------------------------- float64
# DOUBLE computes natively in binary64, each operation rounded on its own.

def f64_corpus(n, seed):
    bits = datagen.make("bits", "float64", (n,), seed, 0)
    mid = datagen.normal(seed, 1, n).astype(np.float64) * 100.0 + \
        datagen.normal(seed, 2, n).astype(np.float64) * 1e-6
    sp = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 5e-324, -5e-324,
                   2.2250738585072014e-308, 1.7976931348623157e308, 3.0, -7.0], np.float64)
    return np.concatenate([bits, mid, sp])


@pytest.mark.parametrize("op,fn", [("Add", np.add), ("Sub", np.subtract), ("Mul", np.multiply),
                                   ("Div", np.divide), ("RSub", lambda a, b: b - a),
                                   ("RDiv", lambda a, b: b / a)])
def test_f64_arith_matches_numpy(op, fn):
    a, b = f64_corpus(20000, 91), np.roll(f64_corpus(20000, 92), 5)
    got, st = oracle.run(op, a, b, "float64")
    with np.errstate(all="ignore"):
        want = fn(a, b)
    assert st == 0
    assert_bits_equal(got, want, "float64", op)


def test_f64_mod_matches_numpy_remainder_and_fmod():
    """fmod=0: numpy's floating remainder takes the divisor's sign by the same
    rule (one rounded add, zeros copysigned); fmod=1: C fmod."""
    a = f64_corpus(20000, 93)
    b = np.roll(f64_corpus(20000, 94), 3)
    with np.errstate(all="ignore"):
        got0, _ = oracle.run("Mod", a, b, "float64", fmod=0)
        got1, _ = oracle.run("Mod", a, b, "float64", fmod=1)
        assert_bits_equal(got1, np.fmod(a, b), "float64", "fmod=1")
        fin = np.isfinite(a) & np.isfinite(b) & (b != 0)
        assert_bits_equal(got0[fin], np.remainder(a[fin], b[fin]), "float64", "fmod=0")


def test_f64_pow_within_one_ulp_of_mpmath():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 120
    a = np.abs(datagen.normal(95, 0, 3000).astype(np.float64)) * 3 + 1e-3
    b = datagen.uniform(95, 1, 3000, -6.0, 6.0).astype(np.float64)
    got, _ = oracle.run("Pow", a, b, "float64")
    for x, y, g in zip(a.tolist(), b.tolist(), got.tolist()):
        exact = mpmath.power(mpmath.mpf(x), mpmath.mpf(y))
        assert abs(mpmath.mpf(g) - exact) <= mpmath.mpf(np.spacing(abs(g))), (x, y, g)


def test_f64_compare_max_min_clip_match_numpy():
    a, b = f64_corpus(20000, 96), np.roll(f64_corpus(20000, 97), 7)
    b[::9] = a[::9]
    for op, fn in CMP:
        got, _ = oracle.run(op, a, b, "float64")
        with np.errstate(all="ignore"):
            assert (got == fn(a, b).astype(np.uint8)).all(), op
    a2, b2 = _no_zero_pairs(a, b)
    for op, fn in (("Max", np.maximum), ("Min", np.minimum)):
        got, _ = oracle.run(op, a2, b2, "float64")
        assert_bits_equal(got, fn(a2, b2), "float64", op)
    got, _ = oracle.run("Max", np.array([-0.0, 0.0]), np.array([0.0, -0.0]), "float64")
    assert_bits_equal(got, np.array([0.0, 0.0]), "float64", "Max zeros")
    fin = a[np.isfinite(a)]
    got, _ = oracle.run("Clip", fin, np.array([-50.0, 75.5]), "float64")
    assert_bits_equal(got, np.clip(fin, -50.0, 75.5), "float64", "Clip")


def test_f64_channel_ops_and_muladd_match_numpy():
    C = 5
    x = datagen.normal(98, 0, 4 * C * 6).astype(np.float64).reshape(4, C, 6) * 3
    p = np.stack([datagen.normal(98, k, C).astype(np.float64) for k in (1, 2, 3)] +
                 [datagen.uniform(98, 4, C, 0.1, 2.0).astype(np.float64)])
    got, _ = oracle.run("BatchNormalization", x, p, "float64", eps=1e-5)
    rs = lambda v: v.reshape(1, C, 1)
    want = (x - rs(p[2])) / np.sqrt(rs(p[3]) + np.float64(np.float32(1e-5))) * rs(p[0]) + rs(p[1])
    assert_bits_equal(got, want, "float64", "BN")
    bs = p[:2].copy()
    got, _ = oracle.run("BiasPRelu", x, bs, "float64")
    t = x + rs(bs[0])
    assert_bits_equal(got, np.where(t >= 0, t, rs(bs[1]) * t), "float64", "BiasPRelu")
    a, b, c = x, p[0].reshape(1, C, 1), np.roll(x, 1)
    assert_bits_equal(oracle.run3("MulAdd", a, b, c, "float64"), a * b + c, "float64", "MulAdd")


def test_clip_matches_numpy_and_bounds_are_optional():
    x = float_corpus(5000, 48)
    lohi = f32(-2.5, 3.0)
    got, _ = oracle.run("Clip", x, lohi, "float32")
    ok = ~np.isnan(x)
    assert_bits_equal(got[ok], np.minimum(np.maximum(x[ok], lohi[0]), lohi[1]), "float32", "Clip")
    assert np.isnan(got[~ok]).all()
    only_max, _ = oracle.run("Clip", x, lohi, "float32", has_min=False)
    assert_bits_equal(only_max[ok], np.minimum(x[ok], lohi[1]), "float32", "Clip max only")
    none, _ = oracle.run("Clip", x, lohi, "float32", has_min=False, has_max=False)
    assert_bits_equal(none, x, "float32", "Clip without bounds")
    xi = datagen.make("bits", "int32", (3000,), 48, 1)
    gi, _ = oracle.run("Clip", xi, np.array([-1000, 5000], np.int32), "int32")
    assert (gi == np.clip(xi, -1000, 5000)).all()


# --------------------------------------------------------------------------- descriptor

def test_descriptor_rules_from_the_mod_section():
    cd = oracle.check_descriptor
    assert cd("Mod", 28, 0, 0, "float32", "float32") == "ok"
    assert cd("Mod", 27, 0, 0, "float32", "float32") == "invalid_attr"
    assert cd("Mod", 27, 1, 0, "float16", "float16") == "ok"
    assert cd("Mod", 10, 0, 0, "int32", "int32") == "ok"
    assert cd("Mod", 9, 1, 0, "int32", "int32") == "invalid_attr"
    assert cd("Mod", 28, 2, 0, "int32", "int32") == "invalid_attr"
    assert cd("BitShift", 11, 0, 2, "uint8", "uint8") == "invalid_attr"
    assert cd("BitShift", 11, 0, 1, "int32", "int32") == "unsupported_type"
    assert cd("And", 7, 0, 0, "float32", "float32") == "unsupported_type"
    assert cd("Add", 14, 0, 0, "float32", "float16") == "unsupported_type"
    for op in ("Equal", "Less", "Greater", "LessOrEqual", "GreaterOrEqual", "And", "Or", "Xor"):
        assert oracle.output_type(op, "bool" if op in ("And", "Or", "Xor") else "int32") == "bool"
    assert oracle.output_type("Add", "bfloat16") == "bfloat16"
