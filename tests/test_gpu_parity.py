"""GPU parity: the CUDA path, called through the C ABI, against the oracle.

Every (operator, type) of the manifest runs on shapes chosen to land in each
loop family (with ragged tails and several CTAs of work), once with the
family the planner picks and once forced through the general strided kernel.
Results must be bit-identical (any NaN matches any NaN; signed zeros by
bits), except floating Pow, which must be within 2 ulp of the oracle.
"""
import numpy as np
import pytest

import datagen
import oracle
from conftest import assert_bits_equal, ulp_distance
from engine_util import (FLOATS, MANIFEST, ONE_WAY, PARAM_ROWS, chain_params,
                         every_16bit_value, inputs_for, run_engine, to_device)

eb = pytest.importorskip("broadcast_elementwise_gb300")

pytestmark = pytest.mark.gpu

TWO_WAY_CASES = [
    ("contiguous", (300007,), (300007,)),
    ("right_scalar", (300007,), ()),
    ("left_scalar", (1,), (300007,)),
    ("repeated_block", (300, 256), (300, 1)),
    ("repeated_block", (300, 256), (256,)),
    ("repeated_block", (300, 1), (300, 256)),
    ("repeated_block", (256,), (300, 256)),
    ("inner_vector_outer", (4, 16, 3, 256), (16, 1, 1)),
    ("inner_vector_outer", (6, 1, 5, 1), (1, 7, 1, 256)),
    ("general_strided", (2, 3, 4, 5), (3, 1, 5)),
    ("general_strided", (7, 1, 93), (1, 5, 93)),
    ("repeated_block", (33, 65), (33, 1)),
    # rows off the 16-byte pack width: the periodic flat kernel
    ("repeated_block", (1000, 3), (3,)),
    ("repeated_block", (1000, 3), (1000, 1)),
    ("repeated_block", (3,), (1000, 3)),
    ("repeated_block", (1000, 1), (1000, 13)),
    ("repeated_block", (257, 17), (17,)),
    # a block length dividing the pack: the broadcast values are read once
    ("repeated_block", (1000, 4), (4,)),
    ("repeated_block", (2,), (999, 2)),
    ("empty", (0, 5), (5,)),
    ("contiguous", (), ()),
]
PRELU_CASES = [
    ("inner_vector_outer", (4, 16, 3, 256), (16, 1, 1)),
    ("repeated_block", (300, 256), (256,)),
    ("repeated_block", (300, 256), (300, 1)),
    ("right_scalar", (300007,), (1,)),
    ("contiguous", (50001,), (50001,)),
    ("general_strided", (2, 3, 4, 5), (3, 1, 5)),
    ("repeated_block", (300, 7), (7,)),
    # a 1-D slope [C] is per channel (axis 1), whether or not the last extent is C
    ("general_strided", (2, 8, 5, 8), (8,)),
    ("general_strided", (2, 8, 5, 7), (8,)),
    ("inner_vector_outer", (2, 16, 8, 16), (16,)),
]
BN_CASES = [
    ("inner_vector_outer", (4, 16, 8, 32), (4, 16)),
    ("repeated_block", (300, 64), (4, 64)),
    ("repeated_block", (301, 6), (4, 6)),
    ("general_strided", (3, 16, 9, 11), (4, 16)),
    ("contiguous", (1, 64), (4, 64)),
    ("empty", (0, 16, 4), (4, 16)),
]
BIAS_PRELU_CASES = [(fam, sa, (2, sb[1])) for fam, sa, sb in BN_CASES]
CHAIN_CASES = [(fam, sa, (6, sb[1])) for fam, sa, sb in BN_CASES]
CLIP_CASES = [
    ("right_scalar", (300007,), (2,)),
    ("right_scalar", (40, 77), (2,)),
    ("contiguous", (1,), (2,)),
]


def cases_for(op):
    if op == "PRelu":
        return PRELU_CASES
    if op == "BatchNormalization":
        return BN_CASES
    if op == "BiasPRelu":
        return BIAS_PRELU_CASES
    if op == "BiasPReluBN":
        return CHAIN_CASES
    if op == "Clip":
        return CLIP_CASES
    return TWO_WAY_CASES


def attr_variants(op):
    if op == "Mod":
        return [{"fmod": 0}, {"fmod": 1}]
    if op == "BitShift":
        return [{"direction": 0}, {"direction": 1}]
    if op in ("BatchNormalization", "BiasPReluBN"):
        return [{"epsilon": 1e-5}]
    return [{}]


def oracle_kwargs(attrs):
    kw = {}
    if "fmod" in attrs:
        kw["fmod"] = attrs["fmod"]
    if "direction" in attrs:
        kw["direction"] = attrs["direction"]
    if "epsilon" in attrs:
        kw["eps"] = attrs["epsilon"]
    return kw


def compare(op, dtype, got, want, what):
    if op == "Pow" and dtype in FLOATS:
        d = ulp_distance(got, want, dtype)
        assert d.max(initial=0) <= 2, "%s: Pow differs by %d ulp" % (what, d.max())
    else:
        otype = "bool" if got.dtype == np.uint8 and op in (
            "Equal", "Less", "Greater", "LessOrEqual", "GreaterOrEqual", "And", "Or",
            "Xor") else dtype
        assert_bits_equal(got, want, otype, what)


PAIRS = [(op, dt) for op, dts in MANIFEST.items() for dt in dts]


@pytest.mark.parametrize("op,dtype", PAIRS, ids=["%s-%s" % p for p in PAIRS])
def test_parity_all_families(op, dtype):
    for attrs in attr_variants(op):
        for i, (fam, sa, sb) in enumerate(cases_for(op)):
            a, b = inputs_for(op, dtype, sa, sb, seed=i)
            want, want_bits = oracle.run(op, a, b, dtype, **oracle_kwargs(attrs))
            for forced in (None, "general_strided"):
                what = "%s %s %s %s x %s forced=%s" % (op, dtype, attrs, sa, sb, forced)
                got, bits, family = run_engine(op, dtype, a, b, family=forced, attrs=attrs)
                if forced is None:
                    assert family == fam, (what, family)
                compare(op, dtype, got, want, what)
                assert bits == want_bits, (what, bits, want_bits)


# (family, x shape, C): the block geometries of BN_CASES plus one channel
# (a single parameter per row, the right-scalar kernel)
F32_BLOCK_CASES = [(fam, sa, sb[1]) for fam, sa, sb in BN_CASES] + [
    ("right_scalar", (5, 1, 3001), 1)]


@pytest.mark.parametrize("op", list(PARAM_ROWS))
@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float64"])
def test_float32_parameter_block(op, dtype):
    """Parameters stored as float32 beside float16, bfloat16 or float64 x enter
    the chain unrounded: bit-identical to the oracle on every family the block
    reaches, natural and forced through the general kernel."""
    for i, (fam, sa, C) in enumerate(F32_BLOCK_CASES):
        sb = (PARAM_ROWS[op], C)
        a, _ = inputs_for(op, dtype, sa, sb, seed=40 + i)
        _, b = inputs_for(op, "float32", sa, sb, seed=40 + i)
        assert b.dtype == np.float32
        want = oracle.run_params(op, a, b, dtype, "float32")
        for forced in (None, "general_strided"):
            what = "%s %s x %s + float32 %s forced=%s" % (op, dtype, sa, sb, forced)
            got, bits, family = run_engine(op, dtype, a, b, family=forced,
                                           attrs={"dtype_b": "float32"})
            if forced is None:
                assert family == fam, (what, family)
            assert_bits_equal(got, want, dtype, what)
            assert bits == 0, what


@pytest.mark.parametrize("op,dtype", [("Add", "float32"), ("Greater", "float16"),
                                      ("Mod", "int32"), ("Xor", "bool"), ("Sub", "uint8")])
def test_inner_vector_kernel_on_other_geometries(op, dtype):
    """The inner-vector kernel forced onto contiguous, scalar and block geometries."""
    for i, (sa, sb) in enumerate([((300032,), (300032,)), ((300032,), ()), ((1,), (300032,)),
                                  ((300, 256), (256,)), ((300, 256), (300, 1))]):
        a, b = inputs_for(op, dtype, sa, sb, seed=40 + i)
        want, _ = oracle.run(op, a, b, dtype)
        got, _, fam = run_engine(op, dtype, a, b, family="inner_vector_outer")
        assert fam == "inner_vector_outer"
        compare(op, dtype, got, want, "%s %s %s %s" % (op, dtype, sa, sb))


@pytest.mark.parametrize("op", ["Greater", "Equal", "LessOrEqual"])
@pytest.mark.parametrize("dtype,inner", [("float32", 72), ("float16", 72), ("bfloat16", 88),
                                         ("int64", 70), ("int32", 68)])
def test_packed_compare_rows_with_ragged_ends(op, dtype, inner):
    """Comparisons write adjacent groups as one narrow pack; rows whose width
    is not a multiple of the pack finish group by group."""
    for i, (sa, sb) in enumerate([((9, 1, inner), (1, 3, inner)), ((5, 1, 7, 1), (1, 3, 1, inner)),
                                  ((40, inner), (inner,))]):
        a, b = inputs_for(op, dtype, sa, sb, seed=60 + i)
        want, _ = oracle.run(op, a, b, dtype)
        got, _, fam = run_engine(op, dtype, a, b)
        assert fam in ("inner_vector_outer", "repeated_block"), fam
        compare(op, dtype, got, want, "%s %s %s x %s" % (op, dtype, sa, sb))


MULADD_CASES = [
    ("contiguous", (300016,), (300016,), (300016,)),
    ("right_scalar", (300016,), (1,), (300016,)),
    ("right_scalar", (), (300016,), ()),
    ("inner_vector_outer", (4, 16, 8, 64), (1, 16, 1, 1), (4, 16, 8, 64)),
    ("inner_vector_outer", (1, 16, 1, 1), (4, 16, 8, 64), (4, 16, 8, 64)),
    ("inner_vector_outer", (6, 256), (256,), (6, 1)),
    # one operand one value per row, the other two dense: the per-row flat
    # kernel, with rows shorter than a thread's run (rows change inside runs)
    # and rows long enough for runs that stay in one row
    ("inner_vector_outer", (6, 256), (6, 256), (6, 1)),
    ("inner_vector_outer", (3, 37, 528), (1, 37, 1), (3, 37, 528)),
    ("inner_vector_outer", (2, 6, 16384), (1, 6, 1), (2, 6, 16384)),
    ("inner_vector_outer", (6, 1), (2, 6, 16384), (2, 6, 16384)),
    ("inner_vector_outer", (2, 6, 16384), (2, 6, 16384), (2, 6, 1)),
    ("general_strided", (3, 1, 5), (1, 4, 1), (4, 5)),
    ("general_strided", (7, 1, 93), (1, 5, 93), (93,)),
    ("empty", (0, 4), (4,), (1, 4)),
]


@pytest.mark.parametrize("dtype", FLOATS + ("int32", "int64", "uint8", "uint32"))
def test_muladd_parity_all_families(dtype):
    """MulAdd (0verkilll/onnx ops, MulAddOp) through ebin_execute3: the pages'
    fast paths (a scalar or per-channel multiplier, c shaped like the other
    operand), general three-way broadcasts, natural and forced-general, and
    buffers off 16-byte alignment."""
    from engine_util import run_engine3
    for i, (fam, sa, sb, sc) in enumerate(MULADD_CASES):
        kind = "normal" if dtype in FLOATS else "bits"
        a, b, c = [datagen.make(kind, dtype, s, 50 + i, k) for k, s in enumerate((sa, sb, sc))]
        if dtype in FLOATS:
            for x in (a, b, c):
                sp = datagen.float_to(np.array([0.0, -0.0, np.inf, np.nan, -1.5], np.float32),
                                      dtype)
                x.reshape(-1)[: min(x.size, 5)] = sp[: min(x.size, 5)]
        want = oracle.run3("MulAdd", a, b, c, dtype)
        for forced, offset in ((None, 0), ("general_strided", 0), (None, 1)):
            got, family = run_engine3("MulAdd", dtype, a, b, c, family=forced, offset=offset)
            if forced is None and offset == 0:
                assert family == fam, (sa, sb, sc, family)
            assert_bits_equal(got, want, dtype, "MulAdd %s %s %s %s forced=%s offset=%d" %
                              (dtype, sa, sb, sc, forced, offset))


STRIDED_VIEWS = [  # (base length, shape, element strides) of A, shape of B
    (64 * 48, (48, 64), (1, 48), (64,)),
    (200 * 9, (100, 3), (18, 3), (100, 1)),
    (64, (7, 64), (0, 1), (7, 64)),
    (64 * 1008, (64, 1000), (1008, 1), (1000,)),
    (64 * 1001, (64, 1000), (1001, 1), (64, 1)),
    (5 * 6 * 7 * 3, (5, 6, 7), (126, 21, 3), (6, 1)),
]


@pytest.mark.parametrize("op,dtype", [("Add", "float32"), ("Mul", "bfloat16"),
                                      ("Greater", "float16"), ("Mod", "int32"),
                                      ("Sub", "uint8"), ("PRelu", "float32")])
def test_strided_input_views(op, dtype):
    """Strided A views (transposed, sliced with steps, expanded, padded rows,
    inner stride 3) read in place: the result equals the oracle on the view's
    contiguous copy, in the natural family and forced through the general one."""
    import torch
    for i, (base_n, shape, strides, shape_b) in enumerate(STRIDED_VIEWS):
        if op == "PRelu":
            # a slope along the inner dim: [W] on rank <= 2, [1, ..., 1, W] above
            # (a 1-D slope on rank >= 3 data is per channel, axis 1)
            shape_b = ((1,) * (len(shape) - 1) + (shape[-1],)) if len(shape) else ()
        base, b = inputs_for(op, dtype, (base_n,), shape_b, seed=70 + i)
        view = np.lib.stride_tricks.as_strided(base, shape, [x * base.itemsize for x in strides])
        want, _ = oracle.run(op, np.ascontiguousarray(view), b, dtype)
        desc = eb.descriptor(op, dtype)
        dA, dB = to_device(base), to_device(b)
        for forced in (None, "general_strided"):
            plan = eb.Plan(desc, shape, shape_b, family=forced, strides_a=strides)
            osz = eb.ITEMSIZE[desc.out_dtype]
            out = torch.empty(plan.numel * osz, dtype=torch.uint8, device="cuda")
            eb.execute(plan, dA, dB, out)
            got = out.cpu().numpy().view(datagen.STORAGE[desc.out_dtype]).reshape(want.shape)
            compare(op, dtype, got, want, "%s %s view %s/%s forced=%s family=%s" %
                    (op, dtype, shape, strides, forced, plan.family))


# (M, N, ld): output [M, N]; the transposed input is a buffer of N * ld
# elements read as (i, j) -> i + j * ld (a transposed view, padded when ld > M)
TRANSPOSED = [(300, 257, 300), (1000, 70, 1003), (33, 2049, 40)]


@pytest.mark.parametrize("op,dtype", [("Add", "float32"), ("Mul", "bfloat16"),
                                      ("Sub", "float16"), ("Greater", "float32"),
                                      ("Div", "int32"), ("BitwiseXor", "uint8"),
                                      ("Max", "float64"), ("Mod", "int64"), ("RSub", "int32")])
def test_transposed_input(op, dtype):
    """A transposed view beside a dense input (general family, the tiled
    kernel): both orders, tiles cut by the edges, a padded leading dimension,
    1- to 8-byte elements, a BOOL output, and an integer divide whose zero
    divisor sets the status word; each against the oracle on contiguous
    copies."""
    import torch
    for i, (M, N, ld) in enumerate(TRANSPOSED):
        for t_is_b in (True, False):
            if t_is_b:
                a, base = inputs_for(op, dtype, (M, N), (N * ld,), seed=90 + i)
                if op in ("Div", "Mod") and dtype not in FLOATS:
                    base[2 * ld + 3] = 0                    # divisor (3, 2)
            else:
                base, b = inputs_for(op, dtype, (N * ld,), (M, N), seed=90 + i)
            t = np.lib.stride_tricks.as_strided(base, (M, N), (base.itemsize, ld * base.itemsize))
            a_c, b_c = (a, np.ascontiguousarray(t)) if t_is_b else (np.ascontiguousarray(t), b)
            want, wbits = oracle.run(op, a_c, b_c, dtype)
            desc = eb.descriptor(op, dtype)
            strides = (1, ld)
            plan = eb.Plan(desc, (M, N), (M, N), strides_a=None if t_is_b else strides,
                           strides_b=strides if t_is_b else None)
            assert plan.family == "general_strided"
            dA, dB = (to_device(a), to_device(base)) if t_is_b else (to_device(base), to_device(b))
            osz = eb.ITEMSIZE[desc.out_dtype]
            out = torch.empty(plan.numel * osz, dtype=torch.uint8, device="cuda")
            eb.execute(plan, dA, dB, out)
            bits = eb.get_device_status()
            got = out.cpu().numpy().view(datagen.STORAGE[desc.out_dtype]).reshape(want.shape)
            what = "%s %s [%d,%d] ld %d, %s transposed" % (op, dtype, M, N, ld,
                                                            "B" if t_is_b else "A")
            compare(op, dtype, got, want, what)
            assert bits == wbits, (what, bits, wbits)


MIXED_POW = [(ta, tb) for ta in ("float32", "float16", "bfloat16", "float64", "int32", "int64")
             for tb in ("float32", "float16", "bfloat16", "float64", "int32", "int64", "uint8",
                        "uint32", "int8", "int16", "uint16", "uint64")
             if ta != tb]


@pytest.mark.parametrize("ta,tb", MIXED_POW, ids=["%s^%s" % p for p in MIXED_POW])
def test_pow_with_exponent_of_another_type(ta, tb):
    """Pow base T / exponent T1 through the typed-adapter (general) kernel
    against the oracle: floating bases within 2 ulp, integer bases exactly,
    status bits equal."""
    import torch
    rng_a = {"float32": (0.0, 6.0), "float16": (0.0, 4.0), "bfloat16": (0.0, 6.0),
             "float64": (0.0, 6.0)}
    for i, (sa, sb) in enumerate([((3000,), (3000,)), ((40, 75), (75,)), ((6, 1, 50), (1, 7, 1))]):
        na, nb = int(np.prod(sa)), int(np.prod(sb))
        if ta in FLOATS:
            lo, hi = rng_a[ta]
            a = datagen.float_to(datagen.uniform(80 + i, 0, na, lo, hi), ta).reshape(sa)
        else:
            a = datagen.make("int_range", ta, sa, 80 + i, 0, lo=-6, hi=6)
        if tb in FLOATS:
            e = datagen.uniform(80 + i, 1, nb, -3.0, 3.0)
            e[::4] = np.round(e[::4])
            b = datagen.float_to(e, tb).reshape(sb)
        else:
            lo = 0 if tb.startswith("u") else -2
            b = datagen.make("int_range", tb, sb, 80 + i, 1, lo=lo, hi=12)
        want, wbits = oracle.run_pow_mixed(a, b, ta, tb)
        got, bits, fam = run_engine("Pow", ta, a, b, attrs={"dtype_b": tb})
        assert fam == "general_strided"
        assert bits == wbits
        if ta in FLOATS:
            d = ulp_distance(got, want, ta)
            assert d.max(initial=0) <= 2, ("Pow %s^%s" % (ta, tb), d.max())
        elif tb in FLOATS:
            # pow in binary64 is within 2 ulp on the device; where the power lies
            # within 4 ulp of an integer, truncation may land one unit apart
            bf = b.astype(np.float64) if tb != "bfloat16" else \
                (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            with np.errstate(all="ignore"):
                y = np.broadcast_to(np.power(a.astype(np.float64), bf), want.shape)
                near = np.abs(y - np.round(y)) <= 4 * np.spacing(np.abs(y))
            diff = np.abs(got.astype(np.int64) - want.astype(np.int64))
            assert ((diff == 0) | (near & (diff == 1))).all(), ("Pow %s^%s" % (ta, tb))
        else:
            assert (got == want).all(), ("Pow %s^%s" % (ta, tb))



@pytest.mark.parametrize("op", ["BatchNormalization", "BiasPReluBN"])
@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_prepared_division_on_every_16bit_value(op, dtype):
    """16-bit BatchNormalization and BiasPReluBN divide by each channel's
    sqrt(var + eps) through the prepared exact division (the reciprocal formed
    once, two corrections per quotient, the IEEE divide outside the proven
    ranges): every bfloat16 / float16 x pattern, in every channel, through the
    flat per-row kernel (pairs of elements), the general kernel (single
    elements) and rows of odd length, with 16-bit and float32 parameter blocks
    of ordinary and wide-ranging values, bit-identical to the oracle.  The
    inputs hold elements whose result changes when the chain's last multiply
    and add are merged into one fused multiply-add (test_chain_inputs checks
    that on the CPU), so a merged tail fails here."""
    C = 64
    for shape, fams in (((16, C, 64, 64), ("inner_vector_outer", "general_strided")),
                        ((16, C, 4097), ("general_strided",))):
        x = every_16bit_value(shape).view(datagen.STORAGE[dtype])
        for k, (wide, ptype) in enumerate(((False, dtype), (True, dtype), (True, "float32"))):
            p = chain_params(op, C, 90 + k, wide)
            b = datagen.float_to(p, ptype) if ptype != "float32" else p
            want = oracle.run_params(op, x, b, dtype, ptype)
            attrs = {"epsilon": 1e-5}
            if ptype != dtype:
                attrs["dtype_b"] = ptype
            for fam in fams:
                forced = None if fam == fams[0] else fam
                got, bits, family = run_engine(op, dtype, x, b, family=forced, attrs=attrs)
                what = "%s %s x%s params %s wide=%s family %s" % (op, dtype, shape, ptype, wide,
                                                                 family)
                assert family == fam, what
                assert_bits_equal(got, want, dtype, what)
                assert bits == 0, what


@pytest.mark.parametrize("op", ["Add", "Sub", "Mul", "RSub"])
@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_pair_forms_on_every_16bit_value(op, dtype):
    """16-bit Add, Sub, Mul and RSub run two elements per 32-bit word through
    mixed-precision operations (Mul: a 16-bit by 16-bit fused multiply-add
    with a -0 addend; the others: one operand widened, one 16-bit add).  Every
    bfloat16 / float16 pattern (NaNs, infinities, subnormals, both zeros) as
    each operand, against a seeded permutation of every pattern, through the
    contiguous kernel; every pattern against a value per row (the per-row flat
    kernel) and against a short reused row (the block-row kernel): bit-identical
    to the oracle."""
    st = datagen.STORAGE[dtype]
    every = np.arange(65536, dtype=np.uint16)
    rng = np.random.default_rng(2024)
    perm = rng.permutation(every)
    cases = [
        ("contiguous", every, perm),
        ("contiguous", perm, every),
        ("repeated_block", every.reshape(256, 256), rng.permutation(every)[:256].reshape(256, 1)),
        ("repeated_block", every.reshape(16384, 4), rng.permutation(every)[:4]),
    ]
    for fam, a16, b16 in cases:
        a, b = np.ascontiguousarray(a16).view(st), np.ascontiguousarray(b16).view(st)
        want, _ = oracle.run(op, a, b, dtype)
        got, bits, family = run_engine(op, dtype, a, b)
        what = "%s %s %s x %s" % (op, dtype, a.shape, b.shape)
        assert family == fam, what
        assert_bits_equal(got, want, dtype, what)
        assert bits == 0, what


# k_periodic: [n0,] n1, n2 with each input dense in the block, one value per
# row, or one reused row; (shape A, shape B, the pattern of A and of B)
PERIODIC_CASES = [
    ((7, 1, 5), (1, 12, 5)),        # reused row x dense block (the [a,1,k] x [1,b,k] shape)
    ((6, 8, 3), (6, 1, 3)),         # dense x reused row, outer strides 24 and 3
    ((5, 8, 3), (1, 8, 1)),         # dense x one value per row (per channel, short rows)
    ((1, 8, 1), (5, 8, 3)),         # one value per row x dense
    ((4, 8, 1), (4, 1, 6)),         # one value per row x reused row, with an outer index
    ((9, 1), (1, 7)),               # short outer products, both orders
    ((1, 7), (9, 1)),
    ((300, 7), (7,)),               # rank 2: dense x reused row
    # blocks of at least one k_blockrow tile (row rotations in shared memory)
    ((3, 1, 5), (1, 4000, 5)),      # reused row x dense block
    ((1, 4000, 5), (3, 1, 5)),      # dense block x reused row
    ((4001, 3), (3,)),              # rank 2, with a ragged tail of numel % 16-byte packs
    ((3, 1, 32), (1, 700, 32)),     # the longest row taken (32)
    ((3, 1, 33), (1, 700, 33)),     # one longer: element by element
]


def _run_offset(op, dtype, a, b, offset, attrs=None):
    """The engine on buffers shifted `offset` bytes off 16-byte alignment."""
    import torch
    desc = eb.descriptor(op, dtype, **(attrs or {}))
    plan = eb.Plan(desc, a.shape, b.shape)
    bufs = []
    for x in (a, b):
        raw = np.ascontiguousarray(x).reshape(-1).view(np.uint8)
        bufs.append(to_device(np.concatenate([np.zeros(offset, np.uint8), raw,
                                              np.zeros(16, np.uint8)])))
    osz = eb.ITEMSIZE[desc.out_dtype]
    out = torch.zeros(plan.numel * osz + offset + 16, dtype=torch.uint8, device="cuda")
    eb.ebin_execute(plan.handle, bufs[0].data_ptr() + offset, bufs[1].data_ptr() + offset,
                    out.data_ptr() + offset, None)
    bits = eb.get_device_status()
    host = out.cpu().numpy()[offset:offset + plan.numel * osz]
    return host.view(datagen.STORAGE[desc.out_dtype]).reshape(plan.output_shape), bits


@pytest.mark.parametrize("op,dtype", [("Add", "float32"), ("Mul", "bfloat16"),
                                      ("Sub", "float64"), ("Greater", "float16"),
                                      ("Mod", "int32"), ("BitwiseXor", "uint8"),
                                      ("Max", "int64")])
def test_short_rows_stream_flat(op, dtype):
    """Short-row repeated blocks, [a,1,k] x [1,b,k] general broadcasts and short
    outer products stream flat (k_periodic) when the buffers are aligned, and
    through the general row traversal when they are not: bit-identical to the
    oracle either way, status bits included."""
    attrs = {"fmod": 0} if op == "Mod" else {}
    for i, (sa, sb) in enumerate(PERIODIC_CASES):
        a, b = inputs_for(op, dtype, sa, sb, seed=60 + i)
        want, want_bits = oracle.run(op, a, b, dtype, **oracle_kwargs(attrs))
        for forced in (None, "general_strided"):
            got, bits, fam = run_engine(op, dtype, a, b, family=forced, attrs=attrs)
            what = "%s %s %s x %s forced=%s family %s" % (op, dtype, sa, sb, forced, fam)
            compare(op, dtype, got, want, what)
            assert bits == want_bits, what
        got, bits = _run_offset(op, dtype, a, b, eb.ITEMSIZE[dtype], attrs)
        compare(op, dtype, got, want, "%s %s %s x %s unaligned" % (op, dtype, sa, sb))
        assert bits == want_bits


@pytest.mark.parametrize("dtype", ["bfloat16", "float32"])
def test_per_channel_short_rows_stream_flat(dtype):
    """BatchNormalization and PRelu per channel on short spatial rows (NCW with
    W = 3): one value per row against dense data, with an outer index."""
    for op, sb in (("BatchNormalization", (4, 8)), ("PRelu", (8, 1)), ("BiasPReluBN", (6, 8))):
        sa = (5, 8, 3)
        a, b = inputs_for(op, dtype, sa, sb, seed=77)
        want, _ = oracle.run(op, a, b, dtype, **({"eps": 1e-5} if op != "PRelu" else {}))
        for forced in (None, "general_strided"):
            got, bits, fam = run_engine(op, dtype, a, b, family=forced,
                                        attrs={"epsilon": 1e-5} if op != "PRelu" else {})
            assert_bits_equal(got, want, dtype, "%s %s forced=%s" % (op, dtype, forced))
            assert bits == 0
