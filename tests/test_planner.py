"""Host logic of the C ABI, run on the CPU (no kernel is launched here).

The library loads without a GPU; descriptor creation, planning, the plan
cache, the alias check and empty executions never touch CUDA.
"""
import itertools
import os
import re

import numpy as np
import pytest

import oracle

eb = pytest.importorskip("broadcast_elementwise_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ALL_DTYPES = ["float32", "float16", "bfloat16", "int32", "int64", "uint8", "uint32", "bool",
              "int8", "int16", "uint16", "uint64", "float64"]


def header_functions():
    text = open(os.path.join(ROOT, "include", "ebin.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ebin_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(eb.lib, n), n


def test_descriptor_rules_match_oracle():
    for op, dt, opset, fmod, direction in itertools.product(
            list(eb.OPS), ALL_DTYPES, (9, 10, 27, 28, 29), (0, 1, 2), (0, 1, 2)):
        want = oracle.check_descriptor(op, opset, fmod, direction, dt, dt)
        try:
            d = eb.Descriptor(op, dt, opset=opset, fmod=fmod, direction=direction)
            got = "ok"
            assert d.out_dtype == oracle.output_type(op, dt)
            d.close()
        except eb.EbinError as e:
            got = e.code
        # the oracle only applies opset/fmod to Mod and direction to BitShift, as the engine does
        assert got == want, (op, dt, opset, fmod, direction, got, want)


def test_descriptor_rejects_mixed_types_and_bad_ops():
    with pytest.raises(eb.EbinError) as e:
        eb.ebin_descriptor_create(2, 14, None, eb.DTYPES["float32"], eb.DTYPES["float16"])
    assert e.value.code == "unsupported_type"
    with pytest.raises(eb.EbinError) as e:
        eb.ebin_descriptor_create(99, 14, None, 1, 1)
    assert e.value.code == "unsupported_op"


def test_descriptor_ids_are_monotonic():
    ids = [eb.Descriptor("Add", "float32").id for _ in range(5)]
    assert ids == sorted(ids) and len(set(ids)) == 5


def small_shapes():
    shapes = [()]
    for r in (1, 2, 3):
        shapes += list(itertools.product((0, 1, 2, 3), repeat=r))
    return shapes


def test_output_shapes_brute_force():
    d = eb.Descriptor("Add", "float32")
    for sa in small_shapes():
        for sb in small_shapes():
            try:
                want = oracle.output_shape("Add", sa, sb)
            except ValueError:
                want = None
            try:
                p = eb.Plan(d, sa, sb)
                got = p.output_shape
                p.close()
            except eb.EbinError as e:
                assert e.code == "incompatible_shapes"
                got = None
            assert got == want, (sa, sb)


def flat_offsets(n, sa, sb, idx):
    """Offsets of flat output indices through a coalesced geometry."""
    oa = np.zeros(idx.size, np.int64)
    ob = np.zeros(idx.size, np.int64)
    rem = idx.copy()
    for d in range(len(n) - 1, -1, -1):
        i = rem % n[d]
        rem //= n[d]
        oa += i * sa[d]
        ob += i * sb[d]
    return oa, ob


SHAPE_PAIRS = [((2, 3, 4, 5), (3, 1, 5)), ((8, 64, 16, 16), (64, 1, 1)),
               ((64, 1, 32, 1), (1, 8, 1, 64)), ((4096,), ()), ((40, 96), (40, 1)),
               ((40, 96), (96,)), ((1, 96), (40, 96)), ((7, 1, 9), (1, 5, 9)),
               ((2, 1, 3, 1, 4), (1, 5, 1, 6, 1)), ((3, 4, 5), (3, 4, 5)), ((1, 1, 1), (1,)),
               ((6, 1, 1, 7), (1, 1, 1)), ((2, 3, 1, 1, 5, 1, 7, 2), (3, 4, 1, 5, 6, 1, 2))]


@pytest.mark.parametrize("sa,sb", SHAPE_PAIRS)
def test_coalesced_geometry_preserves_the_element_mapping(sa, sb):
    d = eb.Descriptor("Add", "float32")
    p = eb.Plan(d, sa, sb)
    n, gsa, gsb = p.geometry()
    total = p.numel
    idx = np.arange(total, dtype=np.int64)
    want_a, want_b = oracle.offsets(sa, sb, idx)
    got_a, got_b = flat_offsets(n, gsa, gsb, idx)
    assert int(np.prod(n)) == total
    assert (got_a == want_a).all() and (got_b == want_b).all()
    # coalescing is maximal: no adjacent pair could still merge
    for i in range(len(n) - 1):
        assert not (gsa[i] == gsa[i + 1] * n[i + 1] and gsb[i] == gsb[i + 1] * n[i + 1])
    assert all(x > 1 for x in n) or total == 1


def family(op, dt, sa, sb, **kw):
    d = eb.Descriptor(op, dt, **kw)
    p = eb.Plan(d, sa, sb)
    return p.family, p.geometry()


def test_families_of_the_benchmark_workloads():
    assert family("Add", "float32", (2, 3, 4, 5), (3, 1, 5))[0] == "general_strided"
    assert family("Mul", "float32", (1 << 28,), (1 << 28,))[0] == "contiguous"
    f, (n, sa, sb) = family("Add", "bfloat16", (8, 64, 256, 256), (64, 1, 1))
    assert f == "inner_vector_outer" and n == [8, 64, 65536] and sb == [0, 1, 0]
    assert family("PRelu", "bfloat16", (8, 64, 256, 256), (64, 1, 1))[0] == "inner_vector_outer"
    assert family("BatchNormalization", "bfloat16", (8, 64, 256, 256), (4, 64))[0] == \
        "inner_vector_outer"
    assert family("Mod", "float32", (4096, 4096), (1,), fmod=1)[0] == "right_scalar"
    assert family("Mod", "float32", (4096, 4096), (), fmod=0)[0] == "right_scalar"
    assert family("Mod", "float32", (4096, 4096), (4096, 1), fmod=0)[0] == "repeated_block"
    assert family("Mod", "int32", (4096, 4096), (4096, 1))[0] == "repeated_block"
    f, (n, sa, sb) = family("Greater", "float16", (64, 1, 512, 1), (1, 32, 1, 1024))
    assert f == "inner_vector_outer" and n == [64, 32, 512, 1024]
    assert family("BitShift", "uint32", (1 << 26,), (1,), direction=1)[0] == "right_scalar"
    assert family("Add", "float32", (1,), (1 << 20,))[0] == "left_scalar"
    assert eb.Plan(eb.descriptor("Add", "float32"), (8192, 8192), (8192, 8192),
                   strides_b=(1, 8192)).family == "general_strided"      # a transposed view
    assert family("Add", "float32", (0, 5), (5,))[0] == "empty"
    assert family("Clip", "float32", (30, 40), (2,))[0] == "right_scalar"
    assert family("BatchNormalization", "float32", (300, 64), (4, 64))[0] == "repeated_block"
    assert family("Add", "float32", (1 << 24, 3), (3,))[0] == "repeated_block"
    f, (n, sa, sb) = family("Add", "float32", (8192, 1, 5), (1, 4096, 5))
    assert f == "general_strided" and n == [8192, 4096, 5] and sa == [5, 0, 1] and sb == [0, 5, 1]
    assert family("Mul", "bfloat16", (16384, 1, 3), (1, 8192, 3))[0] == "general_strided"


def test_repeated_block_rule_for_any_row_length():
    """Rank 2, one input dense and the other a reused row block (0,1) or one
    value per row (1,0) is REPEATED_BLOCK whatever the row length; with both
    inputs broadcast it stays GENERAL_STRIDED, and a one-way operator cannot
    have a dense B with a broadcast A."""
    for P in (2, 3, 5, 13, 17, 63, 64, 65):
        for sa, sb in (((100, P), (P,)), ((100, P), (100, 1)), ((P,), (100, P)),
                       ((100, 1), (100, P))):
            f, (n, ga, gb) = family("Sub", "int16", sa, sb)
            assert f == "repeated_block" and n == [100, P], (sa, sb, f, n)
        # both broadcast: the outer-product row kernel when rows are long
        # whole packs, else the general kernel -- never the block kernel
        want = "inner_vector_outer" if P >= 64 and P % 4 == 0 else "general_strided"
        assert family("Add", "float32", (100, 1), (1, P))[0] == want
        assert family("PRelu", "float32", (100, P), (P,))[0] == "repeated_block"


def test_prelu_one_dimensional_slope_plans_per_channel():
    """A 1-D PRelu slope of C > 1 elements on data of rank >= 2 is per channel
    (0verkilll/onnx ops, PReluOp): accepted exactly where the oracle accepts it,
    and planned as its [C, 1, ..., 1] form."""
    d = eb.Descriptor("PRelu", "float32")
    for sa in small_shapes():
        for c in (0, 1, 2, 3):
            try:
                want = oracle.output_shape("PRelu", sa, (c,))
            except ValueError:
                want = None
            try:
                p = eb.Plan(d, sa, (c,))
            except eb.EbinError as e:
                assert e.code == "incompatible_shapes" and want is None, (sa, c)
                continue
            assert p.output_shape == want == tuple(sa), (sa, c)
            if len(sa) >= 2 and c != 1 and p.numel:
                q = eb.Plan(d, sa, (c,) + (1,) * (len(sa) - 2))
                assert p.family == q.family and p.geometry() == q.geometry(), (sa, c)
                q.close()
            p.close()
    f, (n, ga, gb) = family("PRelu", "bfloat16", (8, 64, 256, 256), (64,))
    assert f == "inner_vector_outer" and n == [8, 64, 65536] and gb == [0, 1, 0]
    for sa in ((2, 8, 5, 8), (2, 8, 5, 7)):
        assert eb.Plan(d, sa, (8,)).output_shape == sa
    with pytest.raises(eb.EbinError):
        eb.Plan(d, (2, 7, 5, 8), (8,))            # the length is the last extent, not C


def test_one_way_broadcasts():
    for op, sb in (("PRelu", (3, 4)), ("BatchNormalization", (4, 5)), ("Clip", (3,))):
        d = eb.Descriptor(op, "float32")
        with pytest.raises(eb.EbinError) as e:
            eb.Plan(d, (3, 1), sb)
        assert e.value.code == "incompatible_shapes"
    d = eb.Descriptor("BatchNormalization", "float32")
    with pytest.raises(eb.EbinError):
        eb.Plan(d, (8,), (4, 8))                     # rank 1 has no channel axis
    assert eb.Plan(d, (2, 8, 3), (4, 8)).output_shape == (2, 8, 3)


def test_rank_and_dims_are_checked():
    d = eb.Descriptor("Add", "float32")
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (1,) * 9, (1,))
    assert e.value.code == "rank_too_large"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (3, -1), (1,))
    assert e.value.code == "invalid_arg"
    assert eb.Plan(d, (1,) * 8, (2,) * 8).output_shape == (2,) * 8


def test_element_counts_are_bounded():
    """Every element count and view span stays below 2^60, so that offsets and
    byte sizes fit in int64: a larger shape is refused, never wrapped.  A zero
    extent makes any shape empty, whatever its other extents."""
    d = eb.Descriptor("Add", "float32")
    big = 1 << 30
    assert eb.Plan(d, (big, big >> 1), (1,)).numel == 1 << 59
    for sa, sb in [((big, big), (1,)),                  # exactly 2^60
                   ((1 << 32, 1 << 32), (1,)),          # 2^64 wraps to 0
                   ((1 << 40,) * 3, ()),                # wraps past 2^64
                   ((1,), (1 << 61,)),                  # B alone
                   ((big, 1), (1, big))]:               # the output alone
        with pytest.raises(eb.EbinError) as e:
            eb.Plan(d, sa, sb)
        assert e.value.code == "invalid_arg", (sa, sb)
    for sa, sb in [((1 << 40, 1 << 40, 0), (1,)), ((0, 1 << 62, 1 << 62), (1,)),
                   ((1 << 40, 0, 1 << 40), (1, 1, 1 << 40))]:
        p = eb.Plan(d, sa, sb)
        assert p.numel == 0 and p.family == "empty", (sa, sb)
        assert p.geometry() == ([0], [0], [0])
    # a view's storage span: (n - 1) * stride summed over its dims
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (2, 64), (64,), strides_a=(1 << 60, 1))
    assert e.value.code == "invalid_arg"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (1 << 20, 64), (64,), strides_a=(1 << 62, 1))
    assert e.value.code == "invalid_arg"
    assert eb.Plan(d, (0, 64), (64,), strides_a=(1 << 62, 1)).family == "empty"
    m = eb.Descriptor("MulAdd", "float32")
    with pytest.raises(eb.EbinError) as e:
        eb.Plan3(m, (big,), (big, 1), (1,))
    assert e.value.code == "invalid_arg"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan3(m, (1,), (1,), (1 << 62, 4))
    assert e.value.code == "invalid_arg"
    p = eb.Plan3(m, (1 << 40, 0), (1 << 40, 1), (1,))
    assert p.numel == 0 and p.family == "empty"


def test_forced_families():
    d = eb.Descriptor("Add", "float32")
    for fam in ("general_strided", "inner_vector_outer"):
        assert eb.Plan(d, (40, 96), (40, 1), family=fam).family == fam
    assert eb.Plan(d, (4096,), (), family="general_strided").family == "general_strided"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (2, 3, 4, 5), (3, 1, 5), family="contiguous")
    assert e.value.code == "family"
    with pytest.raises(eb.EbinError):
        eb.Plan(d, (40, 90), (40, 1), family="inner_vector_outer")   # 90 % 4 != 0
    assert eb.Plan(d, (0, 4), (4,), family="contiguous").family == "empty"


SCALAR_ATTR_OPS = ("Add", "Sub", "Mul", "Div", "Pow", "Max", "Min", "RSub", "RDiv")


def test_with_scalar_descriptor_rules():
    """ncnn binaryop's with_scalar (operators.md, binaryop): the nine operation
    types, on floating types only (the page gives b as a float)."""
    for op in eb.OPS:
        for dt in ALL_DTYPES:
            legal = oracle.type_allowed(op, dt)
            try:
                eb.Descriptor(op, dt, scalar_b=0.5).close()
                got = "ok"
            except eb.EbinError as e:
                got = e.code
            if not legal:
                assert got == "unsupported_type", (op, dt, got)
            elif op in SCALAR_ATTR_OPS and dt in ("float32", "float16", "bfloat16", "float64"):
                assert got == "ok", (op, dt, got)
            else:
                assert got == "invalid_attr", (op, dt, got)
    bad = eb.ebin_attrs(0, 0, 1e-5, 1, 1, 2, 0.0)
    with pytest.raises(eb.EbinError) as e:
        eb.ebin_descriptor_create(eb.OPS["Add"], 28, bad, 1, 1)
    assert e.value.code == "invalid_attr"


def test_with_scalar_plans_ignore_shape_b():
    d = eb.Descriptor("Mul", "float32", scalar_b=3.0)
    p1 = eb.Plan(d, (64, 1000), (7, 1, 3))                 # any shape B: not read
    p2 = eb.Plan(d, (64, 1000), ())
    assert p1.handle == p2.handle                          # one cached plan
    assert p1.output_shape == (64, 1000) and p1.family == "right_scalar"
    assert eb.Plan(d, (), ()).numel == 1
    assert eb.Plan(d, (64, 1000), (), family="general_strided").family == "general_strided"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (64, 1000), (), family="inner_vector_outer")
    assert e.value.code == "family"
    # B may be NULL: an empty execute checks nothing else
    assert eb.Plan(d, (0, 5), ()).family == "empty"


def test_three_input_plans():
    """MulAdd plans: broadcast(broadcast(A, B), C) against the oracle, the row
    family for the pages' scalar and per-channel patterns, the shape-C cache key
    and the separation from two-input entry points."""
    d = eb.Descriptor("MulAdd", "float32")
    rng = np.random.default_rng(5)
    dims = [()] + [s for r in (1, 2, 3) for s in itertools.product((0, 1, 2, 3), repeat=r)]
    for _ in range(400):
        sh = [dims[i] for i in rng.integers(0, len(dims), 3)]
        try:
            want = oracle.output_shape3(*sh)
        except ValueError:
            with pytest.raises(eb.EbinError) as e:
                eb.Plan3(d, *sh)
            assert e.value.code == "incompatible_shapes"
            continue
        p = eb.Plan3(d, *sh)
        assert p.output_shape == want and p.numel == int(np.prod(want))
    x = (8, 64, 256, 256)
    assert eb.Plan3(d, x, (1,), x).family == "right_scalar"
    assert eb.Plan3(d, x, (1, 64, 1, 1), x).family == "inner_vector_outer"
    assert eb.Plan3(d, (4096,), (4096,), (4096,)).family == "contiguous"
    assert eb.Plan3(d, (3, 1, 5), (1, 4, 1), (4, 5)).family == "general_strided"
    p1, p2 = eb.Plan3(d, (64, 64), (64,), (64, 64)), eb.Plan3(d, (64, 64), (64,), (64, 1))
    assert p1.handle != p2.handle                          # shape C is part of the key
    assert eb.Plan3(d, (64, 64), (64,), (64, 64)).handle == p1.handle
    assert eb.Plan3(d, x, (1,), x, family="general_strided").family == "general_strided"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan3(d, x, (1,), x, family="inner_vector_outer")
    assert e.value.code == "family"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (4,), (4,))                             # three inputs need plan_create3
    assert e.value.code == "invalid_arg"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan3(eb.Descriptor("Add", "float32"), (4,), (4,), (4,))
    assert e.value.code == "invalid_arg"
    pe = eb.Plan3(d, (0, 4), (4,), (4,))
    assert pe.family == "empty"
    # (stream 0: no CUDA call is reached on these paths)
    eb.ebin_execute3(pe.handle, None, None, None, None, None)   # nothing to do, nothing read
    with pytest.raises(eb.EbinError) as e:
        eb.ebin_execute(p1.handle, 16, 16, 16, None)       # a three-input plan
    assert e.value.code == "invalid_arg"
    with pytest.raises(eb.EbinError) as e:
        eb.ebin_execute3(p1.handle, 16, None, 16, 4096, None)
    assert e.value.code == "invalid_arg"
    with pytest.raises(eb.EbinError) as e:                 # C overlaps out, not identical
        eb.ebin_execute3(p1.handle, 1 << 20, 2 << 20, 3 << 20, (3 << 20) + 64, None)
    assert e.value.code == "alias"


def _geometry_offsets(plan, numel):
    """Element offsets of A and B for every output index, from the plan's
    coalesced geometry (extents n, strides sa, sb)."""
    n, sa, sb = plan.geometry()
    f = np.arange(numel, dtype=np.int64)
    oa = np.zeros(numel, np.int64)
    ob = np.zeros(numel, np.int64)
    for d in range(len(n) - 1, -1, -1):
        digit = f % n[d]
        f //= n[d]
        oa += digit * sa[d]
        ob += digit * sb[d]
    return oa, ob


VIEWS = [  # (base length, shape, element strides) of A; B dense of the given shape
    (64 * 48, (48, 64), (1, 48), (64,)),               # transpose
    (200 * 9, (100, 3), (18, 3), (100, 1)),             # every other row, every third column
    (64, (7, 64), (0, 1), (7, 64)),                     # expanded rows
    (64 * 1008, (64, 1000), (1008, 1), (1000,)),         # padded rows, 16-byte aligned
    (64 * 1001, (64, 1000), (1001, 1), (64, 1)),         # padded rows, not aligned
    (5 * 6 * 7 * 3, (5, 6, 7), (126, 21, 3), (6, 1)),    # inner stride 3
]


def test_strided_views_map_every_element():
    """Each view is built over arange(base) so that its values are its storage
    offsets: the geometry must address exactly numpy's broadcast of the view."""
    d = eb.Descriptor("Add", "float32")
    for base, shape, strides, shape_b in VIEWS:
        view = np.lib.stride_tricks.as_strided(np.arange(base, dtype=np.int64), shape,
                                               [x * 8 for x in strides])
        p = eb.Plan(d, shape, shape_b, strides_a=strides)
        out_shape = np.broadcast_shapes(shape, shape_b)
        assert p.output_shape == out_shape
        oa, ob = _geometry_offsets(p, p.numel)
        want_a = np.broadcast_to(view, out_shape).reshape(-1)
        want_b = np.broadcast_to(np.arange(int(np.prod(shape_b))).reshape(shape_b),
                                 out_shape).reshape(-1)
        assert (oa == want_a).all() and (ob == want_b).all(), (shape, strides)


def test_strided_view_rules():
    d = eb.Descriptor("Add", "float32")
    dense = eb.Plan(d, (64, 1000), (1000,))
    assert eb.Plan(d, (64, 1000), (1000,), strides_a=(1000, 1)).handle == dense.handle
    # padded rows: not dense, so the inner-vector traversal (any aligned run stride)
    assert eb.Plan(d, (64, 1000), (1000,), strides_a=(1008, 1)).family == "inner_vector_outer"
    assert eb.Plan(d, (64, 1000), (1000,), strides_a=(1001, 1)).family == "general_strided"
    assert eb.Plan(d, (64, 1000), (1000,), strides_a=(1008, 1),
                   family="general_strided").family == "general_strided"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (64, 1000), (1000,), strides_a=(-1000, 1))
    assert e.value.code == "invalid_arg"
    bn = eb.Descriptor("BatchNormalization", "float32")
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(bn, (2, 4, 8), (4, 4), strides_b=(8, 2))
    assert e.value.code == "invalid_arg"
    assert eb.Plan(bn, (2, 4, 8), (4, 4), strides_a=(64, 16, 2)).family in (
        "general_strided", "inner_vector_outer")
    # a strided A is never in place: the identical buffer is ALIAS too
    p = eb.Plan(d, (48, 64), (64,), strides_a=(1, 48))
    with pytest.raises(eb.EbinError) as e:
        eb.ebin_execute(p.handle, 1 << 20, 4 << 20, 1 << 20, None)
    assert e.value.code == "alias"


PARAM_BLOCK_OPS = ("BatchNormalization", "BiasPRelu", "BiasPReluBN")


def test_mixed_type_pow_rules():
    """Pow's exponent may have any non-BOOL type (typed scalar adapters), and the
    parameter block of BatchNormalization, BiasPRelu and BiasPReluBN may be
    float32 beside float16, bfloat16 or float64 x (scale, bias, mean and var
    in x's type or float32); every other pair needs equal types.  Mixed Pow
    plans run the general kernel."""
    for op in eb.OPS:
        for ta in ALL_DTYPES:
            for tb in ALL_DTYPES:
                if ta == tb:
                    continue
                legal = ((op == "Pow" and oracle.type_allowed("Pow", ta) and tb != "bool") or
                         (op in PARAM_BLOCK_OPS and tb == "float32" and
                          ta in ("float16", "bfloat16", "float64")))
                try:
                    eb.Descriptor(op, ta, dtype_b=tb).close()
                    got = True
                except eb.EbinError as e:
                    assert e.code == "unsupported_type"
                    got = False
                assert got == legal, (op, ta, tb)
    d = eb.Descriptor("Pow", "bfloat16", dtype_b="uint8")
    assert d.out_dtype == "bfloat16"
    assert eb.Plan(d, (300, 256), (256,)).family == "general_strided"
    assert eb.Plan(d, (0, 256), (256,)).family == "empty"
    with pytest.raises(eb.EbinError) as e:
        eb.Plan(d, (300, 256), (256,), family="repeated_block")
    assert e.value.code == "family"


@pytest.mark.parametrize("op", PARAM_BLOCK_OPS)
@pytest.mark.parametrize("dtype", ["float16", "bfloat16", "float64"])
def test_float32_parameter_block_keeps_the_family(op, dtype):
    """A float32 parameter block is read one value per channel row, so it plans
    exactly as a block of x's own type: same family and geometry for the
    per-channel, channels-innermost, single-row and one-channel layouts."""
    rows = {"BatchNormalization": 4, "BiasPRelu": 2, "BiasPReluBN": 6}[op]
    same, mixed = eb.Descriptor(op, dtype), eb.Descriptor(op, dtype, dtype_b="float32")
    assert mixed.out_dtype == dtype and mixed.dtype_b == "float32"
    for xs in [(8, 64, 256, 256), (2, 3, 5, 7), (1000, 64), (1, 48), (4, 1, 16, 16),
               (3, 5, 0, 2)]:
        bs = (rows, xs[1])
        a, b = eb.Plan(same, xs, bs), eb.Plan(mixed, xs, bs)
        assert (b.family, b.output_shape) == (a.family, a.output_shape), (op, dtype, xs)
        assert b.geometry() == a.geometry()
        g = eb.Plan(mixed, xs, bs, family="general_strided")
        assert g.family == ("empty" if 0 in xs else "general_strided")
    for bad in ("float16", "bfloat16", "int32"):
        if bad != dtype:
            with pytest.raises(eb.EbinError) as e:
                eb.Descriptor(op, dtype, dtype_b=bad)
            assert e.value.code == "unsupported_type"


def test_binary_helper_parameter_block_types():
    """binary() takes the parameter block's type from its tensor: a float16
    block beside bfloat16 x is refused by the descriptor rule, before any
    memory check; a float32 block passes the rule and then meets the
    pinned-memory check of CPU tensors."""
    torch = pytest.importorskip("torch")
    x = torch.zeros((2, 3, 4), dtype=torch.bfloat16)
    with pytest.raises(eb.EbinError) as e:
        eb.binary("BatchNormalization", x, torch.ones((4, 3), dtype=torch.float16))
    assert e.value.code == "unsupported_type"
    with pytest.raises(eb.EbinError) as e:
        eb.binary("BiasPRelu", x, torch.ones((2, 3), dtype=torch.float64))
    assert e.value.code == "unsupported_type"
    with pytest.raises(ValueError, match="pinned"):
        eb.binary("BiasPReluBN", x, torch.ones((6, 3), dtype=torch.float32))


def test_plan_cache_is_an_8_entry_lru():
    eb.ebin_plan_cache_clear()
    d = eb.Descriptor("Sub", "int32")
    plans = [eb.Plan(d, (i + 1, 3), (3,)) for i in range(8)]
    h, m, s = eb.ebin_plan_cache_stats()
    assert (h, m, s) == (0, 8, 8)
    again = eb.Plan(d, (1, 3), (3,))                  # hit; becomes most recent
    assert again.handle == plans[0].handle
    assert eb.ebin_plan_cache_stats() == (1, 8, 8)
    eb.Plan(d, (100, 3), (3,))                        # miss; evicts the LRU entry (2, 3)
    assert eb.ebin_plan_cache_stats() == (1, 9, 8)
    fresh = eb.Plan(d, (2, 3), (3,))                  # was evicted: a miss, a new plan
    assert eb.ebin_plan_cache_stats()[1] == 10
    assert fresh.handle != plans[1].handle
    # the evicted plan is still usable by its holder
    assert plans[1].output_shape == (2, 3)
    eb.Plan(d, (1, 3), (3,))
    assert eb.ebin_plan_cache_stats()[0] == 2


def test_destroyed_descriptor_never_hits():
    eb.ebin_plan_cache_clear()
    d = eb.Descriptor("Mul", "float32")
    p = eb.Plan(d, (5, 7), (7,))
    old_id = d.id
    d.close()
    assert p.output_shape == (5, 7)                   # held plan outlives its descriptor
    d2 = eb.Descriptor("Mul", "float32")
    assert d2.id != old_id
    eb.Plan(d2, (5, 7), (7,))
    h, m, _ = eb.ebin_plan_cache_stats()
    assert h == 0 and m == 2


def test_empty_execute_reads_nothing():
    d = eb.Descriptor("Div", "int32")
    p = eb.Plan(d, (0, 5), (5,))
    before = eb.ebin_launch_count()
    eb.ebin_execute(p.handle, None, None, None, None)
    assert eb.ebin_launch_count() == before


def test_alias_rule():
    d = eb.Descriptor("Add", "float32")
    p = eb.Plan(d, (4, 8), (8,))
    base = 1 << 40                                     # never dereferenced: the check fails first
    with pytest.raises(eb.EbinError) as e:            # A overlaps out, shifted by one element
        eb.ebin_execute(p.handle, base, base + 4096, base + 4, None)
    assert e.value.code == "alias"
    with pytest.raises(eb.EbinError) as e:            # broadcast B inside out
        eb.ebin_execute(p.handle, base + 8192, base + 16, base, None)
    assert e.value.code == "alias"
    dc = eb.Descriptor("Greater", "float32")
    pc = eb.Plan(dc, (4, 8), (4, 8))
    with pytest.raises(eb.EbinError) as e:            # BOOL out over a float input
        eb.ebin_execute(pc.handle, base, base + 4096, base, None)
    assert e.value.code == "alias"
    db = eb.Descriptor("BatchNormalization", "float32")
    pb = eb.Plan(db, (4, 8), (4, 8))
    with pytest.raises(eb.EbinError) as e:            # parameter block never aliases out
        eb.ebin_execute(pb.handle, base + 4096, base, base, None)
    assert e.value.code == "alias"


def test_null_buffers_rejected():
    d = eb.Descriptor("Add", "float32")
    p = eb.Plan(d, (4,), (4,))
    with pytest.raises(eb.EbinError) as e:
        eb.ebin_execute(p.handle, None, 16, 32, None)
    assert e.value.code == "invalid_arg"


def test_dtype_sizes_and_strings():
    for name, code in eb.DTYPES.items():
        assert eb.ebin_dtype_size(code) == eb.ITEMSIZE[name]
    assert eb.ebin_status_string(7) == "input aliases the output"


def test_execute_mapped_host_checks():
    """ebin_execute_mapped refuses before any device work: NULL buffers, a
    three-input plan, and host memory that is not pinned and mapped (here,
    pageable numpy memory; the check runs without a GPU too)."""
    import numpy as np
    d = eb.descriptor("Add", "float32")
    p = eb.Plan(d, (1024,), (1024,))
    a = np.zeros(1024, np.float32)
    o = np.zeros(1024, np.float32)
    pe = eb.Plan(d, (0, 4), (4,))
    eb.ebin_execute_mapped(pe.handle, None, None, None, None)       # nothing to do
    for args in ((None, a.ctypes.data, o.ctypes.data), (a.ctypes.data, a.ctypes.data, None),
                 (a.ctypes.data, a.ctypes.data, o.ctypes.data)):
        with pytest.raises(eb.EbinError, match="invalid_arg"):
            eb.ebin_execute_mapped(p.handle, *args, None)
    p3 = eb.Plan3(eb.descriptor("MulAdd", "float32"), (8,), (8,), (8,))
    with pytest.raises(eb.EbinError, match="invalid_arg"):
        eb.ebin_execute_mapped(p3.handle, a.ctypes.data, a.ctypes.data, o.ctypes.data, None)
    # the three-input form: pageable buffers and a two-input plan are refused too
    for plan in (p3, p):
        with pytest.raises(eb.EbinError, match="invalid_arg"):
            eb.ebin_execute3_mapped(plan.handle, a.ctypes.data, a.ctypes.data, a.ctypes.data,
                                    o.ctypes.data, None)


def test_plans_and_descriptors_from_many_host_threads():
    """The C ABI is thread-safe: eight host threads create descriptors and
    plans (hits, misses and evictions of the shared 8-entry LRU) and release
    them, concurrently (ctypes drops the GIL around each call)."""
    import threading
    import numpy as np
    shapes = [((64, 32), (32,)), ((8, 16, 4), (16, 1)), ((5, 1, 7), (1, 6, 7)), ((3,), ()),
              ((2, 3, 4, 5), (3, 1, 5)), ((100,), (100,)), ((9, 9), (9, 1)), ((4, 1), (1, 4)),
              ((7, 2, 3), (2, 3)), ((1, 11), (11, 1))]
    want = {(sa, sb): tuple(np.broadcast_shapes(sa, sb)) for sa, sb in shapes}
    errors = []

    def work(tid):
        try:
            for it in range(300):
                sa, sb = shapes[(tid * 7 + it) % len(shapes)]
                op = ("Add", "Mul", "Greater")[it % 3]
                d = eb.ebin_descriptor_create(eb.OPS[op], 18, None, eb.DTYPES["float32"],
                                              eb.DTYPES["float32"])
                h = eb.ebin_plan_create(d, sa, sb)
                assert eb.ebin_plan_output_shape(h) == want[(sa, sb)]
                eb.ebin_plan_release(h)
                eb.ebin_descriptor_destroy(d)
        except Exception as e:          # reported below, in the main thread
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=work, args=(t,)) for t in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]
    hits, misses, size = eb.ebin_plan_cache_stats()
    assert size <= eb.PLAN_CACHE_CAPACITY


def test_concurrent_misses_keep_one_entry_per_key(tmp_path):
    """Threads that miss on one key at the same time all receive the same
    plan: the cache keeps a single entry per key.  Python threads are too
    slow to meet inside the planner, so a C driver (tests/plan_cache_race.c)
    releases eight pthreads together on each of 2000 new keys."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(os.path.abspath(eb.lib._name))
    exe = str(tmp_path / "plan_cache_race")
    subprocess.run([gcc, "-O2", "-I", os.path.join(os.path.dirname(here), "include"),
                    os.path.join(here, "plan_cache_race.c"), "-o", exe, "-L", libdir,
                    "-lebin", "-lpthread", "-Wl,-rpath," + libdir], check=True)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert int(run.stdout) == 0, "keys that came back as more than one plan: " + run.stdout


def test_binary_helper_refuses_b_of_another_type():
    """binary() checks B's type against the descriptor before it touches any
    memory (no GPU needed): Pow's exponent may differ only when declared."""
    torch = pytest.importorskip("torch")
    a = torch.zeros(4, 8)
    with pytest.raises(ValueError, match="takes B of float32"):
        eb.binary("Add", a, torch.zeros(8, dtype=torch.float16))
    with pytest.raises(ValueError, match="takes B of float32"):
        eb.binary("Pow", a, torch.zeros(8, dtype=torch.int32))
    with pytest.raises(ValueError, match="takes B of int32"):
        eb.binary("Pow", a, torch.zeros(8), dtype_b="int32")
    # the declared exponent type passes the type check (then wants pinned memory)
    with pytest.raises(ValueError, match="pinned"):
        eb.binary("Pow", a, torch.zeros(8, dtype=torch.int32), dtype_b="int32")
