"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (same plans, same kernels, inputs resident on the device).

Outputs small enough for the oracle to finish in seconds are compared in full;
the 2^28-element and 2^30-element outputs are compared on sampled indices
(the oracle evaluates each sampled element from its full multi-index), plus
the whole first and last 64 Ki elements, which hold the tails of the tiling.
"""
import numpy as np
import pytest

import oracle
from conftest import assert_bits_equal
from datagen import workloads
from engine_util import run_engine

pytestmark = pytest.mark.gpu

FULL_COMPARE_LIMIT = 1 << 25


def oracle_kwargs(attrs):
    kw = {}
    if "fmod" in attrs:
        kw["fmod"] = attrs["fmod"]
    if "direction" in attrs:
        kw["direction"] = attrs["direction"]
    if "epsilon" in attrs:
        kw["eps"] = attrs["epsilon"]
    return kw


NAMES = [c.name for c in workloads.cases()]


def _view_parity(c, a, base):
    """A workload whose B is a strided view of the buffer `base`: the engine
    reads the view in place; the oracle evaluates sampled outputs on the
    view's contiguous copy."""
    import torch
    import broadcast_elementwise_gb300 as eb
    from engine_util import to_device
    desc = eb.descriptor(c.op, c.dtype, **c.attrs)
    plan = eb.Plan(desc, c.shape_a, c.shape_b, strides_b=c.strides_b)
    assert plan.family == c.family
    osz = eb.ITEMSIZE[desc.out_dtype]
    out = torch.empty(plan.numel * osz, dtype=torch.uint8, device="cuda")
    eb.execute(plan, to_device(a), to_device(base), out)
    bits = eb.get_device_status()
    got = out.cpu().numpy().view(a.dtype)
    b = np.ascontiguousarray(np.lib.stride_tricks.as_strided(
        base, c.shape_b, [x * base.itemsize for x in c.strides_b]))
    rng = np.random.default_rng(12345)
    numel = got.size
    edge = 1 << 16
    idx = np.unique(np.concatenate([np.arange(edge), np.arange(numel - edge, numel),
                                    rng.integers(0, numel, 1 << 21)]))
    want, wbits = oracle.run(c.op, a, b, c.dtype, idx=idx)
    assert_bits_equal(got[idx], want, c.dtype, c.name + " (sampled)")
    assert bits == wbits == 0


@pytest.mark.parametrize("name", NAMES)
def test_workload_parity(name):
    c = workloads.by_name(name)
    a, b = c.make_a(), c.make_b()
    if c.make_c is not None:                       # three inputs (MulAdd)
        from engine_util import run_engine3
        cc = c.make_c()
        got, fam = run_engine3(c.op, c.dtype, a, b, cc)
        assert fam == c.family
        rng = np.random.default_rng(12345)
        numel = got.size
        idx = np.unique(np.concatenate([np.arange(1 << 16), np.arange(numel - (1 << 16), numel),
                                        rng.integers(0, numel, 1 << 21)]))
        want = oracle.run3(c.op, a, b, cc, c.dtype, idx=idx)
        assert_bits_equal(got.reshape(-1)[idx], want, c.dtype, name + " (sampled)")
        return
    if c.strides_b is not None:                    # B a view of its buffer
        _view_parity(c, a, b)
        return
    got, bits, fam = run_engine(c.op, c.dtype, a, b, attrs=c.attrs)
    assert fam == c.family
    otype = "bool" if c.op == "Greater" else c.dtype
    numel = got.size
    kw = oracle_kwargs(c.attrs)
    if numel <= FULL_COMPARE_LIMIT:
        want, wbits = oracle.run(c.op, a, b, c.dtype, **kw)
        assert_bits_equal(got, want, otype, name)
        assert bits == wbits
    else:
        rng = np.random.default_rng(12345)
        edge = 1 << 16
        idx = np.unique(np.concatenate([np.arange(edge), np.arange(numel - edge, numel),
                                        rng.integers(0, numel, 1 << 21)]))
        want, _ = oracle.run(c.op, a, b, c.dtype, idx=idx, **kw)
        assert_bits_equal(got.reshape(-1)[idx], want, otype, name + " (sampled)")
        assert bits == 0


def test_greater_rows_are_consistent():
    """Property at full size: every output row is B's row compared against one A value."""
    c = workloads.by_name("greater_f16_outer_broadcast")
    a, b = c.make_a(), c.make_b()
    got, _, _ = run_engine(c.op, c.dtype, a, b)
    got = got.reshape(64, 32, 512, 1024)
    av = a.reshape(64, 512).astype(np.float32)
    bv = b.reshape(32, 1024).astype(np.float32)
    for i in (0, 17, 63):
        for j in (0, 31):
            want = (av[i][:, None] > bv[j][None, :]).astype(np.uint8)
            assert (got[i, j] == want).all()


def test_bitshift_all_counts_at_full_length():
    c = workloads.by_name("bitshift_u32_right_scalar")
    a = c.make_a()
    rng = np.random.default_rng(7)
    idx = rng.integers(0, a.size, 1 << 16)
    for s in range(32):
        b = np.array([s], np.uint32)
        got, bits, _ = run_engine("BitShift", "uint32", a, b, attrs={"direction": 1})
        assert bits == 0
        assert (got[idx] == (a[idx] >> np.uint32(s))).all(), s
