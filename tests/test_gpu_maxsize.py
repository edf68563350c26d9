"""Parity past the 32-bit index range: outputs of more than 2^31 and 2^32
elements, and buffers larger than 4 GiB.

The row kernels divide tile and prefix indices in 32 bits unless some index
may reach 2^32 (then in 64 bits); the flat kernels and every element offset
use 64-bit arithmetic.  These cases put outputs across both limits, with a
ragged tail, and check sampled outputs against the oracle: the oracle maps
each sampled flat output index to its A and B offsets, the test gathers those
input elements from the device and the oracle evaluates them.  The samples
hold the whole first and last tiles and the elements on either side of
2^31 and 2^32 (and of 2^35, where 16-byte pack indices of one-byte elements
pass 2^31), where a truncated index would land.

Inputs are drawn on the device from a seeded torch generator (a host copy of
several GiB would dominate the test); the oracle reads back the elements it
needs, so it sees exactly what the kernel read.
"""
import numpy as np
import pytest

import oracle
from conftest import assert_bits_equal

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TORCH = {"uint8": torch.uint8, "float32": torch.float32, "int64": torch.int64}
NP = {"uint8": np.uint8, "float32": np.float32, "int64": np.int64}


def _device_input(shape, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    n = int(np.prod(shape))
    if dtype == "float32":
        return torch.randn(n, dtype=torch.float32, device="cuda", generator=g)
    if dtype == "uint8":
        return torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    return torch.randint(-(1 << 62), 1 << 62, (n,), dtype=torch.int64, device="cuda",
                         generator=g)


def _samples(numel, seed=2024):
    rng = np.random.default_rng(seed)
    edge = 1 << 14
    parts = [np.arange(min(edge, numel)), np.arange(max(numel - edge, 0), numel),
             rng.integers(0, numel, 1 << 18)]
    for wall in (1 << 31, 1 << 32, 1 << 35):
        if wall < numel:
            parts.append(np.arange(max(wall - edge, 0), min(wall + edge, numel)))
    return np.unique(np.concatenate(parts)).astype(np.int64)


def _gather(t, idx):
    return t[torch.from_numpy(idx).cuda()].cpu().numpy()


CASES = [
    # (op, dtype, shape A, shape B, family)
    ("BitwiseXor", "uint8", ((1 << 32) + 4099,), ((1 << 32) + 4099,), "contiguous"),
    ("Add", "uint8", ((1 << 32) + 7,), (1,), "right_scalar"),
    ("Add", "uint8", ((1 << 32) + 7, 1), (1, 2), "general_strided"),
    ("Mul", "float32", (2, 64, (1 << 24) + 4), (1, 64, 1), "inner_vector_outer"),
    ("BitwiseXor", "int64", ((1 << 28) + 5, 4), (4,), "repeated_block"),
    # rows off the pack width: the periodic kernel's 32-bit indices just below
    # 2^31 elements, and the general kernel past it
    ("Add", "uint8", (715827882, 3), (3,), "repeated_block"),
    ("Sub", "uint8", ((1 << 31) + 3, 3), ((1 << 31) + 3, 1), "repeated_block"),
    # one value per row past 2^31 packs of 16 bytes (2^35 elements): the flat
    # per-row kernel's 64-bit pack indices (two 32 GiB buffers)
    ("Add", "uint8", ((1 << 24) + 3, 2048), ((1 << 24) + 3, 1), "repeated_block"),
]


@pytest.mark.parametrize("op,dtype,sa,sb,family", CASES,
                         ids=["xor_u8_2p32", "add_u8_scalar_2p32", "add_u8_general_wide",
                              "mul_f32_channel_2p31", "xor_i64_rows_8GiB",
                              "add_u8_block3_below_2p31", "sub_u8_rows3_past_2p31",
                              "add_u8_rows_past_2p31_packs"])
def test_past_32bit_indices(op, dtype, sa, sb, family):
    import broadcast_elementwise_gb300 as eb
    plan = eb.Plan(eb.descriptor(op, dtype), sa, sb)
    if family is not None:
        assert plan.family == family
    numel = plan.numel
    assert numel == int(np.prod(oracle.output_shape(op, sa, sb)))
    a = _device_input(sa, dtype, 11)
    b = _device_input(sb, dtype, 12)
    out = torch.empty(numel, dtype=TORCH[dtype], device="cuda")
    eb.execute(plan, a, b, out)
    torch.cuda.synchronize()
    assert eb.get_device_status() == 0
    idx = _samples(numel)
    oa, ob = oracle.offsets(sa, sb, idx)
    av, bv = _gather(a, oa), _gather(b, ob)
    want, st = oracle.run(op, av, bv, dtype)
    assert st == 0
    got = _gather(out, idx)
    assert_bits_equal(got, want, dtype, "%s %s %s x %s" % (op, dtype, sa, sb))
    del a, b, out
    torch.cuda.empty_cache()


def test_muladd_per_row_past_2p31_packs():
    """MulAdd x * s + y with s one value per row past 2^31 packs of 16 bytes
    (2^35 uint8 elements): the three-input per-row flat kernel's 64-bit pack
    indices (three 32 GiB buffers).  x and y are shaped like the output, so
    their offsets are the output index; s's come from the oracle's mapping."""
    import broadcast_elementwise_gb300 as eb
    sx, ss = ((1 << 24) + 3, 2048), ((1 << 24) + 3, 1)
    plan = eb.Plan3(eb.descriptor("MulAdd", "uint8"), sx, ss, sx)
    assert plan.family == "inner_vector_outer"
    numel = plan.numel
    assert numel // 16 >= 1 << 31
    x = _device_input(sx, "uint8", 21)
    s = _device_input(ss, "uint8", 22)
    y = _device_input(sx, "uint8", 23)
    out = torch.empty(numel, dtype=torch.uint8, device="cuda")
    eb.execute3(plan, x.data_ptr(), s.data_ptr(), y.data_ptr(), out.data_ptr())
    torch.cuda.synchronize()
    idx = _samples(numel)
    ox, os_ = oracle.offsets(sx, ss, idx)
    want = oracle.run3("MulAdd", _gather(x, ox), _gather(s, os_), _gather(y, ox), "uint8")
    assert_bits_equal(_gather(out, idx), want, "uint8", "MulAdd uint8 %s * %s + %s" % (sx, ss, sx))
    del x, s, y, out
    torch.cuda.empty_cache()
