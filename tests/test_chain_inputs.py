"""The exhaustive 16-bit inputs of the GPU parity test for BatchNormalization
and BiasPReluBN (test_prepared_division_on_every_16bit_value) can tell the
chain's last two steps, y = RN(RN(q * scale) + bias), from the same steps
merged into one fused multiply-add, y = RN(q * scale + bias).

The merge is a plausible compiler-made mistake: a paired binary32 multiply
followed by a paired add was merged into one fused multiply-add even with
contraction switched off, which moved a few outputs per million by one unit in
the last place.  For every operator and 16-bit type this file checks on the CPU
that the GPU test's inputs (ordinary parameters) hold at least one element
where the merged tail gives another 16-bit result than the oracle, so that the
GPU test would fail on such a build.  It also checks that the same chain
written out with numpy's binary32 operations agrees with the oracle bit for bit
everywhere else.  The fused multiply-add is emulated in binary64 (the product
exact, the sum rounded to binary64 and then to binary32); that can differ from
a true fused multiply-add only when the binary64 sum lies within one of its
units of a binary32 rounding midpoint, which the count allows for by asking
for a single element.
"""
import numpy as np
import pytest

import datagen
import oracle
from conftest import _is_nan
from engine_util import chain_params, every_16bit_value

SHAPE = (16, 64, 64, 64)        # every 16-bit pattern once per channel


def _widen(x, dtype):
    if dtype == "float16":
        return x.astype(np.float32)
    return (x.astype(np.uint32) << 16).view(np.float32)


def _round16(y, dtype):
    """binary32 -> 16-bit storage, nearest even (NaN positions are not used)."""
    if dtype == "float16":
        with np.errstate(over="ignore"):
            return y.astype(np.float16).view(np.uint16)
    u = y.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _chain(op, x, rows, fused):
    """The chain in numpy binary32 steps; fused: the last multiply and add as
    one fused multiply-add (emulated in binary64)."""
    with np.errstate(all="ignore"):
        if op == "BatchNormalization":
            scale, bias, mean, var = rows
            t = x
        else:
            b0, slope, scale, bias, mean, var = rows
            t = x + b0
            t = np.where(t >= 0, t, slope * t).astype(np.float32)
        q = (t - mean) / np.sqrt(var + np.float32(1e-5))
        if fused:
            return (q.astype(np.float64) * scale.astype(np.float64) +
                    bias.astype(np.float64)).astype(np.float32)
        return q * scale + bias


@pytest.mark.parametrize("op", ["BatchNormalization", "BiasPReluBN"])
@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_exhaustive_inputs_tell_a_fused_tail_apart(op, dtype):
    C = SHAPE[1]
    x = every_16bit_value(SHAPE).view(datagen.STORAGE[dtype])
    b = datagen.float_to(chain_params(op, C, 90, False), dtype)
    want = np.ascontiguousarray(oracle.run_params(op, x, b, dtype, dtype))
    keep = ~_is_nan(want, dtype).reshape(-1)
    wbits = want.view(np.uint16).reshape(-1)[keep]

    xf = _widen(x.view(np.uint16) if dtype == "bfloat16" else x, dtype).reshape(SHAPE[0], C, -1)
    bf = _widen(b, dtype)
    rows = [bf[i][None, :, None] for i in range(bf.shape[0])]
    plain = _round16(_chain(op, xf, rows, False), dtype).reshape(-1)[keep]
    fused = _round16(_chain(op, xf, rows, True), dtype).reshape(-1)[keep]
    assert (plain == wbits).all(), (op, dtype, int((plain != wbits).sum()))
    assert (fused != wbits).sum() >= 1, (op, dtype)
