import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


FLOAT_BITS = {"float32": np.uint32, "float16": np.uint16, "bfloat16": np.uint16,
              "float64": np.uint64}


def _is_nan(arr: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "float32":
        u = arr.view(np.uint32)
        return (u & 0x7FFFFFFF) > 0x7F800000
    if dtype == "float16":
        u = arr.view(np.uint16)
        return (u & 0x7FFF) > 0x7C00
    if dtype == "bfloat16":
        u = arr.view(np.uint16)
        return (u & 0x7FFF) > 0x7F80
    if dtype == "float64":
        u = arr.view(np.uint64)
        return (u & np.uint64(0x7FFFFFFFFFFFFFFF)) > np.uint64(0x7FF0000000000000)
    return np.zeros(arr.shape, bool)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    """Bit-identical, except that any NaN matches any NaN; signed zeros compare by bits."""
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if dtype in FLOAT_BITS:
        nan_g, nan_w = _is_nan(got, dtype), _is_nan(want, dtype)
        gb = got.view(FLOAT_BITS[dtype])
        wb = want.view(FLOAT_BITS[dtype])
        bad = (gb != wb) & ~(nan_g & nan_w)
    else:
        bad = got != want
    if bad.any():
        pos = np.flatnonzero(bad.reshape(-1))
        i = pos[0]
        raise AssertionError("%s: %d of %d elements differ; first at flat %d: got %r want %r"
                             % (what, pos.size, bad.size, i, got.reshape(-1)[i],
                                want.reshape(-1)[i]))


def ulp_distance(got: np.ndarray, want: np.ndarray, dtype: str) -> np.ndarray:
    """Distance in units in the last place of ``dtype`` (NaN vs NaN = 0, NaN vs number = huge)."""
    ut = FLOAT_BITS[dtype]
    if dtype == "float64":
        # signed-magnitude bits to a monotone integer line; exact distance when
        # both have one sign, capped when they straddle zero (no int64 overflow)
        g = np.ascontiguousarray(got).view(np.int64)
        w = np.ascontiguousarray(want).view(np.int64)
        mag = np.int64(0x7FFFFFFFFFFFFFFF)
        mg, mw = g & mag, w & mag
        same = (g < 0) == (w < 0)
        d = np.where(same, np.abs(mg - mw), np.minimum(mg, 1 << 40) + np.minimum(mw, 1 << 40))
    else:
        g = np.ascontiguousarray(got).view(ut).astype(np.int64)
        w = np.ascontiguousarray(want).view(ut).astype(np.int64)
        width = 32 if ut == np.uint32 else 16
        sign = 1 << (width - 1)

        def ordered(u):
            return np.where(u & sign, -(u & (sign - 1)), u)

        d = np.abs(ordered(g) - ordered(w))
    ng, nw = _is_nan(np.ascontiguousarray(got), dtype), _is_nan(np.ascontiguousarray(want), dtype)
    d = np.where(ng & nw, 0, d)
    d = np.where(ng ^ nw, 1 << 40, d)
    return d
