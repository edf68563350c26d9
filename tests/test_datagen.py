"""The seeded input generator: deterministic, chunk-independent, in range."""
import numpy as np

import datagen


def test_counter_based_slices_agree():
    whole = datagen.normal(1, 0, 10000)
    part = datagen.normal(1, 0, 3000, offset=4000)
    assert whole[4000:7000].tobytes() == part.tobytes()
    big = datagen.raw_u32(3, 2, (1 << 22) + 5)          # crosses the threaded chunking
    assert big[(1 << 22) - 3:].tobytes() == datagen.raw_u32(3, 2, 8, offset=(1 << 22) - 3).tobytes()


def test_streams_differ_and_repeat():
    a = datagen.uniform(0, 0, 1000, -1, 1)
    b = datagen.uniform(0, 1, 1000, -1, 1)
    assert not np.array_equal(a, b)
    assert np.array_equal(a, datagen.uniform(0, 0, 1000, -1, 1))


def test_splitmix64_first_outputs():
    # SplitMix64 from state 0: the published first outputs of the generator
    got = datagen.raw_u64(0, 0, 3)
    assert [hex(int(v)) for v in got] == ["0xe220a8397b1dcdaf", "0x6e789e6aa1b965f4",
                                          "0x6c45d188009454f"]


def test_distributions():
    u = datagen.uniform(5, 0, 200000, -1, 1)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 0.01
    n = datagen.normal(5, 1, 200000)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1) < 0.01
    z = datagen.uniform_zeros(5, 2, 200000, -100, 100, 0.01)
    zeros = z == 0
    assert 0.008 < zeros.mean() < 0.012
    neg = np.signbit(z[zeros]).mean()
    assert 0.4 < neg < 0.6
    r = datagen.uniform_reject(5, 3, 200000, -7, 7, 0.01)
    assert (np.abs(r) >= 0.01).all() and r.min() >= -7 and r.max() < 7
    i = datagen.int_range(5, 4, 200000, -1000, 1000, skip_zero=True)
    assert (i != 0).all() and i.min() == -1000 and i.max() == 1000


def test_make_storage():
    assert datagen.make("normal", "bfloat16", (3, 4), 0, 0).dtype == np.uint16
    assert datagen.make("bits", "uint8", (7,), 0, 0).dtype == np.uint8
    assert datagen.make("bits", "int64", (7,), 0, 0).dtype == np.int64
    b = datagen.make("bool", "bool", (1000,), 0, 0)
    assert set(np.unique(b)) <= {0, 1}
