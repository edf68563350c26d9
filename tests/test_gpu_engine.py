"""GPU behaviour around the kernels: validation status, aliasing, alignment
fallback, streams, the host-buffer entry point and launch accounting."""
import numpy as np
import pytest

import datagen
import oracle
from conftest import assert_bits_equal
from engine_util import inputs_for, run_engine, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
eb = pytest.importorskip("broadcast_elementwise_gb300")


def test_division_by_zero_sets_status_and_clears():
    a = np.arange(1, 100001, dtype=np.int32)
    b = np.ones(100000, np.int32)
    b[777] = 0
    got, bits, _ = run_engine("Div", "int32", a, b)
    want, wbits = oracle.run("Div", a, b, "int32")
    assert bits == eb.DEVICE_DIV_BY_ZERO == wbits
    assert (got == want).all()
    # read-and-clear: the next read on the stream is clean
    assert eb.get_device_status() == 0
    got, bits, _ = run_engine("Mod", "int32", a, np.full(1, 7, np.int32).reshape(()),
                              attrs={"fmod": 0})
    assert bits == 0


def test_scalar_zero_divisor_and_negative_power():
    a = datagen.make("bits", "int64", (5000,), 1, 0)
    _, bits, fam = run_engine("Mod", "int64", a, np.zeros((), np.int64), attrs={"fmod": 1})
    assert fam == "right_scalar" and bits == eb.DEVICE_DIV_BY_ZERO
    base = np.array([0, 2, 3], np.int32)
    _, bits, _ = run_engine("Pow", "int32", base, np.array([-1], np.int32))
    assert bits == eb.DEVICE_DIV_BY_ZERO


@pytest.mark.parametrize("dtype", ["uint8", "uint32"])
def test_shift_range(dtype):
    w = 8 * np.dtype(datagen.STORAGE[dtype]).itemsize
    a = datagen.make("bits", dtype, (4096,), 2, 0)
    for direction in (0, 1):
        for s in range(w):
            b = np.array([s], datagen.STORAGE[dtype])
            got, bits, _ = run_engine("BitShift", dtype, a, b, attrs={"direction": direction})
            want, _ = oracle.run("BitShift", a, b, dtype, direction=direction)
            assert bits == 0 and (got == want).all(), (direction, s)
        _, bits, _ = run_engine("BitShift", dtype, a, np.array([w], datagen.STORAGE[dtype]),
                                attrs={"direction": direction})
        assert bits == eb.DEVICE_SHIFT_RANGE


def test_status_words_are_per_stream():
    a = torch.arange(1, 1025, dtype=torch.int32, device="cuda")
    z = torch.zeros(1024, dtype=torch.int32, device="cuda")
    o = torch.ones(1024, dtype=torch.int32, device="cuda")
    out = torch.empty_like(a)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    d = eb.descriptor("Div", "int32")
    p = eb.Plan(d, (1024,), (1024,))
    eb.execute(p, a, z, out, stream=s1)
    eb.execute(p, a, o, out, stream=s2)
    assert eb.get_device_status(s2) == 0
    assert eb.get_device_status(s1) == eb.DEVICE_DIV_BY_ZERO
    assert eb.get_device_status(s1) == 0


def test_in_place_execution():
    a, b = inputs_for("Add", "float32", (1000, 256), (256,), seed=3)
    want, _ = oracle.run("Add", a, b, "float32")
    dA, dB = to_device(a), to_device(b)
    p = eb.Plan(eb.descriptor("Add", "float32"), a.shape, b.shape)
    eb.execute(p, dA, dB, dA)                             # out == A: allowed
    torch.cuda.synchronize()
    assert_bits_equal(dA.cpu().numpy().view(np.float32).reshape(want.shape), want, "float32")


def test_misaligned_pointers_take_the_general_kernel():
    a, b = inputs_for("Mul", "float32", (100001,), (100001,), seed=4)
    want, _ = oracle.run("Mul", a, b, "float32")
    dA = to_device(np.concatenate([np.zeros(1, np.float32), a]))
    dB = to_device(np.concatenate([np.zeros(3, np.float32), b]))
    out = torch.zeros((100001 + 1) * 4, dtype=torch.uint8, device="cuda")
    p = eb.Plan(eb.descriptor("Mul", "float32"), a.shape, b.shape)
    eb.execute(p, dA.data_ptr() + 4, dB.data_ptr() + 12, out.data_ptr() + 4)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.float32)[1:]
    assert_bits_equal(got, want, "float32")


def test_execute_host_round_trip():
    a, b = inputs_for("Sub", "bfloat16", (64, 3000), (64, 1), seed=5)
    want, _ = oracle.run("Sub", a, b, "bfloat16")
    p = eb.Plan(eb.descriptor("Sub", "bfloat16"), a.shape, b.shape)
    ha = torch.from_numpy(a.reshape(-1).view(np.int16).copy()).pin_memory()
    hb = torch.from_numpy(b.reshape(-1).view(np.int16).copy()).pin_memory()
    ho = torch.empty(p.numel, dtype=torch.int16).pin_memory()
    da = torch.empty_like(ha, device="cuda")
    db = torch.empty_like(hb, device="cuda")
    do = torch.empty_like(ho, device="cuda")
    s = torch.cuda.current_stream()
    eb.ebin_execute_host(p.handle, ha.data_ptr(), hb.data_ptr(), ho.data_ptr(), da.data_ptr(),
                         db.data_ptr(), do.data_ptr(), s.cuda_stream)
    s.synchronize()
    assert_bits_equal(ho.numpy().view(np.uint16).reshape(want.shape), want, "bfloat16")


def _host_run(op, dtype, a, b, attrs=None, stream=None):
    """ebin_execute_host with pinned host buffers; returns (out, family, launches)."""
    desc = eb.descriptor(op, dtype, **(attrs or {}))
    p = eb.Plan(desc, a.shape, b.shape)
    view = {1: np.uint8, 2: np.int16, 4: np.int32, 8: np.int64}
    isz, isz_b = eb.ITEMSIZE[dtype], eb.ITEMSIZE[desc.dtype_b]
    osz = eb.ITEMSIZE[desc.out_dtype]
    ha = torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(view[isz]).copy()).pin_memory()
    hb = torch.from_numpy(np.ascontiguousarray(b).reshape(-1).view(view[isz_b]).copy()).pin_memory()
    ho = torch.empty(p.numel * osz, dtype=torch.uint8).pin_memory()
    da, db = torch.empty_like(ha, device="cuda"), torch.empty_like(hb, device="cuda")
    do = torch.empty(p.numel * osz, dtype=torch.uint8, device="cuda")
    s = stream or torch.cuda.current_stream()
    before = eb.ebin_launch_count()
    eb.ebin_execute_host(p.handle, ha.data_ptr(), hb.data_ptr(), ho.data_ptr(), da.data_ptr(),
                         db.data_ptr(), do.data_ptr(), s.cuda_stream)
    s.synchronize()
    return ho.numpy(), p.family, eb.ebin_launch_count() - before


@pytest.mark.parametrize("op,dtype,sa,sb,fam,chunks", [
    ("Mul", "float32", (5000003,), (5000003,), "contiguous", 5),
    ("Add", "bfloat16", (3000001,), (), "right_scalar", 3),
    ("Sub", "int32", (1,), (2500000,), "left_scalar", 3),
    ("Greater", "float16", (2621447,), (2621447,), "contiguous", 3),
    ("Div", "float32", (1 << 21,), (1 << 21,), "contiguous", 2),
    # parameter blocks whose rows move with the output: copied whole, and each
    # chunk's kernel starts that chunk's offset into every row
    ("BatchNormalization", "float32", (1, 2097155), (4, 2097155), "contiguous", 3),
    ("BiasPRelu", "float16", (1, 2097155), (2, 2097155), "contiguous", 3),
    ("BiasPReluBN", "bfloat16", (1, 2097155, 1, 1), (6, 2097155), "contiguous", 3),
    ("Clip", "float32", (2097155,), (2,), "right_scalar", 3),
    # a prepared scalar: whole-pack chunks on the per-row kernel as one row,
    # the short last chunk on the scalar kernel
    ("Mod", "float32", (3000001,), (), "right_scalar", 3),
    ("PRelu", "float32", (2097155,), (2097155,), "contiguous", 3),
])
def test_execute_host_pipelined(op, dtype, sa, sb, fam, chunks):
    """Large contiguous and scalar plans run as a pipeline of chunks over two
    copy streams; ragged lengths end in a short chunk."""
    a, b = inputs_for(op, dtype, sa, sb, seed=81)
    want, _ = oracle.run(op, a, b, dtype)
    got, family, launches = _host_run(op, dtype, a, b)
    assert family == fam and launches == chunks
    otype = "bool" if op == "Greater" else dtype
    ov = {"float32": np.float32, "float16": np.float16, "bfloat16": np.uint16, "int32": np.int32,
          "bool": np.uint8}[otype]
    assert_bits_equal(got.view(ov).reshape(want.shape), want, otype, op)


@pytest.mark.parametrize("op,dtype,sa,sb", [
    ("BatchNormalization", "float16", (1, 2097155), (4, 2097155)),
    ("BiasPReluBN", "bfloat16", (1, 2097155, 1, 1), (6, 2097155)),
    ("BiasPRelu", "float64", (1, 2097155), (2, 2097155)),
])
def test_execute_host_pipelined_float32_block(op, dtype, sa, sb):
    """A float32 parameter block that moves with a 16-bit or float64 output:
    copied whole with its own element size, and each chunk's kernel starts that
    chunk's offset, in float32 elements, into every row."""
    a, _ = inputs_for(op, dtype, sa, sb, seed=83)
    _, b = inputs_for(op, "float32", sa, sb, seed=83)
    want = oracle.run_params(op, a, b, dtype, "float32")
    got, family, launches = _host_run(op, dtype, a, b, attrs={"dtype_b": "float32"})
    assert family == "contiguous" and launches == 3
    ov = {"float16": np.float16, "bfloat16": np.uint16, "float64": np.float64}[dtype]
    assert_bits_equal(got.view(ov).reshape(want.shape), want, dtype, op)


def test_binary_helper_with_float32_block():
    """binary() takes a float32 parameter block beside bfloat16 x on the device
    and on pinned host memory (the block's type read from the tensor)."""
    sa, sb = (2, 64, 30, 40), (6, 64)
    a, _ = inputs_for("BiasPReluBN", "bfloat16", sa, sb, seed=84)
    _, b = inputs_for("BiasPReluBN", "float32", sa, sb, seed=84)
    want = oracle.run_params("BiasPReluBN", a, b, "bfloat16", "float32")
    x = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    w = torch.from_numpy(b.copy())
    y = eb.binary("BiasPReluBN", x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16 and tuple(y.shape) == sa
    assert_bits_equal(y.cpu().view(torch.int16).numpy().view(np.uint16), want, "bfloat16",
                      "device")
    yh = eb.binary("BiasPReluBN", x.pin_memory(), w.pin_memory())
    torch.cuda.synchronize()
    assert_bits_equal(yh.view(torch.int16).numpy().view(np.uint16), want, "bfloat16", "mapped")


def test_execute_host_pipelined_status_and_ordering():
    """The device status word is raised through the chunked path, and two
    calls queued back to back on one stream reuse the device buffers in order."""
    n = 3 << 20
    a = datagen.make("bits", "int32", (n,), 82, 0)
    got, fam, launches = _host_run("Mod", "int32", a, np.zeros((), np.int32), {"fmod": 0})
    assert fam == "right_scalar" and launches == 3
    assert eb.get_device_status() == eb.DEVICE_DIV_BY_ZERO
    assert eb.get_device_status() == 0
    # two pipelined calls on the same buffers without a synchronisation between them
    x1, y1 = inputs_for("Add", "float32", (n,), (n,), seed=83)
    x2, y2 = inputs_for("Mul", "float32", (n,), (n,), seed=84)
    p1 = eb.Plan(eb.descriptor("Add", "float32"), (n,), (n,))
    p2 = eb.Plan(eb.descriptor("Mul", "float32"), (n,), (n,))
    pin = lambda v: torch.from_numpy(v.copy()).pin_memory()
    h = [pin(x1), pin(y1), pin(x2), pin(y2)]
    o1, o2 = torch.empty(n).pin_memory(), torch.empty(n).pin_memory()
    da, db, do = (torch.empty(n, device="cuda") for _ in range(3))
    s = torch.cuda.current_stream()
    for p, ha, hb, ho in ((p1, h[0], h[1], o1), (p2, h[2], h[3], o2)):
        eb.ebin_execute_host(p.handle, ha.data_ptr(), hb.data_ptr(), ho.data_ptr(),
                             da.data_ptr(), db.data_ptr(), do.data_ptr(), s.cuda_stream)
    s.synchronize()
    assert_bits_equal(o1.numpy(), oracle.run("Add", x1, y1, "float32")[0], "float32")
    assert_bits_equal(o2.numpy(), oracle.run("Mul", x2, y2, "float32")[0], "float32")


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16", "float64"])
def test_with_scalar_matches_a_scalar_tensor(dtype):
    """ncnn binaryop with_scalar: B is the attribute value rounded to the element
    type, so the result equals the oracle's with a 0-d B holding that value.
    Runs the right-scalar kernel, the general kernel (unaligned A), a single
    element, and the host-buffer pipeline."""
    from test_gpu_parity import compare
    for op in ("Add", "Sub", "Mul", "Div", "Pow", "Max", "Min", "RSub", "RDiv"):
        for v in (0.37, -2.5, 0.0, -0.0, float("inf"), float("nan"), 1e-8, 70000.0):
            a, _ = inputs_for(op, dtype, (100003,), (), seed=90)
            bq = datagen.float_to(np.array([v], np.float32), dtype).reshape(())
            want, _ = oracle.run(op, a, bq, dtype)
            desc = eb.descriptor(op, dtype, scalar_b=v)
            for shape, offset in (((100003,), 0), ((100003,), 1), ((), 0)):
                aa = a if shape else a[:1].reshape(())
                ww = want if shape else want[:1].reshape(())
                plan = eb.Plan(desc, aa.shape, ())
                isz = eb.ITEMSIZE[dtype]
                buf = to_device(np.concatenate([np.zeros(offset, aa.dtype), aa.reshape(-1)]))
                out = torch.empty(max(plan.numel, 1) * isz + 16, dtype=torch.uint8,
                                  device="cuda")
                eb.execute(plan, buf.data_ptr() + offset * isz, None, out.data_ptr() + offset * isz)
                got = out.cpu().numpy()[offset * isz: (offset + plan.numel) * isz] \
                    .view(datagen.STORAGE[dtype]).reshape(ww.shape)
                compare(op, dtype, got, ww, "%s %s b=%r shape=%s offset=%d" %
                        (op, dtype, v, shape, offset))
    # through the host-buffer pipeline (2^21 elements: chunked)
    n = 1 << 21
    a = datagen.make("normal", dtype, (n,), 91, 0)
    bq = datagen.float_to(np.array([0.75], np.float32), dtype).reshape(())
    want, _ = oracle.run("RDiv", a, bq, dtype)
    p = eb.Plan(eb.descriptor("RDiv", dtype, scalar_b=0.75), (n,), ())
    view = {2: np.int16, 4: np.int32, 8: np.int64}[eb.ITEMSIZE[dtype]]
    ha = torch.from_numpy(a.reshape(-1).view(view).copy()).pin_memory()
    ho = torch.empty_like(ha).pin_memory()
    da, do = torch.empty_like(ha, device="cuda"), torch.empty_like(ha, device="cuda")
    s = torch.cuda.current_stream()
    eb.ebin_execute_host(p.handle, ha.data_ptr(), None, ho.data_ptr(), da.data_ptr(), None,
                         do.data_ptr(), s.cuda_stream)
    s.synchronize()
    assert_bits_equal(ho.numpy().view(datagen.STORAGE[dtype]), want, dtype, "RDiv host")


def test_int_rdiv_validates_a():
    a = np.array([3, 0, -1, 7] * 1000, np.int32)
    b = np.array([10, 5, -2147483648, -21] * 1000, np.int32)
    got, bits, _ = run_engine("RDiv", "int32", a, b)
    want, wbits = oracle.run("RDiv", a, b, "int32")
    assert bits == wbits == eb.DEVICE_DIV_BY_ZERO
    assert (got == want).all()


def test_binary_helper_reads_strided_tensors_in_place():
    """Non-contiguous torch tensors (a transpose, a step slice) go to the engine
    as strided views, without a copy."""
    x = torch.randn(64, 48, device="cuda").t()             # (48, 64), strides (1, 48)
    y = torch.randn(200, 64, device="cuda")[::4]           # (50, 64) ... broadcast below
    before = eb.ebin_launch_count()
    z = eb.binary("Mul", x, y[:48])
    torch.cuda.synchronize()
    assert eb.ebin_launch_count() == before + 1            # one kernel, no copy kernels
    want, _ = oracle.run("Mul", x.contiguous().cpu().numpy(), y[:48].contiguous().cpu().numpy(),
                         "float32")
    assert_bits_equal(z.cpu().numpy(), want, "float32")


def test_launch_count_and_binary_helper():
    x = torch.randn(4, 8, 32, 32, device="cuda")
    bias = torch.randn(8, 1, 1, device="cuda")
    before = eb.ebin_launch_count()
    y = eb.binary("Add", x, bias)
    torch.cuda.synchronize()
    assert eb.ebin_launch_count() == before + 1
    want, _ = oracle.run("Add", x.cpu().numpy(), bias.cpu().numpy(), "float32")
    assert_bits_equal(y.cpu().numpy(), want, "float32")
    e = eb.binary("Add", torch.empty(0, 5, device="cuda"), torch.empty(5, device="cuda"))
    assert e.shape == (0, 5) and eb.ebin_launch_count() == before + 1


def test_binary_helper_checks_operands_before_launching():
    """binary() refuses, before any launch, an out the kernel would write out of
    bounds or misread (wrong shape, type, layout or device) and a B of another
    type or device; a correct out is written in place."""
    x = torch.randn(4, 8, 32, device="cuda")
    y = torch.randn(8, 1, device="cuda")
    before = eb.ebin_launch_count()
    bad_outs = [torch.empty(4, 8, 31, device="cuda"),                    # too small
                torch.empty(4, 8, 32, dtype=torch.float16, device="cuda"),
                torch.empty(4, 32, 8, device="cuda").transpose(1, 2),    # not contiguous
                torch.empty(4, 8, 32)]                                  # host memory
    for out in bad_outs:
        with pytest.raises(ValueError, match="out"):
            eb.binary("Add", x, y, out)
    with pytest.raises(ValueError, match="takes B of float32"):
        eb.binary("Add", x, y.half())
    with pytest.raises(ValueError, match="B on cpu"):
        eb.binary("Add", x, y.cpu())
    bool_out = torch.empty(4, 8, 32, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError, match="result is bool"):
        eb.binary("Greater", x, y, bool_out)
    assert eb.ebin_launch_count() == before
    out = torch.full((4, 8, 32), float("nan"), device="cuda")
    assert eb.binary("Add", x, y, out) is out
    torch.cuda.synchronize()
    want, _ = oracle.run("Add", x.cpu().numpy(), y.cpu().numpy(), "float32")
    assert_bits_equal(out.cpu().numpy(), want, "float32")


def test_plan_outlives_cache_eviction_on_device():
    eb.ebin_plan_cache_clear()
    d = eb.descriptor("Mul", "float32")
    keep = eb.Plan(d, (64, 64), (64,))
    for i in range(12):
        eb.Plan(d, (i + 1, 64), (64,))                     # evicts `keep` from the cache
    a, b = inputs_for("Mul", "float32", (64, 64), (64,), seed=6)
    want, _ = oracle.run("Mul", a, b, "float32")
    dA, dB = to_device(a), to_device(b)
    out = torch.empty(64 * 64 * 4, dtype=torch.uint8, device="cuda")
    eb.execute(keep, dA, dB, out)
    torch.cuda.synchronize()
    assert_bits_equal(out.cpu().numpy().view(np.float32).reshape(64, 64), want, "float32")


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_mod_with_shared_divisor_is_exact(dtype):
    """Scalar and per-row divisors take the prepared-reciprocal path: stress it
    with dividends at, next to and between multiples of the divisor, raw bit
    patterns, and divisors across the exponent range."""
    divisors = [1.0, 3.0, -2.5, 0.1, 7.0e-3, -1.0e-30, 6.5e20, 1.5e-38, 1e-44, 0.0, -0.0,
                np.inf, np.nan, 65504.0, 3.3333333, -1234.5678]
    rng = np.random.default_rng(99)
    for i, d in enumerate(divisors):
        bq = datagen.float_to(np.array([d], np.float32), dtype)
        dv = float(bq.astype(np.float32)[0]) if dtype != "bfloat16" else \
            float((bq.astype(np.uint32) << 16).view(np.float32)[0])
        k = rng.integers(-5000000, 5000000, 4096).astype(np.float64)
        cand = np.concatenate([k * dv, k * dv + dv * 0.5, np.nextafter(k * dv, np.inf),
                               (rng.random(4096) - 0.5) * 2e6]).astype(np.float32)
        with np.errstate(all="ignore"):
            a = np.concatenate([datagen.float_to(np.nan_to_num(cand, nan=1.0), dtype),
                                datagen.make("bits", dtype, (8192,), 70, i)]).reshape(-1)
        a = a[: (a.size // 64) * 64]
        for fmod in (0, 1):
            got, bits, fam = run_engine("Mod", dtype, a, bq.reshape(()), attrs={"fmod": fmod})
            want, _ = oracle.run("Mod", a, bq.reshape(()), dtype, fmod=fmod)
            assert fam == "right_scalar"
            assert_bits_equal(got, want, dtype, "Mod scalar %r fmod=%d" % (d, fmod))
            rows = a.reshape(64, -1)
            bcol = np.repeat(bq, 64).reshape(64, 1)
            got, _, fam = run_engine("Mod", dtype, rows, bcol, attrs={"fmod": fmod})
            want, _ = oracle.run("Mod", rows, bcol, dtype, fmod=fmod)
            assert_bits_equal(got, want, dtype, "Mod rows %r fmod=%d" % (d, fmod))


def test_int32_mod_with_shared_divisor_is_exact():
    """int32 scalar and per-row divisors take the prepared multiply-high path:
    stress it with divisors across the range (1, -1, powers of two and their
    neighbours, 2^31 - 1, INT_MIN) and dividends at the extremes, at multiples
    of the divisor and one either side, and raw bit patterns."""
    i32 = np.iinfo(np.int32)
    divisors = [1, -1, 2, -2, 3, 7, -7, 10, 1000, -999, 65535, 65536, 65537, (1 << 24) + 1,
                (1 << 30) - 1, 1 << 30, i32.max, -i32.max, i32.min, 123456789, -987654321]
    rng = np.random.default_rng(123)
    for i, d in enumerate(divisors):
        k = rng.integers(-(2 ** 31) // max(abs(d), 1), 2 ** 31 // max(abs(d), 1), 2048,
                         dtype=np.int64)
        cand = np.concatenate([k * d, k * d + 1, k * d - 1,
                               [i32.min, i32.max, i32.min + 1, 0, 1, -1, d, -d if d != i32.min
                                else 0]])
        cand = cand[(cand >= i32.min) & (cand <= i32.max)].astype(np.int32)
        a = np.concatenate([cand, datagen.make("bits", "int32", (4096,), 71, i)])
        a = a[: (a.size // 256) * 256]             # rows of a multiple of 4 elements
        bq = np.array([d], np.int32)
        for fmod in (0, 1):
            got, bits, fam = run_engine("Mod", "int32", a, bq.reshape(()), attrs={"fmod": fmod})
            want, wbits = oracle.run("Mod", a, bq.reshape(()), "int32", fmod=fmod)
            assert fam == "right_scalar" and bits == wbits == 0
            assert_bits_equal(got, want, "int32", "Mod int32 scalar %d fmod=%d" % (d, fmod))
            rows = a.reshape(64, -1)
            bcol = np.repeat(bq, 64).reshape(64, 1)
            got, _, fam = run_engine("Mod", "int32", rows, bcol, attrs={"fmod": fmod})
            want, _ = oracle.run("Mod", rows, bcol, "int32", fmod=fmod)
            assert fam == "repeated_block"
            assert_bits_equal(got, want, "int32", "Mod int32 rows %d fmod=%d" % (d, fmod))
    # a zero divisor among per-row divisors: that row reads 0 and the status is set
    rows = datagen.make("bits", "int32", (8, 512), 72, 0)
    bcol = np.array([3, -5, 0, 7, 1, -1, 100, 9], np.int32).reshape(8, 1)
    got, bits, _ = run_engine("Mod", "int32", rows, bcol, attrs={"fmod": 0})
    want, wbits = oracle.run("Mod", rows, bcol, "int32", fmod=0)
    assert bits == wbits == eb.DEVICE_DIV_BY_ZERO
    assert_bits_equal(got, want, "int32", "Mod int32 rows with a zero divisor")


def test_chained_launches_see_previous_results():
    """Back-to-back kernels overlap their launch with the previous kernel's
    tail; each must still read the finished output of the one before."""
    x = datagen.make("normal", "float32", (64, 4096), 5, 0)
    bias = datagen.make("uniform", "float32", (4096,), 5, 1, lo=-0.5, hi=0.5)
    scale = datagen.make("uniform", "float32", (64, 1), 5, 2, lo=0.5, hi=1.5)
    want = x
    for k in range(6):
        want, _ = oracle.run("Add" if k % 2 == 0 else "Mul", want, bias if k % 2 == 0 else scale,
                             "float32")
    cur = to_device(x)
    bufs = [torch.empty_like(cur) for _ in range(2)]
    dB, dS = to_device(bias), to_device(scale)
    p_add = eb.Plan(eb.descriptor("Add", "float32"), x.shape, bias.shape)
    p_mul = eb.Plan(eb.descriptor("Mul", "float32"), x.shape, scale.shape)
    for k in range(6):
        out = bufs[k % 2]
        eb.execute(p_add if k % 2 == 0 else p_mul, cur, dB if k % 2 == 0 else dS, out)
        cur = out
    torch.cuda.synchronize()
    assert_bits_equal(cur.cpu().numpy().view(np.float32).reshape(want.shape), want, "float32",
                      "six chained launches")


@pytest.mark.parametrize("dtype", ["float32", "float16", "bfloat16"])
def test_batchnorm_division_is_exact(dtype):
    """BatchNormalization divides by one prepared value per channel: stress the
    proof-checked fast division and its fallback with channel divisors across
    the exponent range (and 0, NaN, infinity) and raw-bit-pattern inputs."""
    var = np.array([1.0, 3.0, 0.0, -1.0, 1e-30, 1e30, 2.0 ** -80, 2.0 ** 90, 0.75, 1e-6,
                    np.inf, np.nan, 5.0, 0.2, 123456.0, 7e-3], np.float32)
    C = var.size
    eps = 0.0 if dtype == "float32" else 1e-5
    mean = np.array([0.0, 1.0, -2.0, 0.5, 0.0, 3.0, -0.0, 1e20, 0.25, -1e-3, 0.0, 1.0, 7.0,
                     -3.0, 0.0, 0.5], np.float32)
    scale = np.array([1.0, 2.0, -1.0, 0.5, 1.0, 1e-3, 3.0, 1.0, -2.0, 1.0, 1.0, 1.0, 0.1,
                      1.0, 1e10, 1.0], np.float32)
    bias = np.array([-0.0, 0.5, 0.0, 1.0, -0.0, 2.0, -1.0, 0.0, 0.0, 4.0, 0.0, 0.0, -0.5,
                     0.0, 1.0, -0.0], np.float32)
    params = datagen.float_to(np.stack([scale, bias, mean, var]), dtype)
    x = np.concatenate([datagen.make("bits", dtype, (2, C, 512), 80, 0).reshape(-1),
                        datagen.make("normal", dtype, (2, C, 512), 80, 1).reshape(-1)])
    x = x.reshape(4, C, 512)
    got, _, fam = run_engine("BatchNormalization", dtype, x, params, attrs={"epsilon": eps})
    want, _ = oracle.run("BatchNormalization", x, params, dtype, eps=eps)
    assert fam == "inner_vector_outer"
    assert_bits_equal(got, want, dtype, "BN per-channel rows")
    x2 = x.reshape(4 * 512, C)   # rank 2: one parameter set per element
    got, _, _ = run_engine("BatchNormalization", dtype, x2, params, attrs={"epsilon": eps})
    want, _ = oracle.run("BatchNormalization", x2, params, dtype, eps=eps)
    assert_bits_equal(got, want, dtype, "BN rank-2")


def _pinned(arr: np.ndarray, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(arr).reshape(-1).view(np.uint8).copy())
    return t.pin_memory() if pin else t


@pytest.mark.parametrize("op,dtype,sa,sb,fam", [
    ("Mul", "float32", (3000017,), (3000017,), "contiguous"),
    ("Add", "bfloat16", (1000003,), (), "right_scalar"),
    ("PRelu", "bfloat16", (4, 64, 64, 64), (64, 1, 1), "inner_vector_outer"),
    ("Greater", "float16", (16, 1, 512, 1), (1, 8, 1, 1024), "inner_vector_outer"),
    ("Add", "float32", (2, 3, 4, 5), (3, 1, 5), "general_strided"),
    ("Mod", "int32", (4096, 640), (4096, 1), "repeated_block"),
])
def test_execute_mapped_matches_the_oracle(op, dtype, sa, sb, fam):
    """ebin_execute_mapped: the kernel reads and writes pinned host buffers in
    place, with the results of ebin_execute."""
    a, b = inputs_for(op, dtype, sa, sb, seed=91)
    want, wbits = oracle.run(op, a, b, dtype)
    p = eb.Plan(eb.descriptor(op, dtype), sa, sb)
    assert p.family == fam
    osz = eb.ITEMSIZE[eb.descriptor(op, dtype).out_dtype]
    ha, hb = _pinned(a), _pinned(b)
    ho = torch.full((p.numel * osz,), 0xAB, dtype=torch.uint8).pin_memory()
    s = torch.cuda.current_stream()
    before = eb.ebin_launch_count()
    eb.execute_mapped(p, ha, hb, ho, s)
    s.synchronize()
    assert eb.ebin_launch_count() - before == 1
    otype = "bool" if op == "Greater" else dtype
    got = ho.numpy().view(datagen.STORAGE[otype]).reshape(want.shape)
    assert_bits_equal(got, want, otype, op)
    assert eb.get_device_status() == wbits


def test_execute_mapped_refuses_unmapped_buffers():
    """Pageable memory, or a pinned buffer shorter than the plan, is refused
    with INVALID_ARG before any device work; the output is left alone."""
    n = 1 << 20
    a, b = inputs_for("Add", "float32", (n,), (n,), seed=92)
    p = eb.Plan(eb.descriptor("Add", "float32"), (n,), (n,))
    ha, hb = _pinned(a), _pinned(b)
    ho = torch.full((4 * n,), 0x5A, dtype=torch.uint8).pin_memory()
    pageable = _pinned(a, pin=False)
    short = torch.zeros(4 * n // 2, dtype=torch.uint8).pin_memory()
    before = eb.ebin_launch_count()
    out_pageable = _pinned(np.zeros(4 * n, np.uint8), pin=False)
    for args in ((pageable, hb, ho), (ha, pageable, ho), (ha, hb, out_pageable),
                 (short, hb, ho), (ha, hb, short)):
        with pytest.raises(eb.EbinError, match="invalid_arg"):
            eb.execute_mapped(p, *args)
    torch.cuda.synchronize()
    assert eb.ebin_launch_count() == before
    assert bool((ho == 0x5A).all()) and bool((short == 0).all())


def test_cuda_graph_capture_and_replay():
    """The launch path of a non-validating operator makes no allocation and no
    synchronising call, so plans can be captured in a CUDA graph: a captured
    per-channel BatchNormalization followed by a scalar Mul replays on fresh
    inputs with the oracle's results."""
    sa, C = (4, 16, 64, 64), 16
    bn = eb.descriptor("BatchNormalization", "bfloat16", epsilon=1e-5)
    mul = eb.descriptor("Mul", "bfloat16")
    plan_bn = eb.Plan(bn, sa, (4, C))
    plan_mul = eb.Plan(mul, sa, (1,))
    x0, params = inputs_for("BatchNormalization", "bfloat16", sa, (4, C), seed=93)
    s_val = datagen.float_to(np.array([0.75], np.float32), "bfloat16")
    n = int(np.prod(sa))
    dx, dp, ds = to_device(x0), to_device(params), to_device(s_val)
    dmid = torch.empty(2 * n, dtype=torch.uint8, device="cuda")
    dout = torch.empty(2 * n, dtype=torch.uint8, device="cuda")
    eb.execute(plan_bn, dx, dp, dmid)          # first launches load the kernels
    eb.execute(plan_mul, dmid, ds, dout)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    before = eb.ebin_launch_count()
    with torch.cuda.graph(g):
        eb.execute(plan_bn, dx, dp, dmid)
        eb.execute(plan_mul, dmid, ds, dout)
    assert eb.ebin_launch_count() - before == 2
    for seed in (94, 95, 96):
        x = datagen.make("normal", "bfloat16", sa, seed, 0)
        dx.copy_(to_device(x))
        g.replay()
        torch.cuda.synchronize()
        mid, _ = oracle.run("BatchNormalization", x, params, "bfloat16", eps=1e-5)
        want, _ = oracle.run("Mul", mid, s_val, "bfloat16", shape_b=(1,))
        got = dout.cpu().numpy().view(np.uint16).reshape(sa)
        assert_bits_equal(got, want, "bfloat16", "graph replay %d" % seed)


def test_binary_helper_on_pinned_host_tensors():
    """binary() on pinned CPU tensors runs the kernel on host memory in place."""
    a, b = inputs_for("Mul", "float32", (64, 1000), (1000,), seed=97)
    want, _ = oracle.run("Mul", a, b, "float32")
    ta, tb = torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory()
    out = eb.binary("Mul", ta, tb)
    torch.cuda.synchronize()
    assert out.is_pinned() and not out.is_cuda
    assert_bits_equal(out.numpy(), want, "float32", "binary on pinned host tensors")
    with pytest.raises(ValueError, match="pinned"):
        eb.binary("Mul", torch.from_numpy(a), tb)
    with pytest.raises(ValueError, match="pinned CPU tensor"):
        eb.binary("Mul", ta, tb, torch.empty(out.shape, device="cuda"))
    with pytest.raises(ValueError, match="pinned CPU tensor"):
        eb.binary("Mul", ta, tb, torch.empty(out.shape))


@pytest.mark.parametrize("sb", [(1,), (1, 16, 1, 1), (4, 16, 8, 33)])
def test_execute3_mapped_matches_the_oracle(sb):
    """ebin_execute3_mapped: MulAdd with all four buffers in pinned host memory."""
    sa = (4, 16, 8, 33)
    x = datagen.make("normal", "bfloat16", sa, 98, 0)
    s = datagen.make("uniform", "bfloat16", sb, 98, 1, lo=0.0, hi=0.3)
    y = datagen.make("normal", "bfloat16", sa, 98, 2)
    want = oracle.run3("MulAdd", x, s, y, "bfloat16")
    p = eb.Plan3(eb.descriptor("MulAdd", "bfloat16"), sa, sb, sa)
    out = torch.zeros(2 * p.numel, dtype=torch.uint8).pin_memory()
    eb.execute3_mapped(p, _pinned(x), _pinned(s), _pinned(y), out)
    torch.cuda.synchronize()
    assert_bits_equal(out.numpy().view(np.uint16).reshape(sa), want, "bfloat16", "MulAdd mapped")


def test_execute_mapped_on_registered_host_memory():
    """Memory pinned after the fact with cudaHostRegister is accepted too."""
    n = (1 << 20) + 3
    a, b = inputs_for("Add", "float32", (n,), (n,), seed=99)
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    o = np.zeros(n, np.float32)
    cr = torch.cuda.cudart()
    for arr in (a, b, o):
        assert cr.cudaHostRegister(arr.ctypes.data, arr.nbytes, 0) == cr.cudaError.success
    try:
        p = eb.Plan(eb.descriptor("Add", "float32"), (n,), (n,))
        eb.execute_mapped(p, a.ctypes.data, b.ctypes.data, o.ctypes.data)
        torch.cuda.synchronize()
        want, _ = oracle.run("Add", a, b, "float32")
        assert_bits_equal(o, want, "float32", "registered host memory")
    finally:
        for arr in (a, b, o):
            cr.cudaHostUnregister(arr.ctypes.data)


def test_host_threads_on_their_own_streams():
    """Four host threads, each on its own stream, run int32 Div plans at once;
    only the threads whose divisors hold a zero see DIV_BY_ZERO on their
    stream, and every output equals the oracle's."""
    import threading
    shape = (256, 1024)
    results, errors = {}, []

    def work(tid):
        try:
            stream = torch.cuda.Stream()
            a, b = inputs_for("Div", "int32", shape, shape, seed=100 + tid)
            b = b.copy()
            b[b == 0] = 1
            if tid % 2:
                b[tid, 7] = 0
            p = eb.Plan(eb.descriptor("Div", "int32"), shape, shape)
            dA, dB = to_device(a), to_device(b)
            out = torch.empty(4 * p.numel, dtype=torch.uint8, device="cuda")
            with torch.cuda.stream(stream):
                for _ in range(20):
                    eb.execute(p, dA, dB, out, stream)
            bits = eb.get_device_status(stream)
            results[tid] = (a, b, out.cpu().numpy().view(np.int32).reshape(shape), bits)
        except Exception as e:          # reported below, in the main thread
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=work, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for tid, (a, b, got, bits) in results.items():
        want, wbits = oracle.run("Div", a, b, "int32")
        assert_bits_equal(got, want, "int32", "thread %d" % tid)
        assert bits == wbits == (eb.DEVICE_DIV_BY_ZERO if tid % 2 else 0), (tid, bits, wbits)
