"""ebin_execute_noalloc: the same results as ebin_execute and as the oracle,
without the library allocating device memory.

Some callers cannot let a library call cudaMalloc: applications whose device
memory belongs entirely to their own arena allocator, plugins whose host
framework forbids allocation while work is being enqueued, and latency-critical
loops that cannot take cudaMalloc's implicit synchronisation.  For them this
entry point keeps the validating kernels' status words in a fixed array
compiled into the library, and ebin_noalloc_read_status reads one back.

This file is collected last so that, if it fails, a run stopping at the first
failure has already run every other test; it passes alone in a fresh process
as well as after the rest of the suite.
"""
import numpy as np
import pytest

import oracle
from conftest import assert_bits_equal
from engine_util import inputs_for, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
eb = pytest.importorskip("broadcast_elementwise_gb300")

ISZ = {"float32": 4, "bfloat16": 2, "int32": 4, "uint32": 4}


def _shifted(arr, offset):
    """Device copy of arr starting `offset` bytes into its buffer (off 16-byte
    alignment for offset % 16 != 0); returns (buffer, address)."""
    raw = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
    buf = to_device(np.concatenate([np.zeros(offset, np.uint8), raw, np.zeros(16, np.uint8)]))
    return buf, buf.data_ptr() + offset


CASES = [
    # op, dtype, dtype_b, shape_a, shape_b, attrs, byte offset of every buffer
    ("Div", "int32", None, (512, 1024), (512, 1), {}, 0),            # status word used
    ("Mod", "int32", None, (300007,), (), {"fmod": 0}, 0),           # right scalar, prepared
    ("BitShift", "uint32", None, (4096, 256), (256,), {"direction": 1}, 0),
    ("Mul", "float32", None, (300007,), (300007,), {}, 0),           # no status word at all
    ("BatchNormalization", "bfloat16", "float32", (4, 16, 8, 32), (4, 16),
     {"epsilon": 1e-5}, 0),                                          # float32 parameter block
    ("Div", "int32", None, (300, 256), (256,), {}, 4),                # unaligned: general kernel
    ("Add", "float32", None, (3, 17, 64), (17, 1), {}, 8),
]


@pytest.mark.parametrize("op,dtype,dtype_b,sa,sb,attrs,offset", CASES)
def test_noalloc_matches_oracle_and_execute_on_two_calls(op, dtype, dtype_b, sa, sb, attrs,
                                                          offset):
    a, b = inputs_for(op, dtype, sa, sb, seed=11)
    if dtype_b is not None:
        _, b = inputs_for(op, dtype_b, sa, sb, seed=11)
        want = oracle.run_params(op, a, b, dtype, dtype_b, eps=attrs.get("epsilon", 1e-5))
        want_bits = 0
    else:
        kw = {k: v for k, v in attrs.items() if k in ("fmod", "direction")}
        want, want_bits = oracle.run(op, a, b, dtype, **kw)
    desc = eb.descriptor(op, dtype, dtype_b=dtype_b, **attrs)
    plan = eb.Plan(desc, sa, sb)
    (bufA, pA), (bufB, pB) = _shifted(a, offset), _shifted(b, offset)
    isz = ISZ[desc.out_dtype]
    nbytes = plan.numel * isz
    stream = torch.cuda.current_stream().cuda_stream

    # the allocating entry point on the same buffers
    out_ref = torch.full((nbytes + offset + 16,), 0x5A, dtype=torch.uint8, device="cuda")
    eb.ebin_execute(plan.handle, pA, pB, out_ref.data_ptr() + offset, stream)
    ref_bits = eb.get_device_status()
    ref = out_ref.cpu().numpy()[offset:offset + nbytes]

    for call in range(2):
        out = torch.full((nbytes + offset + 16,), 0x5A, dtype=torch.uint8, device="cuda")
        bits = eb.ebin_execute_noalloc(plan.handle, pA, pB, out.data_ptr() + offset, stream, 3)
        torch.cuda.synchronize()
        got = out.cpu().numpy()[offset:offset + nbytes]
        what = "%s %s %s x %s offset %d call %d" % (op, dtype, sa, sb, offset, call)
        g = got.view(want.dtype).reshape(want.shape)
        assert_bits_equal(g, want, dtype, what + " vs the oracle")
        assert_bits_equal(g, ref.view(want.dtype).reshape(want.shape), dtype,
                          what + " vs ebin_execute")
        assert bits == want_bits == ref_bits, (what, bits, want_bits, ref_bits)
        # the bytes around the output are untouched
        assert (out.cpu().numpy()[:offset] == 0x5A).all()
        assert (out.cpu().numpy()[offset + nbytes:] == 0x5A).all()


def test_noalloc_reports_and_clears_status():
    a = np.arange(1, 65537, dtype=np.int32)
    b = np.ones(65536, np.int32)
    b[1234] = 0
    plan = eb.Plan(eb.descriptor("Div", "int32"), a.shape, b.shape)
    dA, dB = to_device(a), to_device(b)
    out = torch.empty(a.size * 4, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert eb.ebin_execute_noalloc(plan.handle, dA.data_ptr(), dB.data_ptr(), out.data_ptr(),
                                   s, 0) == eb.DEVICE_DIV_BY_ZERO
    want, bits = oracle.run("Div", a, b, "int32")
    assert bits == eb.DEVICE_DIV_BY_ZERO
    assert_bits_equal(out.cpu().numpy().view(np.int32), want, "int32", "A / B with one zero")
    good = to_device(np.ones(65536, np.int32))
    # the slot is cleared at the start of every call: the clean call reports nothing
    assert eb.ebin_execute_noalloc(plan.handle, dA.data_ptr(), good.data_ptr(), out.data_ptr(),
                                   s, 0) == 0
    assert_bits_equal(out.cpu().numpy().view(np.int32), a, "int32", "A / 1")


def test_noalloc_slots_read_back_later():
    """Calls that do not wait (status_bits NULL) leave their bits in their
    slot; ebin_noalloc_read_status returns them after the stream's work,
    without clearing, and each slot keeps its own call's bits."""
    n = 1 << 16
    a = np.arange(n, dtype=np.int32) - 5000
    zero_b = np.full(n, 3, np.int32)
    zero_b[777] = 0
    shifts = np.full(n, 5, np.uint32)
    shifts[4242] = 40
    pdiv = eb.Plan(eb.descriptor("Div", "int32"), (n,), (n,))
    pshift = eb.Plan(eb.descriptor("BitShift", "uint32", direction=0), (n,), (n,))
    dA, dZ = to_device(a), to_device(zero_b)
    dU, dS = to_device(a.view(np.uint32)), to_device(shifts)
    outs = [torch.empty(n * 4, dtype=torch.uint8, device="cuda") for _ in range(3)]
    s = torch.cuda.current_stream().cuda_stream
    eb.ebin_execute_noalloc(pdiv.handle, dA.data_ptr(), dZ.data_ptr(), outs[0].data_ptr(), s, 5,
                            want_status=False)
    eb.ebin_execute_noalloc(pshift.handle, dU.data_ptr(), dS.data_ptr(), outs[1].data_ptr(), s, 6,
                            want_status=False)
    eb.ebin_execute_noalloc(pdiv.handle, dA.data_ptr(), dA.data_ptr(), outs[2].data_ptr(), s, 7,
                            want_status=False)            # A / A: the element 5000 divides 0 / 0
    for slot, want in ((5, eb.DEVICE_DIV_BY_ZERO), (6, eb.DEVICE_SHIFT_RANGE),
                       (7, eb.DEVICE_DIV_BY_ZERO)):
        for _ in range(2):                                  # reading does not clear
            assert eb.ebin_noalloc_read_status(slot, s) == want, slot
    want_div, _ = oracle.run("Div", a, zero_b, "int32")
    want_shift, _ = oracle.run("BitShift", a.view(np.uint32), shifts, "uint32", direction=0)
    assert_bits_equal(outs[0].cpu().numpy().view(np.int32), want_div, "int32", "Div slot 5")
    assert_bits_equal(outs[1].cpu().numpy().view(np.uint32), want_shift, "uint32",
                      "BitShift slot 6")
    # a clean call on slot 5 clears it
    ones = to_device(np.ones(n, np.int32))
    eb.ebin_execute_noalloc(pdiv.handle, dA.data_ptr(), ones.data_ptr(), outs[0].data_ptr(), s, 5,
                            want_status=False)
    assert eb.ebin_noalloc_read_status(5, s) == 0
    assert eb.ebin_noalloc_read_status(6, s) == eb.DEVICE_SHIFT_RANGE


def test_noalloc_rejects_slots_beyond_the_array():
    plan = eb.Plan(eb.descriptor("Add", "float32"), (16,), (16,))
    x = torch.zeros(16, device="cuda")
    for slot in (-1, eb.NOALLOC_STATUS_SLOTS):
        with pytest.raises(eb.EbinError) as e:
            eb.ebin_execute_noalloc(plan.handle, x.data_ptr(), x.data_ptr(), x.data_ptr(), None,
                                    slot)
        assert e.value.code == "invalid_arg"
        with pytest.raises(eb.EbinError) as e:
            eb.ebin_noalloc_read_status(slot, None)
        assert e.value.code == "invalid_arg"
