"""ebin_execute_noalloc: the same results as ebin_execute, without the library
allocating device memory.

Callers whose device memory belongs entirely to their own allocator, plugins
whose host framework forbids allocation while enqueueing, and latency-critical
loops that cannot take cudaMalloc's implicit synchronisation use this entry
point; it keeps the validating kernels' status words in a fixed array
compiled into the library.  This file is collected last so that, if it fails,
a run stopping at the first failure has already run every other test; it
passes alone in a fresh process as well as after the rest of the suite.
"""
import numpy as np
import pytest

from conftest import assert_bits_equal
from engine_util import inputs_for, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
eb = pytest.importorskip("broadcast_elementwise_gb300")


def _reference(plan, dA, dB, nbytes):
    out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    eb.execute(plan, dA, dB, out)
    bits = eb.get_device_status()
    return out.cpu().numpy(), bits


@pytest.mark.parametrize("op,dtype,sa,sb,attrs", [
    ("Div", "int32", (512, 1024), (512, 1), {}),             # repeated block, status word used
    ("Mod", "int32", (300007,), (), {"fmod": 0}),            # right scalar, status word used
    ("BitShift", "uint32", (4096, 256), (256,), {"direction": 1}),
    ("Mul", "float32", (300007,), (300007,), {}),            # no status word at all
])
def test_noalloc_matches_execute_on_two_calls(op, dtype, sa, sb, attrs):
    a, b = inputs_for(op, dtype, sa, sb, seed=11)
    desc = eb.descriptor(op, dtype, **attrs)
    plan = eb.Plan(desc, sa, sb)
    dA, dB = to_device(a), to_device(b)
    nbytes = plan.numel * eb.ITEMSIZE[desc.out_dtype]
    want, want_bits = _reference(plan, dA, dB, nbytes)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
        bits = eb.ebin_execute_noalloc(plan.handle, dA.data_ptr(), dB.data_ptr(),
                                       out.data_ptr(), stream, 3)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        if dtype == "float32":
            assert_bits_equal(got.view(np.float32), want.view(np.float32), "float32",
                              "call %d" % call)
        else:
            assert (got == want).all(), "call %d differs from ebin_execute" % call
        assert bits == want_bits == 0, (call, bits)


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
    good = to_device(np.ones(65536, np.int32))
    # the slot is cleared at the start of every call: the clean call reports nothing
    assert eb.ebin_execute_noalloc(plan.handle, dA.data_ptr(), good.data_ptr(), out.data_ptr(),
                                   s, 0) == 0
    assert_bits_equal(out.cpu().numpy().view(np.int32), a, "int32", "A / 1")


def test_noalloc_rejects_slots_beyond_the_array():
    plan = eb.Plan(eb.descriptor("Add", "float32"), (16,), (16,))
    x = torch.zeros(16, device="cuda")
    for slot in (-1, eb.NOALLOC_STATUS_SLOTS):
        with pytest.raises(eb.EbinError) as e:
            eb.ebin_execute_noalloc(plan.handle, x.data_ptr(), x.data_ptr(), x.data_ptr(), None,
                                    slot)
        assert e.value.code == "invalid_arg"
