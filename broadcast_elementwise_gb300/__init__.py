"""GB300-native ONNX broadcast binary elementwise engine: Python binding.

A thin ctypes binding of ``libebin.so``, whose C ABI (``include/ebin.h``) is
the product's boundary.  The ``ebin_*`` functions here have the C names and
only marshal arguments; every step of the path (descriptor checks, planning,
the plan cache, validation and the elementwise kernels) runs in the library.
PyTorch is used for device memory and streams only.

Importing this package loads the library and fails loudly if it is missing:
there is no CPU or eager fallback.

Typical use::

    import torch, broadcast_elementwise_gb300 as eb
    y = eb.binary("Add", x, b)                   # allocates y, runs on the current stream

    desc = eb.Descriptor("Mod", "float32", fmod=0, opset=28)
    plan = eb.Plan(desc, a.shape, b.shape)
    eb.execute(plan, a, b, out)
"""
from __future__ import annotations

import ctypes
import os
import struct

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libebin.so")

OPS = {"Add": 0, "Sub": 1, "Mul": 2, "Div": 3, "Mod": 4, "Pow": 5,
       "Equal": 6, "Less": 7, "Greater": 8, "LessOrEqual": 9, "GreaterOrEqual": 10,
       "And": 11, "Or": 12, "Xor": 13,
       "BitwiseAnd": 14, "BitwiseOr": 15, "BitwiseXor": 16,
       "BitShift": 17, "PRelu": 18, "BatchNormalization": 19, "Clip": 20,
       "Max": 21, "Min": 22, "RSub": 23, "RDiv": 24, "BiasPRelu": 25, "MulAdd": 26,
       "BiasPReluBN": 27}
DTYPES = {"float32": 1, "uint8": 2, "int8": 3, "uint16": 4, "int16": 5, "int32": 6, "int64": 7,
          "bool": 9, "float16": 10, "float64": 11, "uint32": 12, "uint64": 13, "bfloat16": 16}
DTYPE_NAMES = {v: k for k, v in DTYPES.items()}
ITEMSIZE = {"float32": 4, "uint8": 1, "int32": 4, "int64": 8, "bool": 1, "float16": 2,
            "uint32": 4, "bfloat16": 2, "int8": 1, "int16": 2, "uint16": 2, "uint64": 8,
            "float64": 8}
FAMILIES = {"auto": -1, "empty": 0, "contiguous": 1, "left_scalar": 2, "right_scalar": 3,
            "repeated_block": 4, "inner_vector_outer": 5, "general_strided": 6}
FAMILY_NAMES = {v: k for k, v in FAMILIES.items()}
STATUS = {0: "ok", 1: "invalid_arg", 2: "unsupported_op", 3: "unsupported_type",
          4: "invalid_attr", 5: "incompatible_shapes", 6: "rank_too_large", 7: "alias",
          8: "cuda", 9: "family"}
DEVICE_DIV_BY_ZERO = 0x1
DEVICE_SHIFT_RANGE = 0x2
MAX_RANK = 8
PLAN_CACHE_CAPACITY = 8


class EbinError(RuntimeError):
    """A non-OK status returned by the C ABI; ``.code`` holds its name."""

    def __init__(self, status: int, where: str):
        self.status = status
        self.code = STATUS.get(status, "unknown")
        super().__init__("%s: %s" % (where, self.code))


class ebin_attrs(ctypes.Structure):
    _fields_ = [("fmod", ctypes.c_int32), ("direction", ctypes.c_int32),
                ("epsilon", ctypes.c_float), ("clip_has_min", ctypes.c_int32),
                ("clip_has_max", ctypes.c_int32), ("with_scalar", ctypes.c_int32),
                ("scalar_b", ctypes.c_float)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libebin.so is not built (%s); run __graft_entry__.build() or "
                          "python broadcast_elementwise_gb300/_build.py" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    p_i64 = ctypes.POINTER(ctypes.c_int64)
    sigs = {
        "ebin_descriptor_create": (i32, [i32, i32, ctypes.POINTER(ebin_attrs), i32, i32,
                                         ctypes.POINTER(vp)]),
        "ebin_descriptor_output_dtype": (i32, [vp, ctypes.POINTER(ctypes.c_int)]),
        "ebin_descriptor_id": (i32, [vp, ctypes.POINTER(ctypes.c_uint64)]),
        "ebin_descriptor_destroy": (None, [vp]),
        "ebin_plan_create": (i32, [vp, p_i64, i32, p_i64, i32, ctypes.POINTER(vp)]),
        "ebin_plan_create_forced": (i32, [vp, p_i64, i32, p_i64, i32, i32, ctypes.POINTER(vp)]),
        "ebin_plan_create3": (i32, [vp, p_i64, i32, p_i64, i32, p_i64, i32, ctypes.POINTER(vp)]),
        "ebin_plan_create_strided": (i32, [vp, p_i64, p_i64, i32, p_i64, p_i64, i32, i32,
                                           ctypes.POINTER(vp)]),
        "ebin_plan_create3_forced": (i32, [vp, p_i64, i32, p_i64, i32, p_i64, i32, i32,
                                           ctypes.POINTER(vp)]),
        "ebin_execute3": (i32, [vp, vp, vp, vp, vp, vp]),
        "ebin_plan_output_shape": (i32, [vp, p_i64, ctypes.POINTER(ctypes.c_int)]),
        "ebin_plan_numel": (i32, [vp, p_i64]),
        "ebin_plan_family": (i32, [vp, ctypes.POINTER(ctypes.c_int)]),
        "ebin_plan_geometry": (i32, [vp, ctypes.POINTER(ctypes.c_int), p_i64, p_i64, p_i64]),
        "ebin_plan_release": (None, [vp]),
        "ebin_plan_cache_stats": (i32, [ctypes.POINTER(ctypes.c_uint64),
                                        ctypes.POINTER(ctypes.c_uint64),
                                        ctypes.POINTER(ctypes.c_int)]),
        "ebin_plan_cache_clear": (None, []),
        "ebin_execute": (i32, [vp, vp, vp, vp, vp]),
        "ebin_execute_host": (i32, [vp, vp, vp, vp, vp, vp, vp, vp]),
        "ebin_execute_mapped": (i32, [vp, vp, vp, vp, vp]),
        "ebin_execute3_mapped": (i32, [vp, vp, vp, vp, vp, vp]),
        "ebin_get_device_status": (i32, [vp, ctypes.POINTER(ctypes.c_uint32)]),
        "ebin_execute_noalloc": (i32, [vp, vp, vp, vp, vp, i32, ctypes.POINTER(ctypes.c_uint32)]),
        "ebin_noalloc_read_status": (i32, [i32, vp, ctypes.POINTER(ctypes.c_uint32)]),
        "ebin_launch_count": (ctypes.c_uint64, []),
        "ebin_dtype_size": (ctypes.c_size_t, [i32]),
        "ebin_status_string": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _check(status: int, where: str):
    if status != 0:
        raise EbinError(status, where)


def _shape(shape):
    dims = [int(d) for d in shape]
    arr = (ctypes.c_int64 * max(1, len(dims)))(*dims)
    return arr, len(dims)


def _ptr(x) -> int | None:
    """Device address of a tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- the C ABI, by name

def ebin_descriptor_create(op, opset, attrs, dtype_a, dtype_b) -> int:
    out = ctypes.c_void_p()
    _check(lib.ebin_descriptor_create(op, opset, ctypes.byref(attrs) if attrs else None,
                                      dtype_a, dtype_b, ctypes.byref(out)),
           "ebin_descriptor_create")
    return out.value


def ebin_descriptor_output_dtype(desc) -> int:
    v = ctypes.c_int()
    _check(lib.ebin_descriptor_output_dtype(desc, ctypes.byref(v)), "ebin_descriptor_output_dtype")
    return v.value


def ebin_descriptor_id(desc) -> int:
    v = ctypes.c_uint64()
    _check(lib.ebin_descriptor_id(desc, ctypes.byref(v)), "ebin_descriptor_id")
    return v.value


def ebin_descriptor_destroy(desc) -> None:
    lib.ebin_descriptor_destroy(desc)


def ebin_plan_create(desc, shape_a, shape_b) -> int:
    sa, ra = _shape(shape_a)
    sb, rb = _shape(shape_b)
    out = ctypes.c_void_p()
    _check(lib.ebin_plan_create(desc, sa, ra, sb, rb, ctypes.byref(out)), "ebin_plan_create")
    return out.value


def ebin_plan_create_forced(desc, shape_a, shape_b, family) -> int:
    sa, ra = _shape(shape_a)
    sb, rb = _shape(shape_b)
    out = ctypes.c_void_p()
    _check(lib.ebin_plan_create_forced(desc, sa, ra, sb, rb, family, ctypes.byref(out)),
           "ebin_plan_create_forced")
    return out.value


def ebin_plan_create_strided(desc, shape_a, strides_a, shape_b, strides_b, family=-1) -> int:
    """Marshal ebin_plan_create_strided (strides None = dense)."""
    sa, ra = _shape(shape_a)
    sb, rb = _shape(shape_b)
    ta = _shape(strides_a)[0] if strides_a is not None else None
    tb = _shape(strides_b)[0] if strides_b is not None else None
    out = ctypes.c_void_p()
    _check(lib.ebin_plan_create_strided(desc, sa, ta, ra, sb, tb, rb, family, ctypes.byref(out)),
           "ebin_plan_create_strided")
    return out.value


def ebin_plan_create3(desc, shape_a, shape_b, shape_c, family=None) -> int:
    """Marshal ebin_plan_create3 (family None) or ebin_plan_create3_forced."""
    sa, ra = _shape(shape_a)
    sb, rb = _shape(shape_b)
    sc, rc = _shape(shape_c)
    out = ctypes.c_void_p()
    if family is None:
        _check(lib.ebin_plan_create3(desc, sa, ra, sb, rb, sc, rc, ctypes.byref(out)),
               "ebin_plan_create3")
    else:
        _check(lib.ebin_plan_create3_forced(desc, sa, ra, sb, rb, sc, rc, family,
                                            ctypes.byref(out)), "ebin_plan_create3_forced")
    return out.value


def ebin_plan_output_shape(plan) -> tuple:
    shape = (ctypes.c_int64 * MAX_RANK)()
    rank = ctypes.c_int()
    _check(lib.ebin_plan_output_shape(plan, shape, ctypes.byref(rank)), "ebin_plan_output_shape")
    return tuple(shape[i] for i in range(rank.value))


def ebin_plan_numel(plan) -> int:
    v = ctypes.c_int64()
    _check(lib.ebin_plan_numel(plan, ctypes.byref(v)), "ebin_plan_numel")
    return v.value


def ebin_plan_family(plan) -> int:
    v = ctypes.c_int()
    _check(lib.ebin_plan_family(plan, ctypes.byref(v)), "ebin_plan_family")
    return v.value


def ebin_plan_geometry(plan):
    rank = ctypes.c_int()
    n, sa, sb = ((ctypes.c_int64 * MAX_RANK)() for _ in range(3))
    _check(lib.ebin_plan_geometry(plan, ctypes.byref(rank), n, sa, sb), "ebin_plan_geometry")
    r = rank.value
    return [n[i] for i in range(r)], [sa[i] for i in range(r)], [sb[i] for i in range(r)]


def ebin_plan_release(plan) -> None:
    lib.ebin_plan_release(plan)


def ebin_plan_cache_stats():
    h, m, s = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_int()
    _check(lib.ebin_plan_cache_stats(ctypes.byref(h), ctypes.byref(m), ctypes.byref(s)),
           "ebin_plan_cache_stats")
    return h.value, m.value, s.value


def ebin_plan_cache_clear() -> None:
    lib.ebin_plan_cache_clear()


def ebin_execute(plan, A, B, out, stream) -> None:
    _check(lib.ebin_execute(plan, A, B, out, stream), "ebin_execute")


def ebin_execute3(plan, A, B, C, out, stream) -> None:
    _check(lib.ebin_execute3(plan, A, B, C, out, stream), "ebin_execute3")


def ebin_execute_host(plan, host_a, host_b, host_out, dev_a, dev_b, dev_out, stream) -> None:
    _check(lib.ebin_execute_host(plan, host_a, host_b, host_out, dev_a, dev_b, dev_out, stream),
           "ebin_execute_host")


def ebin_execute_mapped(plan, host_a, host_b, host_out, stream) -> None:
    _check(lib.ebin_execute_mapped(plan, host_a, host_b, host_out, stream), "ebin_execute_mapped")


def ebin_execute3_mapped(plan, host_a, host_b, host_c, host_out, stream) -> None:
    _check(lib.ebin_execute3_mapped(plan, host_a, host_b, host_c, host_out, stream),
           "ebin_execute3_mapped")


def ebin_execute_noalloc(plan, A, B, out, stream, status_slot, want_status=True):
    """Marshal ebin_execute_noalloc; returns the status bits (0 when not requested)."""
    bits = ctypes.c_uint32(0)
    _check(lib.ebin_execute_noalloc(plan, A, B, out, stream, int(status_slot),
                                    ctypes.byref(bits) if want_status else None),
           "ebin_execute_noalloc")
    return bits.value


NOALLOC_STATUS_SLOTS = 64


def ebin_noalloc_read_status(status_slot, stream) -> int:
    """Marshal ebin_noalloc_read_status; returns the slot's status bits."""
    v = ctypes.c_uint32(0)
    _check(lib.ebin_noalloc_read_status(int(status_slot), stream, ctypes.byref(v)),
           "ebin_noalloc_read_status")
    return v.value


def ebin_get_device_status(stream) -> int:
    v = ctypes.c_uint32()
    _check(lib.ebin_get_device_status(stream, ctypes.byref(v)), "ebin_get_device_status")
    return v.value


def ebin_launch_count() -> int:
    return int(lib.ebin_launch_count())


def ebin_dtype_size(dtype) -> int:
    return int(lib.ebin_dtype_size(dtype))


def ebin_status_string(status) -> str:
    return lib.ebin_status_string(status).decode()


# ----------------------------------------------------------------- thin object wrappers

def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    if isinstance(dtype, str):
        return DTYPES[dtype]
    return DTYPES[torch_dtype_name(dtype)]


def torch_dtype_name(t) -> str:
    import torch
    table = {torch.float32: "float32", torch.float16: "float16", torch.bfloat16: "bfloat16",
             torch.int32: "int32", torch.int64: "int64", torch.uint8: "uint8",
             torch.bool: "bool", torch.uint32: "uint32", torch.int8: "int8",
             torch.int16: "int16", torch.uint16: "uint16", torch.uint64: "uint64",
             torch.float64: "float64"}
    return table[t]


def torch_dtype(name: str):
    import torch
    return {"float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16,
            "int32": torch.int32, "int64": torch.int64, "uint8": torch.uint8,
            "bool": torch.bool, "uint32": torch.uint32, "int8": torch.int8,
            "int16": torch.int16, "uint16": torch.uint16, "uint64": torch.uint64,
            "float64": torch.float64}[name]


class Descriptor:
    """Owns an ebin descriptor (operator, opset, attributes, element type)."""

    def __init__(self, op: str, dtype, *, opset: int = 28, fmod: int = 0, direction: int = 0,
                 epsilon: float = 1e-5, has_min: bool = True, has_max: bool = True,
                 scalar_b: float | None = None, dtype_b=None):
        """``scalar_b`` given: ncnn binaryop's with_scalar, B is that value.
        ``dtype_b``: B's type where it may differ from A's (Pow's exponent;
        a float32 parameter block of BatchNormalization, BiasPRelu or
        BiasPReluBN beside float16, bfloat16 or float64 x)."""
        self.op = op
        self.dtype = DTYPE_NAMES[_dtype_code(dtype)]
        self.dtype_b = self.dtype if dtype_b is None else DTYPE_NAMES[_dtype_code(dtype_b)]
        self.with_scalar = scalar_b is not None
        attrs = ebin_attrs(int(fmod), int(direction), float(epsilon), int(bool(has_min)),
                           int(bool(has_max)), int(self.with_scalar),
                           float(scalar_b) if self.with_scalar else 0.0)
        code = _dtype_code(dtype)
        code_b = code if dtype_b is None else _dtype_code(dtype_b)
        self.handle = ebin_descriptor_create(OPS[op], int(opset), attrs, code, code_b)
        self.out_dtype = DTYPE_NAMES[ebin_descriptor_output_dtype(self.handle)]
        self.id = ebin_descriptor_id(self.handle)

    def close(self):
        if self.handle:
            ebin_descriptor_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Plan:
    """Holds one plan reference for (descriptor, shape_a, shape_b)."""

    def __init__(self, desc: Descriptor, shape_a, shape_b, family: str | None = None,
                 strides_a=None, strides_b=None):
        """strides_a / strides_b: element strides of strided input views (None = dense)."""
        self.desc = desc
        self.shape_a = tuple(int(d) for d in shape_a)
        self.shape_b = tuple(int(d) for d in shape_b)
        if strides_a is not None or strides_b is not None:
            self.handle = ebin_plan_create_strided(
                desc.handle, self.shape_a, strides_a, self.shape_b, strides_b,
                -1 if family is None else FAMILIES[family])
        elif family is None:
            self.handle = ebin_plan_create(desc.handle, self.shape_a, self.shape_b)
        else:
            self.handle = ebin_plan_create_forced(desc.handle, self.shape_a, self.shape_b,
                                                  FAMILIES[family])
        self.output_shape = ebin_plan_output_shape(self.handle)
        self.numel = ebin_plan_numel(self.handle)
        self.family = FAMILY_NAMES[ebin_plan_family(self.handle)]

    def geometry(self):
        return ebin_plan_geometry(self.handle)

    def close(self):
        if self.handle:
            ebin_plan_release(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Plan3(Plan):
    """Holds one three-input plan reference (MulAdd) for (descriptor, shapes A, B, C)."""

    def __init__(self, desc: Descriptor, shape_a, shape_b, shape_c, family: str | None = None):
        self.desc = desc
        self.shape_a = tuple(int(d) for d in shape_a)
        self.shape_b = tuple(int(d) for d in shape_b)
        self.shape_c = tuple(int(d) for d in shape_c)
        self.handle = ebin_plan_create3(desc.handle, self.shape_a, self.shape_b, self.shape_c,
                                        None if family is None else FAMILIES[family])
        self.output_shape = ebin_plan_output_shape(self.handle)
        self.numel = ebin_plan_numel(self.handle)
        self.family = FAMILY_NAMES[ebin_plan_family(self.handle)]


def execute3(plan: Plan3, A, B, C, out, stream=None) -> None:
    """Enqueue a three-input plan on device buffers (torch tensors or int addresses)."""
    ebin_execute3(plan.handle, _ptr(A), _ptr(B), _ptr(C), _ptr(out), _stream(stream))


def execute(plan: Plan, A, B, out, stream=None) -> None:
    """Enqueue the plan on device buffers (torch tensors or int addresses)."""
    ebin_execute(plan.handle, _ptr(A), _ptr(B), _ptr(out), _stream(stream))


def execute_mapped(plan: Plan, A, B, out, stream=None) -> None:
    """Enqueue the plan on pinned host buffers, read and written in place by the
    kernel (torch pinned tensors or int addresses)."""
    ebin_execute_mapped(plan.handle, _ptr(A), _ptr(B), _ptr(out), _stream(stream))


def execute3_mapped(plan: Plan3, A, B, C, out, stream=None) -> None:
    """Enqueue a three-input plan on pinned host buffers, in place."""
    ebin_execute3_mapped(plan.handle, _ptr(A), _ptr(B), _ptr(C), _ptr(out), _stream(stream))


def get_device_status(stream=None) -> int:
    return ebin_get_device_status(_stream(stream))


_descriptors: dict = {}


def _attr_key(v):
    """Cache key of an attribute value: floats by bit pattern (-0.0 is not 0.0,
    and a NaN matches itself)."""
    return ("f", struct.pack("<d", v)) if isinstance(v, float) else v


def descriptor(op: str, dtype, **attrs) -> Descriptor:
    """A process-wide Descriptor per (op, dtype, attributes), so plans stay cached."""
    key = (op, _dtype_code(dtype), tuple(sorted((k, _attr_key(v)) for k, v in attrs.items())))
    d = _descriptors.get(key)
    if d is None:
        d = _descriptors[key] = Descriptor(op, dtype, **attrs)
    return d


def binary(op: str, a, b, out=None, *, stream=None, **attrs):
    """One-shot call: returns ``out`` (allocated if None).

    On torch CUDA tensors, inputs that are not contiguous run as strided views
    (no copy), except a BatchNormalization / Clip / BiasPRelu / BiasPReluBN
    parameter block, which is copied.  On pinned CPU tensors (contiguous),
    the kernel reads and writes host memory in place (ebin_execute_mapped;
    ``out`` is allocated pinned); synchronise ``stream`` before reading it.
    """
    import torch
    if (b is not None and op in ("BatchNormalization", "BiasPRelu", "BiasPReluBN")
            and b.dtype != a.dtype and "dtype_b" not in attrs):
        attrs["dtype_b"] = b.dtype      # a float32 parameter block beside 16-bit or float64 x
    desc = descriptor(op, a.dtype, **attrs)
    plain_b = op not in ("BatchNormalization", "Clip", "BiasPRelu", "BiasPReluBN")
    if b is not None and b.dtype != torch_dtype(desc.dtype_b):
        raise ValueError("binary: B is %s; %s on %s takes B of %s"
                         % (b.dtype, op, desc.dtype, desc.dtype_b))
    if not a.is_cuda:
        if not a.is_pinned() or (b is not None and not b.is_pinned()):
            raise ValueError("binary: CPU tensors must be pinned (tensor.pin_memory())")
        if not a.is_contiguous() or (b is not None and not b.is_contiguous()):
            raise ValueError("binary: pinned CPU tensors must be contiguous")
        plan = Plan(desc, a.shape, b.shape if b is not None else (2,))
        out = _output(out, plan, desc, None)
        execute_mapped(plan, a, b, out, stream)
        return out
    if b is not None and b.device != a.device:
        raise ValueError("binary: A is on %s and B on %s" % (a.device, b.device))
    if b is not None and not plain_b:
        b = b.contiguous()
    ta = None if a.is_contiguous() else tuple(a.stride())
    tb = None if (b is None or b.is_contiguous()) else tuple(b.stride())
    plan = Plan(desc, a.shape, b.shape if b is not None else (2,), strides_a=ta, strides_b=tb)
    out = _output(out, plan, desc, a.device)
    with torch.cuda.device(a.device):
        execute(plan, a, b, out, stream)
    return out


def _output(out, plan, desc, device):
    """The output tensor of binary(): allocated when None (pinned host memory
    when device is None), else checked to be what the kernel writes: the
    output's type and shape, contiguous, on that device (or pinned)."""
    import torch
    want = torch_dtype(desc.out_dtype)
    if out is None:
        if device is None:
            return torch.empty(plan.output_shape, dtype=want).pin_memory()
        return torch.empty(plan.output_shape, dtype=want, device=device)
    if out.dtype != want or tuple(out.shape) != tuple(plan.output_shape):
        raise ValueError("binary: out is %s %s; the result is %s %s"
                         % (out.dtype, tuple(out.shape), desc.out_dtype, tuple(plan.output_shape)))
    if not out.is_contiguous():
        raise ValueError("binary: out must be contiguous")
    if device is None and (out.is_cuda or not out.is_pinned()):
        raise ValueError("binary: out must be a pinned CPU tensor, as the inputs are")
    if device is not None and out.device != device:
        raise ValueError("binary: A is on %s and out on %s" % (device, out.device))
    return out
