"""ORACLE -- test infrastructure only.

Python access to the plain single-threaded C reference in ``ebin_oracle.c``.
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product (``broadcast_elementwise_gb300``)
never imports it, and this package never imports the product: they share no
code, no header and no table.

Operators and types are named by strings (ONNX operator names, numpy-style
type names) and mapped here to the oracle's own private codes.

Parity pins: see the header of ``ebin_oracle.c``.  Integer Pow with a negative
exponent follows a reading the pages leave open (the exact power truncated
toward zero); the oracle is pinned to that reading by exact rationals.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ebin_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

OPS = ["Add", "Sub", "Mul", "Div", "Mod", "Pow",
       "Equal", "Less", "Greater", "LessOrEqual", "GreaterOrEqual",
       "And", "Or", "Xor",
       "BitwiseAnd", "BitwiseOr", "BitwiseXor",
       "BitShift", "PRelu",
       "BatchNormalization", "Clip",
       "Max", "Min", "RSub", "RDiv", "BiasPRelu", "MulAdd", "BiasPReluBN"]
DTYPES = ["float32", "float16", "bfloat16", "int32", "int64", "uint8", "uint32", "bool",
          "int8", "int16", "uint16", "uint64", "float64"]
STORAGE = {"float32": np.float32, "float16": np.float16, "bfloat16": np.uint16,
           "int32": np.int32, "int64": np.int64, "uint8": np.uint8, "uint32": np.uint32,
           "bool": np.uint8, "int8": np.int8, "int16": np.int16, "uint16": np.uint16,
           "uint64": np.uint64, "float64": np.float64}
RC = {0: "ok", 1: "incompatible_shapes", 2: "invalid_arg", 3: "unsupported_type", 4: "invalid_attr"}
STATUS_DIV_BY_ZERO = 1
STATUS_SHIFT_RANGE = 2

# The flags are part of the oracle's definition: each float operation rounds alone.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def _elf_matches_host(path: str) -> bool:
    """True if the shared object at `path` was built for this machine's CPU."""
    import platform
    import struct
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
        return want is None or struct.unpack("<H", head[18:20])[0] == want
    except (OSError, struct.error):
        return False


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (plain C, no GPU needed)."""
    if (force or not os.path.exists(_LIB) or not _elf_matches_host(_LIB)
            or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32, i64, p, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
            lib.oracle_eval.argtypes = [i32, i32, i32, i32, f32, i32, i32, p, i32, p, i32,
                                        p, p, p, p, i64, p]
            lib.oracle_eval.restype = i32
            lib.oracle_output_shape.argtypes = [i32, p, i32, p, i32, p, p]
            lib.oracle_output_shape.restype = i32
            lib.oracle_eval_params.argtypes = [i32, i32, i32, f32, p, i32, p, i32, p, p, p, p,
                                               i64, p]
            lib.oracle_eval_params.restype = i32
            lib.oracle_eval_pow_mixed.argtypes = [i32, i32, p, i32, p, i32, p, p, p, p, i64, p]
            lib.oracle_eval_pow_mixed.restype = i32
            lib.oracle_eval3.argtypes = [i32, i32, p, i32, p, i32, p, i32, p, p, p, p, p, i64]
            lib.oracle_eval3.restype = i32
            lib.oracle_output_shape3.argtypes = [p, i32, p, i32, p, i32, p, p]
            lib.oracle_output_shape3.restype = i32
            lib.oracle_broadcast_shape.argtypes = [p, i32, p, i32, p, p]
            lib.oracle_broadcast_shape.restype = i32
            lib.oracle_offsets.argtypes = [p, i32, p, i32, p, i64, p, p]
            lib.oracle_offsets.restype = i32
            lib.oracle_check_descriptor.argtypes = [i32] * 6
            lib.oracle_check_descriptor.restype = i32
            lib.oracle_type_allowed.argtypes = [i32, i32]
            lib.oracle_type_allowed.restype = i32
            lib.oracle_output_type.argtypes = [i32, i32]
            lib.oracle_output_type.restype = i32
            for name in ("oracle_f32_to_f16_n", "oracle_f32_to_bf16_n", "oracle_f16_to_f32_n",
                         "oracle_bf16_to_f32_n"):
                getattr(lib, name).argtypes = [p, p, i64]
                getattr(lib, name).restype = None
            _lib = lib
    return _lib


def _shape_arr(shape):
    arr = np.array([int(d) for d in shape] or [0], dtype=np.int64)
    return arr, len(shape)


def output_shape(op: str, shape_a, shape_b):
    """Output shape of ``op`` on these input shapes, or raise ValueError with the code name."""
    lib = _load()
    sa, ra = _shape_arr(shape_a)
    sb, rb = _shape_arr(shape_b)
    so = np.zeros(8, np.int64)
    ro = ctypes.c_int(0)
    rc = lib.oracle_output_shape(OPS.index(op), sa.ctypes.data, ra, sb.ctypes.data, rb,
                                 so.ctypes.data, ctypes.byref(ro))
    if rc:
        raise ValueError(RC[rc])
    return tuple(int(x) for x in so[:ro.value])


def check_descriptor(op: str, opset: int, fmod: int, direction: int, ta: str, tb: str) -> str:
    rc = _load().oracle_check_descriptor(OPS.index(op), opset, fmod, direction,
                                         DTYPES.index(ta), DTYPES.index(tb))
    return RC[rc]


def type_allowed(op: str, t: str) -> bool:
    return bool(_load().oracle_type_allowed(OPS.index(op), DTYPES.index(t)))


def output_type(op: str, t: str) -> str:
    return DTYPES[_load().oracle_output_type(OPS.index(op), DTYPES.index(t))]


def offsets(shape_a, shape_b, idx):
    """Element offsets into A and B of the given flat output indices."""
    lib = _load()
    sa, ra = _shape_arr(shape_a)
    sb, rb = _shape_arr(shape_b)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    oa = np.empty(idx.size, np.int64)
    ob = np.empty(idx.size, np.int64)
    rc = lib.oracle_offsets(sa.ctypes.data, ra, sb.ctypes.data, rb, idx.ctypes.data, idx.size,
                            oa.ctypes.data, ob.ctypes.data)
    if rc:
        raise ValueError(RC[rc])
    return oa, ob


def run(op: str, a: np.ndarray, b: np.ndarray | None, dtype: str, *, shape_a=None, shape_b=None,
        fmod: int = 0, direction: int = 0, eps: float = 1e-5, has_min: bool = True,
        has_max: bool = True, idx=None):
    """Evaluate ``op`` on host arrays ``a`` and ``b`` (numpy storage of ``dtype``).

    Returns ``(out, status)``: ``out`` has the output shape (or, with ``idx``,
    one element per requested flat output index) in the output type's storage;
    ``status`` holds the validation bits (1 = integer division/modulo by zero
    or integer 0 to a negative power, 2 = shift count out of range).
    """
    lib = _load()
    a = np.ascontiguousarray(a)
    if a.dtype != STORAGE[dtype]:
        raise TypeError("A storage %s does not match %s" % (a.dtype, dtype))
    if b is not None:
        b = np.ascontiguousarray(b)
        if b.dtype != STORAGE[dtype]:
            raise TypeError("B storage %s does not match %s" % (b.dtype, dtype))
    shape_a = tuple(a.shape) if shape_a is None else tuple(shape_a)
    shape_b = (tuple(b.shape) if b is not None else (2,)) if shape_b is None else tuple(shape_b)
    oshape = output_shape(op, shape_a, shape_b)
    otype = output_type(op, dtype)
    sa, ra = _shape_arr(shape_a)
    sb, rb = _shape_arr(shape_b)
    if idx is None:
        out = np.empty(oshape, STORAGE[otype])
        idx_p, n_idx = None, 0
    else:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.empty(idx.size, STORAGE[otype])
        idx_p, n_idx = idx.ctypes.data, idx.size
    status = ctypes.c_uint32(0)
    rc = lib.oracle_eval(OPS.index(op), DTYPES.index(dtype), int(fmod), int(direction),
                         float(eps), int(bool(has_min)), int(bool(has_max)),
                         sa.ctypes.data, ra, sb.ctypes.data, rb,
                         a.ctypes.data, None if b is None else b.ctypes.data, out.ctypes.data,
                         idx_p, n_idx, ctypes.byref(status))
    if rc:
        raise ValueError(RC[rc])
    return out, int(status.value)


def run_params(op: str, a: np.ndarray, b: np.ndarray, dtype: str, dtype_b: str, *,
               eps: float = 1e-5, idx=None):
    """BatchNormalization / BiasPRelu / BiasPReluBN with the parameter block
    ``b`` stored as ``dtype_b`` (float32 beside fp16, bf16 or float64 x, or
    x's own type).  Returns the output like ``run`` (no status bits)."""
    lib = _load()
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if a.dtype != STORAGE[dtype] or b.dtype != STORAGE[dtype_b]:
        raise TypeError("storage %s / %s does not match %s / %s"
                        % (a.dtype, b.dtype, dtype, dtype_b))
    oshape = output_shape(op, a.shape, b.shape)
    sa, ra = _shape_arr(a.shape)
    sb, rb = _shape_arr(b.shape)
    if idx is None:
        out = np.empty(oshape, STORAGE[dtype])
        idx_p, n_idx = None, 0
    else:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.empty(idx.size, STORAGE[dtype])
        idx_p, n_idx = idx.ctypes.data, idx.size
    status = ctypes.c_uint32(0)
    rc = lib.oracle_eval_params(OPS.index(op), DTYPES.index(dtype), DTYPES.index(dtype_b),
                                float(eps), sa.ctypes.data, ra, sb.ctypes.data, rb,
                                a.ctypes.data, b.ctypes.data, out.ctypes.data, idx_p, n_idx,
                                ctypes.byref(status))
    if rc:
        raise ValueError(RC[rc])
    return out


def run_pow_mixed(a: np.ndarray, b: np.ndarray, dtype_a: str, dtype_b: str, *, idx=None):
    """Pow with base type dtype_a and exponent type dtype_b; returns (out, status)."""
    lib = _load()
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    if a.dtype != STORAGE[dtype_a] or b.dtype != STORAGE[dtype_b]:
        raise TypeError("storage does not match the types")
    oshape = tuple(np.broadcast_shapes(a.shape, b.shape))
    sa, ra = _shape_arr(tuple(a.shape))
    sb, rb = _shape_arr(tuple(b.shape))
    if idx is None:
        out = np.empty(oshape, STORAGE[dtype_a])
        idx_p, n_idx = None, 0
    else:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.empty(idx.size, STORAGE[dtype_a])
        idx_p, n_idx = idx.ctypes.data, idx.size
    status = ctypes.c_uint32(0)
    rc = lib.oracle_eval_pow_mixed(DTYPES.index(dtype_a), DTYPES.index(dtype_b), sa.ctypes.data,
                                   ra, sb.ctypes.data, rb, a.ctypes.data, b.ctypes.data,
                                   out.ctypes.data, idx_p, n_idx, ctypes.byref(status))
    if rc:
        raise ValueError(RC[rc])
    return out, int(status.value)


def output_shape3(shape_a, shape_b, shape_c) -> tuple:
    """broadcast(broadcast(A, B), C)."""
    sa, ra = _shape_arr(shape_a)
    sb, rb = _shape_arr(shape_b)
    sc, rc = _shape_arr(shape_c)
    so = np.zeros(8, np.int64)
    ro = ctypes.c_int(0)
    rcode = _load().oracle_output_shape3(sa.ctypes.data, ra, sb.ctypes.data, rb, sc.ctypes.data,
                                         rc, so.ctypes.data, ctypes.byref(ro))
    if rcode:
        raise ValueError(RC[rcode])
    return tuple(int(v) for v in so[: ro.value])


def run3(op: str, a: np.ndarray, b: np.ndarray, c: np.ndarray, dtype: str, *, idx=None):
    """Evaluate the three-input ``op`` (MulAdd) on host arrays in ``dtype``'s storage.

    Returns the output (output shape, or one element per flat index in ``idx``).
    """
    lib = _load()
    arrs = [np.ascontiguousarray(x) for x in (a, b, c)]
    for x in arrs:
        if x.dtype != STORAGE[dtype]:
            raise TypeError("storage %s does not match %s" % (x.dtype, dtype))
    shapes = [_shape_arr(tuple(x.shape)) for x in arrs]
    oshape = output_shape3(*(tuple(x.shape) for x in arrs))
    if idx is None:
        out = np.empty(oshape, STORAGE[dtype])
        idx_p, n_idx = None, 0
    else:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        out = np.empty(idx.size, STORAGE[dtype])
        idx_p, n_idx = idx.ctypes.data, idx.size
    rcode = lib.oracle_eval3(OPS.index(op), DTYPES.index(dtype),
                             shapes[0][0].ctypes.data, shapes[0][1],
                             shapes[1][0].ctypes.data, shapes[1][1],
                             shapes[2][0].ctypes.data, shapes[2][1],
                             arrs[0].ctypes.data, arrs[1].ctypes.data, arrs[2].ctypes.data,
                             out.ctypes.data, idx_p, n_idx)
    if rcode:
        raise ValueError(RC[rcode])
    return out


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint16)
    _load().oracle_f32_to_f16_n(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint16)
    _load().oracle_f32_to_bf16_n(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    y = np.empty(x.shape, np.float32)
    _load().oracle_f16_to_f32_n(x.ctypes.data, y.ctypes.data, x.size)
    return y


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    y = np.empty(x.shape, np.float32)
    _load().oracle_bf16_to_f32_n(x.ctypes.data, y.ctypes.data, x.size)
    return y
