"""Seeded synthetic inputs for the engine's tests and benchmark.

This module only produces input values.  It contains none of the engine's
arithmetic and imports neither the oracle nor the CUDA library; both of those
receive the same arrays from here.

The generator is counter-based SplitMix64 (see ``datagen.c``): element ``i`` of
operand ``j`` under workload seed ``s`` is a pure function of ``(s*16 + j, i)``,
so any slice can be produced independently and in parallel.

Host arrays use plain numpy storage: float32, float16, int32, int64, uint8,
uint32, and uint16 bit patterns for bfloat16.  ``bool`` is one byte (0 or 1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "datagen.c")
_LIB = os.path.join(_HERE, "libdatagen.so")
_lib = None
_lock = threading.Lock()

STORAGE = {
    "float32": np.float32,
    "float16": np.float16,
    "bfloat16": np.uint16,
    "int32": np.int32,
    "int64": np.int64,
    "uint8": np.uint8,
    "uint32": np.uint32,
    "bool": np.uint8,
    "int8": np.int8,
    "int16": np.int16,
    "uint16": np.uint16,
    "uint64": np.uint64,
    "float64": np.float64,
}


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
    """Compile libdatagen.so next to its source (plain C, no GPU)."""
    if (force or not os.path.exists(_LIB) or not _elf_matches_host(_LIB)
            or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, dbl, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.dg_raw_u64.argtypes = [u64, i64, i64, p]
            lib.dg_raw_u32.argtypes = [u64, i64, i64, p]
            lib.dg_uniform_f32.argtypes = [u64, i64, i64, dbl, dbl, p]
            lib.dg_normal_f32.argtypes = [u64, i64, i64, dbl, dbl, p]
            lib.dg_absnormal_f32.argtypes = [u64, i64, i64, dbl, p]
            lib.dg_uniform_zeros_f32.argtypes = [u64, i64, i64, dbl, dbl, dbl, p]
            lib.dg_uniform_reject_f32.argtypes = [u64, i64, i64, dbl, dbl, dbl, p]
            lib.dg_int_range.argtypes = [u64, i64, i64, i64, i64, ctypes.c_int, p]
            for f in (lib.dg_raw_u64, lib.dg_raw_u32, lib.dg_uniform_f32, lib.dg_normal_f32,
                      lib.dg_absnormal_f32, lib.dg_uniform_zeros_f32, lib.dg_uniform_reject_f32,
                      lib.dg_int_range):
                f.restype = None
            _lib = lib
    return _lib


def stream(seed: int, operand: int) -> int:
    """Initial SplitMix64 state of operand ``operand`` under workload seed ``seed``."""
    return (seed * 16 + operand) & 0xFFFFFFFFFFFFFFFF


_CHUNK = 1 << 22


def _fill(fn, out: np.ndarray, s0: int, offset: int, *args) -> np.ndarray:
    n = out.size
    flat = out.reshape(-1)
    item = flat.itemsize
    base = flat.ctypes.data

    def run(lo):
        cnt = min(_CHUNK, n - lo)
        fn(s0, offset + lo, cnt, *args, ctypes.c_void_p(base + lo * item))

    if n <= _CHUNK:
        if n:
            run(0)
    else:
        workers = max(1, min(16, os.cpu_count() or 1))
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(run, range(0, n, _CHUNK)))
    return out


def raw_u32(seed, operand, n, offset=0):
    return _fill(_load().dg_raw_u32, np.empty(n, np.uint32), stream(seed, operand), offset)


def raw_u64(seed, operand, n, offset=0):
    return _fill(_load().dg_raw_u64, np.empty(n, np.uint64), stream(seed, operand), offset)


def uniform(seed, operand, n, lo, hi, offset=0):
    return _fill(_load().dg_uniform_f32, np.empty(n, np.float32), stream(seed, operand), offset,
                 float(lo), float(hi))


def normal(seed, operand, n, mu=0.0, sigma=1.0, offset=0):
    return _fill(_load().dg_normal_f32, np.empty(n, np.float32), stream(seed, operand), offset,
                 float(mu), float(sigma))


def absnormal(seed, operand, n, shift, offset=0):
    return _fill(_load().dg_absnormal_f32, np.empty(n, np.float32), stream(seed, operand), offset,
                 float(shift))


def uniform_zeros(seed, operand, n, lo, hi, pzero, offset=0):
    return _fill(_load().dg_uniform_zeros_f32, np.empty(n, np.float32), stream(seed, operand),
                 offset, float(lo), float(hi), float(pzero))


def uniform_reject(seed, operand, n, lo, hi, min_abs, offset=0):
    return _fill(_load().dg_uniform_reject_f32, np.empty(n, np.float32), stream(seed, operand),
                 offset, float(lo), float(hi), float(min_abs))


def int_range(seed, operand, n, lo, hi, skip_zero=False, offset=0):
    return _fill(_load().dg_int_range, np.empty(n, np.int64), stream(seed, operand), offset,
                 int(lo), int(hi), 1 if skip_zero else 0)


def float_to(values: np.ndarray, dtype: str) -> np.ndarray:
    """Store float32 generator output in ``dtype`` (round to nearest even)."""
    values = np.ascontiguousarray(values, dtype=np.float32)
    if dtype == "float32":
        return values
    if dtype == "float64":
        return values.astype(np.float64)
    if dtype == "float16":
        return values.astype(np.float16)
    if dtype == "bfloat16":
        import torch
        t = torch.from_numpy(values).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError("float_to: not a floating dtype: %s" % dtype)


def int_to(values: np.ndarray, dtype: str) -> np.ndarray:
    """Narrow generator integers to ``dtype`` by two's-complement wrap."""
    v = np.asarray(values).astype(np.int64)
    if dtype == "bool":
        return (v & 1).astype(np.uint8)
    width = np.dtype(STORAGE[dtype]).itemsize
    utype = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[width]
    return v.view(np.uint64).astype(utype, casting="unsafe").view(STORAGE[dtype])


def make(kind: str, dtype: str, shape, seed: int, operand: int, **kw) -> np.ndarray:
    """One operand of a workload as a numpy array of ``shape`` in ``dtype`` storage.

    kind: "uniform" (lo, hi), "normal", "absnormal" (shift), "uniform_zeros"
    (lo, hi, pzero), "uniform_reject" (lo, hi, min_abs), "int_range" (lo, hi,
    skip_zero), "bits" (raw pattern of the dtype's width), "bool".
    """
    shape = tuple(int(d) for d in shape)
    n = int(np.prod(shape, dtype=np.int64)) if shape else 1
    if kind == "uniform":
        v = float_to(uniform(seed, operand, n, kw.get("lo", -1.0), kw.get("hi", 1.0)), dtype) \
            if dtype in ("float32", "float16", "bfloat16", "float64") else None
    elif kind == "normal":
        v = float_to(normal(seed, operand, n), dtype)
    elif kind == "absnormal":
        v = float_to(absnormal(seed, operand, n, kw.get("shift", 0.5)), dtype)
    elif kind == "uniform_zeros":
        v = float_to(uniform_zeros(seed, operand, n, kw["lo"], kw["hi"], kw["pzero"]), dtype)
    elif kind == "uniform_reject":
        v = float_to(uniform_reject(seed, operand, n, kw["lo"], kw["hi"], kw["min_abs"]), dtype)
    elif kind == "int_range":
        v = int_to(int_range(seed, operand, n, kw["lo"], kw["hi"], kw.get("skip_zero", False)),
                   dtype)
    elif kind == "bits":
        width = np.dtype(STORAGE[dtype]).itemsize
        raw = raw_u64(seed, operand, n) if width == 8 else raw_u32(seed, operand, n).astype(np.uint64)
        utype = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[width]
        v = raw.astype(utype, casting="unsafe").view(STORAGE[dtype])
    elif kind == "bool":
        v = (raw_u32(seed, operand, n) >> 31).astype(np.uint8)
    else:
        raise ValueError("unknown input kind %r" % kind)
    if v is None:
        raise ValueError("kind %r does not apply to dtype %s" % (kind, dtype))
    return np.ascontiguousarray(v).reshape(shape)
