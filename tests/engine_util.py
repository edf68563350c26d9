"""Helpers shared by the GPU tests: run the engine through the C ABI on host
arrays, and build seeded inputs for each operator and type."""
from __future__ import annotations

import numpy as np

import datagen

FLOATS = ("float32", "float16", "bfloat16", "float64")
INTS = ("int32", "int64", "uint8", "uint32", "int8", "int16", "uint16", "uint64")
ALL_DTYPES = FLOATS + INTS + ("bool",)

# operator -> element types (the engine's manifest; the oracle's agrees, see test_planner)
MANIFEST = {
    "Add": FLOATS + INTS, "Sub": FLOATS + INTS, "Mul": FLOATS + INTS, "Div": FLOATS + INTS,
    "Mod": FLOATS + INTS, "Pow": FLOATS + ("int32", "int64"),
    "Equal": ALL_DTYPES, "Less": FLOATS + INTS, "Greater": FLOATS + INTS,
    "LessOrEqual": FLOATS + INTS, "GreaterOrEqual": FLOATS + INTS,
    "And": ("bool",), "Or": ("bool",), "Xor": ("bool",),
    "BitwiseAnd": INTS, "BitwiseOr": INTS, "BitwiseXor": INTS,
    "BitShift": ("uint8", "uint16", "uint32", "uint64"),
    "PRelu": FLOATS + ("int32", "int64", "uint32", "uint64"),
    "BatchNormalization": FLOATS,
    "Clip": FLOATS + INTS,
    "Max": FLOATS + INTS, "Min": FLOATS + INTS, "RSub": FLOATS + INTS, "RDiv": FLOATS + INTS,
    "BiasPRelu": FLOATS, "BiasPReluBN": FLOATS,
}
ONE_WAY = ("PRelu", "BatchNormalization", "Clip", "BiasPRelu", "BiasPReluBN")
# parameter rows of the per-channel operators' B blocks
PARAM_ROWS = {"BatchNormalization": 4, "BiasPRelu": 2, "BiasPReluBN": 6}


def every_16bit_value(shape):
    """x[n, c, ...] whose every channel holds every 16-bit pattern (NaNs,
    infinities, subnormals and both zeros included), at least once."""
    N, C = shape[0], shape[1]
    S = int(np.prod(shape[2:]))
    n = np.arange(N, dtype=np.int64)[:, None, None]
    c = np.arange(C, dtype=np.int64)[None, :, None]
    s = np.arange(S, dtype=np.int64)[None, None, :]
    return ((n * S + s + 977 * c) % 65536).astype(np.uint16).reshape(shape)


def chain_params(op, C, seed, wide):
    """Seeded binary32 parameter rows of a per-channel chain, [rows, C]:
    ordinary normal values, or (wide) magnitudes over many binades with signs
    mixed and some exact zeros; the variance row positive, BiasPReluBN's slope
    row in [0, 1)."""
    rows = PARAM_ROWS[op]
    rng = np.random.default_rng(seed)
    p = rng.standard_normal((rows, C)).astype(np.float32)
    if wide:       # magnitudes over many binades, signs mixed, some exact zeros
        p *= np.float32(2.0) ** rng.integers(-30, 30, (rows, C)).astype(np.float32)
        p[rng.random((rows, C)) < 0.05] = 0.0
    p[-1] = np.abs(p[-1]) + np.float32(0.05)                  # variance
    if op == "BiasPReluBN":
        p[1] = np.abs(p[1]) * np.float32(0.3)                 # slope
    return p



def to_device(arr: np.ndarray):
    import torch
    flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
    return torch.from_numpy(flat.copy()).cuda()


def run_engine(op, dtype, a, b, *, shape_a=None, shape_b=None, family=None, attrs=None,
               out_fill=0xAB):
    """Run one plan on the GPU; returns (out as numpy, device status bits, family)."""
    import torch
    import broadcast_elementwise_gb300 as eb
    attrs = attrs or {}
    desc = eb.descriptor(op, dtype, **attrs)
    sa = tuple(a.shape) if shape_a is None else tuple(shape_a)
    sb = (tuple(b.shape) if b is not None else (2,)) if shape_b is None else tuple(shape_b)
    plan = eb.Plan(desc, sa, sb, family=family)
    otype = desc.out_dtype
    osize = eb.ITEMSIZE[otype]
    dA = to_device(a)
    dB = to_device(b) if b is not None else None
    out = torch.full((max(plan.numel, 1) * osize,), out_fill, dtype=torch.uint8, device="cuda")
    eb.execute(plan, dA if a.size else None, dB if (b is not None and b.size) else None,
               out if plan.numel else None)
    bits = eb.get_device_status()
    host = out.cpu().numpy()[: plan.numel * osize].view(datagen.STORAGE[otype])
    return host.reshape(plan.output_shape), bits, plan.family


def run_engine3(op, dtype, a, b, c, *, family=None, offset=0):
    """Run one three-input plan on the GPU (offset: elements by which every
    buffer is shifted off 16-byte alignment); returns (out, family)."""
    import torch
    import broadcast_elementwise_gb300 as eb
    desc = eb.descriptor(op, dtype)
    plan = eb.Plan3(desc, a.shape, b.shape, c.shape, family=family)
    isz = eb.ITEMSIZE[dtype]
    bufs = [to_device(np.concatenate([np.zeros(offset, x.dtype), x.reshape(-1)]))
            for x in (a, b, c)]
    out = torch.full(((max(plan.numel, 1) + offset) * isz + 16,), 0xAB, dtype=torch.uint8,
                     device="cuda")
    ptrs = [x.data_ptr() + offset * isz for x in bufs]
    eb.execute3(plan, *ptrs, out.data_ptr() + offset * isz)
    host = out.cpu().numpy()[offset * isz: (offset + plan.numel) * isz]
    return host.view(datagen.STORAGE[dtype]).reshape(plan.output_shape), plan.family


def specials(dtype):
    v = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 0.5, -2.5, 65504.0, 1e-7,
                  3.0, -7.0, 1e30, -1e-30], np.float32)
    return datagen.float_to(v, dtype)


def inputs_for(op, dtype, shape_a, shape_b, seed=0, attrs=None):
    """Seeded inputs matched to the operator (ranges where its semantics are interesting)."""
    attrs = attrs or {}
    mk = datagen.make
    if op == "BatchNormalization":
        C = shape_b[1]
        a = mk("normal", dtype, shape_a, seed, 0)
        params = np.concatenate([
            datagen.normal(seed, 1, C), datagen.normal(seed, 2, C), datagen.normal(seed, 3, C),
            datagen.uniform(seed, 4, C, 0.1, 2.0)]).astype(np.float32)
        return a, datagen.float_to(params, dtype).reshape(shape_b)
    if op == "BiasPRelu":
        C = shape_b[1]
        a = mk("normal", dtype, shape_a, seed, 0)
        _sprinkle(a, specials(dtype))
        params = np.concatenate([datagen.normal(seed, 1, C),
                                 datagen.uniform(seed, 2, C, -0.5, 0.5)]).astype(np.float32)
        return a, datagen.float_to(params, dtype).reshape(shape_b)
    if op == "BiasPReluBN":
        C = shape_b[1]
        a = mk("normal", dtype, shape_a, seed, 0)
        _sprinkle(a, specials(dtype))
        params = np.concatenate([
            datagen.normal(seed, 1, C), datagen.uniform(seed, 2, C, -0.5, 0.5),
            datagen.normal(seed, 3, C), datagen.normal(seed, 4, C), datagen.normal(seed, 5, C),
            datagen.uniform(seed, 6, C, 0.1, 2.0)]).astype(np.float32)
        return a, datagen.float_to(params, dtype).reshape(shape_b)
    if op == "Clip":
        if dtype in FLOATS:
            a = mk("normal", dtype, shape_a, seed, 0)
            a = (a.astype(np.float32) * 2).astype(a.dtype) if dtype == "float16" else a
            b = datagen.float_to(np.array([-1.0, 1.5], np.float32), dtype)
        else:
            a = mk("bits", dtype, shape_a, seed, 0)
            lo, hi = {"uint8": (20, 200), "uint32": (1000, 3000000000), "int8": (-50, 60),
                      "int16": (-1000, 20000), "uint16": (1000, 50000),
                      "uint64": (1000, (1 << 63) + 5)}.get(dtype, (-1000000, 2000000000))
            b = np.array([lo, hi], dtype=object).astype(datagen.STORAGE[dtype])
        return a, b
    if dtype == "bool":
        return mk("bool", dtype, shape_a, seed, 0), mk("bool", dtype, shape_b, seed, 1)
    if dtype in FLOATS:
        if op == "Mod":
            a = mk("uniform_zeros", dtype, shape_a, seed, 0, lo=-100, hi=100, pzero=0.01)
            b = mk("uniform_reject", dtype, shape_b, seed, 1, lo=-7, hi=7, min_abs=0.01)
            _sprinkle(a, datagen.make("bits", dtype, (64,), seed, 5))
            _sprinkle(b, specials(dtype))
        elif op == "Pow":
            na, nb = int(np.prod(shape_a)), int(np.prod(shape_b))
            af = datagen.uniform(seed, 0, na, -4.0, 6.0)
            bf = datagen.uniform(seed, 1, nb, -4.0, 4.0)
            bf[::3] = np.round(bf[::3])                        # integer exponents too
            a = datagen.float_to(af, dtype).reshape(shape_a)
            b = datagen.float_to(bf, dtype).reshape(shape_b)
            _sprinkle(a, specials(dtype))
        elif op == "PRelu":
            a = mk("normal", dtype, shape_a, seed, 0)
            b = mk("uniform", dtype, shape_b, seed, 1, lo=0.0, hi=0.3)
            _sprinkle(a, specials(dtype))
        else:
            a = mk("normal", dtype, shape_a, seed, 0)
            b = mk("normal", dtype, shape_b, seed, 1)
            if op in ("Equal", "Less", "Greater", "LessOrEqual", "GreaterOrEqual", "Max", "Min"):
                if a.shape == b.shape and a.size > 4:
                    b.reshape(-1)[::5] = a.reshape(-1)[::5]
            _sprinkle(a, specials(dtype))
            _sprinkle(b, specials(dtype)[::-1])
            if op in ("Max", "Min") and a.size > 1 and b.size > 1:
                # (+0, -0) and (-0, +0) as the first two elements of the two operands
                z = datagen.float_to(np.array([0.0, -0.0], np.float32), dtype)
                a.reshape(-1)[:2] = z
                b.reshape(-1)[:2] = z[::-1]
        return a, b
    # integers
    st = datagen.STORAGE[dtype]
    bits = 8 * np.dtype(st).itemsize
    if op == "BitShift":
        a = mk("bits", dtype, shape_a, seed, 0)
        b = mk("int_range", dtype, shape_b, seed, 1, lo=0, hi=bits - 1)
        return a, b
    if op == "Pow":
        a = mk("int_range", dtype, shape_a, seed, 0, lo=-9, hi=9)
        b = mk("int_range", dtype, shape_b, seed, 1, lo=-2, hi=40)
        return a, b
    small = {"int8": 100, "uint8": 200}.get(dtype, 1000)       # divisors within the type
    if op in ("Div", "Mod"):
        a = mk("bits", dtype, shape_a, seed, 0)
        lo = 0 if dtype.startswith("u") else -small
        b = mk("int_range", dtype, shape_b, seed, 1, lo=lo, hi=small, skip_zero=True)
        if dtype.startswith("u"):
            b[b == 0] = 1
        if b.size > 2 and dtype in ("int32", "int64"):
            b.reshape(-1)[1] = -1                              # INT_MIN / -1 path
        if a.size > 2 and dtype in ("int32", "int64"):
            a.reshape(-1)[0] = np.iinfo(st).min
        return a, b
    if op == "RDiv":                                           # B / A: A is the divisor
        lo = 0 if dtype.startswith("u") else -small
        a = mk("int_range", dtype, shape_a, seed, 0, lo=lo, hi=small, skip_zero=True)
        if dtype.startswith("u"):
            a[a == 0] = 1
        b = mk("bits", dtype, shape_b, seed, 1)
        if a.size > 0 and b.size > 0 and dtype in ("int32", "int64"):
            a.reshape(-1)[0] = -1                              # INT_MIN / -1 at output 0
            b.reshape(-1)[0] = np.iinfo(st).min
        return a, b
    if op == "PRelu":
        a = mk("bits", dtype, shape_a, seed, 0)
        b = mk("int_range", dtype, shape_b, seed, 1, lo=0, hi=5)
        return a, b
    a = mk("bits", dtype, shape_a, seed, 0)
    b = mk("bits", dtype, shape_b, seed, 1)
    if op in ("Equal", "Less", "Greater", "LessOrEqual", "GreaterOrEqual", "Max", "Min"):
        if a.shape == b.shape and a.size > 4:
            b.reshape(-1)[::4] = a.reshape(-1)[::4]
    return a, b


def _sprinkle(arr: np.ndarray, vals: np.ndarray):
    """Overwrite a spread of positions with special values (in place)."""
    flat = arr.reshape(-1)
    if flat.size == 0:
        return
    k = min(vals.size, max(1, flat.size // 7))
    pos = np.linspace(0, flat.size - 1, k).astype(np.int64)
    flat[pos] = vals[:k]
