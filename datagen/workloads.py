"""The benchmark workloads as seeded input recipes (no engine arithmetic here).

Each case is (name, op, dtype, attrs, shape_a, shape_b, make_a, make_b, family)
where make_a/make_b build the operand on the host.  Workload k uses seed k-1;
operand j of a workload uses stream seed*16 + j.

  1  Add fp32, A[2,3,4,5] + B[3,1,5], both U(-1,1)                       seed 0
  2  Mul fp32, A and B [2^28] ~ N(0,1); Div with B = |N(0,1)| + 0.5       seed 1
  3  bf16 x[8,64,256,256] ~ N(0,1): Add b[64,1,1] ~ U(-0.5,0.5),
     PRelu slope[64,1,1] ~ U(0,0.3), BatchNormalization with scale, bias,
     mean ~ N(0,1), var ~ U(0.1,2), eps 1e-5 (parameters stored in bf16);
     the fused BiasPRelu with bias ~ N(0,1), slope ~ U(0,0.3); the chain
     BiasPReluBN with the BiasPRelu then BatchNormalization parameters; the
     fused MulAdd x * s + y (residual scaling) with y ~ N(0,1) and s a
     scalar or per-channel [1,64,1,1] ~ U(0,0.3)                          seed 2
  4  Mod opset 28, A[4096,4096] against a scalar B and against B[4096,1]:
     fp32 fmod 0 and 1 with A ~ U(-100,100) holding 1% exact +-0 and
     B ~ U(-7,7) without |B| < 0.01; int32 fmod 0 with A ~ U[-2^31,2^31)
     and B ~ U[-1000,1000] without 0                                     seed 3
  5  Greater fp16 A[64,1,512,1] vs B[1,32,1,1024] ~ N(0,1) -> 1-byte BOOL
     [64,32,512,1024]; BitShift RIGHT uint32 A[2^26] raw bits by B[1] in
     [0,31]                                                               seed 4
Not from the pages:
  6  Add fp32 [2^24,3] ~ N(0,1) + [3] ~ U(-0.5,0.5) (channels-last)       seed 5
  7  general strided, short rows: Add fp32 [8192,1,5] + [1,4096,5] and
     Mul bf16 [16384,1,3] x [1,8192,3], all ~ N(0,1)                      seed 6
  8  general strided, a transposed view: Add fp32 A[8192,8192] + B and Mul
     bf16 the same, B read through element strides (1, 8192) from an
     [8192,8192] buffer (a transposed tensor), all ~ N(0,1)               seed 7
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable

import numpy as np

from . import float_to, make, normal, uniform


@dataclass
class Case:
    name: str
    op: str
    dtype: str
    attrs: dict
    shape_a: tuple
    shape_b: tuple
    make_a: Callable[[], np.ndarray]
    make_b: Callable[[], np.ndarray]
    family: str
    workload: int
    tags: list = field(default_factory=list)
    shape_c: tuple | None = None                 # three-input operators (MulAdd)
    make_c: Callable[[], np.ndarray] | None = None
    strides_b: tuple | None = None               # B a view of make_b()'s buffer


def _bn_params(seed: int, C: int, dtype: str) -> np.ndarray:
    p = np.concatenate([normal(seed, 3, C), normal(seed, 4, C), normal(seed, 5, C),
                        uniform(seed, 6, C, 0.1, 2.0)]).astype(np.float32)
    return float_to(p, dtype).reshape(4, C)


def cases(scale_log2: int = 0) -> list[Case]:
    """All benchmark cases; scale_log2 > 0 shrinks the large 1-D workloads by 2^scale."""
    n2 = 1 << max(28 - scale_log2, 10)
    n5 = 1 << max(26 - scale_log2, 10)
    out = []
    out.append(Case("add_f32_general", "Add", "float32", {}, (2, 3, 4, 5), (3, 1, 5),
                    lambda: make("uniform", "float32", (2, 3, 4, 5), 0, 0, lo=-1, hi=1),
                    lambda: make("uniform", "float32", (3, 1, 5), 0, 1, lo=-1, hi=1),
                    "general_strided", 1))
    out.append(Case("mul_f32_contiguous", "Mul", "float32", {}, (n2,), (n2,),
                    lambda: make("normal", "float32", (n2,), 1, 0),
                    lambda: make("normal", "float32", (n2,), 1, 1),
                    "contiguous", 2, ["headline"]))
    out.append(Case("div_f32_contiguous", "Div", "float32", {}, (n2,), (n2,),
                    lambda: make("normal", "float32", (n2,), 1, 0),
                    lambda: make("absnormal", "float32", (n2,), 1, 2, shift=0.5),
                    "contiguous", 2, ["headline"]))
    x = (8, 64, 256, 256)
    out.append(Case("add_bf16_per_channel", "Add", "bfloat16", {}, x, (64, 1, 1),
                    lambda: make("normal", "bfloat16", x, 2, 0),
                    lambda: make("uniform", "bfloat16", (64, 1, 1), 2, 1, lo=-0.5, hi=0.5),
                    "inner_vector_outer", 3))
    out.append(Case("prelu_bf16_per_channel", "PRelu", "bfloat16", {}, x, (64, 1, 1),
                    lambda: make("normal", "bfloat16", x, 2, 0),
                    lambda: make("uniform", "bfloat16", (64, 1, 1), 2, 2, lo=0.0, hi=0.3),
                    "inner_vector_outer", 3))
    out.append(Case("batchnorm_bf16_per_channel", "BatchNormalization", "bfloat16",
                    {"epsilon": 1e-5}, x, (4, 64),
                    lambda: make("normal", "bfloat16", x, 2, 0),
                    lambda: _bn_params(2, 64, "bfloat16"),
                    "inner_vector_outer", 3))
    out.append(Case("biasprelu_bf16_per_channel", "BiasPRelu", "bfloat16", {}, x, (2, 64),
                    lambda: make("normal", "bfloat16", x, 2, 0),
                    lambda: float_to(np.concatenate([normal(2, 1, 64),
                                                     uniform(2, 2, 64, 0.0, 0.3)])
                                     .astype(np.float32), "bfloat16").reshape(2, 64),
                    "inner_vector_outer", 3, ["fused"]))
    # the chain bias add -> PReLU -> BatchNormalization in one pass, with the
    # parameters of the BiasPRelu and BatchNormalization cases above
    out.append(Case("biasprelubn_bf16_per_channel", "BiasPReluBN", "bfloat16",
                    {"epsilon": 1e-5}, x, (6, 64),
                    lambda: make("normal", "bfloat16", x, 2, 0),
                    lambda: np.concatenate([
                        float_to(np.concatenate([normal(2, 1, 64), uniform(2, 2, 64, 0.0, 0.3)])
                                 .astype(np.float32), "bfloat16").reshape(2, 64),
                        _bn_params(2, 64, "bfloat16")]),
                    "inner_vector_outer", 3, ["fused"]))
    for name, sb, fam in (("muladd_bf16_residual_scale", (1,), "right_scalar"),
                          ("muladd_bf16_per_channel", (1, 64, 1, 1), "inner_vector_outer")):
        out.append(Case(name, "MulAdd", "bfloat16", {}, x, sb,
                        lambda: make("normal", "bfloat16", x, 2, 0),
                        (lambda sb=sb: make("uniform", "bfloat16", sb, 2, 3, lo=0.0, hi=0.3)),
                        fam, 3, ["fused"], shape_c=x,
                        make_c=lambda: make("normal", "bfloat16", x, 2, 4)))
    m = (4096, 4096)
    for fm in (0, 1):
        out.append(Case("mod_f32_fmod%d_scalar" % fm, "Mod", "float32", {"fmod": fm}, m, (),
                        lambda: make("uniform_zeros", "float32", m, 3, 0, lo=-100, hi=100,
                                     pzero=0.01),
                        lambda: make("uniform_reject", "float32", (), 3, 1, lo=-7, hi=7,
                                     min_abs=0.01),
                        "right_scalar", 4))
        out.append(Case("mod_f32_fmod%d_rows" % fm, "Mod", "float32", {"fmod": fm}, m,
                        (4096, 1),
                        lambda: make("uniform_zeros", "float32", m, 3, 0, lo=-100, hi=100,
                                     pzero=0.01),
                        lambda: make("uniform_reject", "float32", (4096, 1), 3, 2, lo=-7, hi=7,
                                     min_abs=0.01),
                        "repeated_block", 4))
    out.append(Case("mod_i32_fmod0_scalar", "Mod", "int32", {"fmod": 0}, m, (),
                    lambda: make("bits", "int32", m, 3, 3),
                    lambda: make("int_range", "int32", (), 3, 4, lo=-1000, hi=1000,
                                 skip_zero=True),
                    "right_scalar", 4))
    out.append(Case("mod_i32_fmod0_rows", "Mod", "int32", {"fmod": 0}, m, (4096, 1),
                    lambda: make("bits", "int32", m, 3, 3),
                    lambda: make("int_range", "int32", (4096, 1), 3, 5, lo=-1000, hi=1000,
                                 skip_zero=True),
                    "repeated_block", 4))
    out.append(Case("greater_f16_outer_broadcast", "Greater", "float16", {}, (64, 1, 512, 1),
                    (1, 32, 1, 1024),
                    lambda: make("normal", "float16", (64, 1, 512, 1), 4, 0),
                    lambda: make("normal", "float16", (1, 32, 1, 1024), 4, 1),
                    "inner_vector_outer", 5))
    out.append(Case("bitshift_u32_right_scalar", "BitShift", "uint32", {"direction": 1},
                    (n5,), (1,),
                    lambda: make("bits", "uint32", (n5,), 4, 2),
                    lambda: make("int_range", "uint32", (1,), 4, 3, lo=0, hi=31),
                    "right_scalar", 5))
    # not from the pages: a channels-last per-channel broadcast (NHWC image
    # data, 3 channels), whose rows are off the 16-byte pack width
    nhwc = (1 << max(24 - scale_log2, 8), 3)
    out.append(Case("add_f32_channels_last_c3", "Add", "float32", {}, nhwc, (3,),
                    lambda: make("normal", "float32", nhwc, 5, 0),
                    lambda: make("uniform", "float32", (3,), 5, 1, lo=-0.5, hi=0.5),
                    "repeated_block", 6, ["extra"]))
    # not from the pages: general-strided broadcasts with short rows, both
    # operands broadcast ([a, 1, k] against [1, b, k]), several times the L2
    # in output bytes: Add fp32 out [8192, 4096, 5] (671 MB) and Mul bf16
    # out [16384, 8192, 3] (805 MB)
    ga, gb = (1 << max(13 - scale_log2, 4), 1, 5), (1, 1 << max(12 - scale_log2, 4), 5)
    out.append(Case("add_f32_general_short_rows", "Add", "float32", {}, ga, gb,
                    lambda: make("normal", "float32", ga, 6, 0),
                    lambda: make("normal", "float32", gb, 6, 1),
                    "general_strided", 7, ["extra"]))
    ma, mb = (1 << max(14 - scale_log2, 4), 1, 3), (1, 1 << max(13 - scale_log2, 4), 3)
    out.append(Case("mul_bf16_general_short_rows", "Mul", "bfloat16", {}, ma, mb,
                    lambda: make("normal", "bfloat16", ma, 6, 2),
                    lambda: make("normal", "bfloat16", mb, 6, 3),
                    "general_strided", 7, ["extra"]))
    t = 1 << max(13 - scale_log2 // 2, 6)
    for name, op, dt, k in (("add_f32_transposed", "Add", "float32", 0),
                            ("mul_bf16_transposed", "Mul", "bfloat16", 2)):
        out.append(Case(name, op, dt, {}, (t, t), (t, t),
                        lambda dt=dt, k=k: make("normal", dt, (t, t), 7, k),
                        lambda dt=dt, k=k: make("normal", dt, (t * t,), 7, k + 1),
                        "general_strided", 8, ["extra"], strides_b=(1, t)))
    return out


def by_name(name: str, scale_log2: int = 0) -> Case:
    for c in cases(scale_log2):
        if c.name == name:
            return c
    raise KeyError(name)
