/*
 * ORACLE -- test infrastructure only.  Nothing in the product path links,
 * loads or calls this file; only the tests, the smoke check and the bench's
 * CPU-baseline leg do.
 *
 * A plain, single-threaded, deliberately slow statement of what the ONNX
 * broadcast binary elementwise engine computes.  For every requested output
 * element it decomposes the flat index over the FULL output shape, maps each
 * dimension to the two inputs (index 0 on a size-1 dimension), reads both
 * inputs, applies the operator and stores the result.  There is no
 * coalescing, no loop family, no vectorisation and no blocking.
 *
 * Sources followed (page title -- section):
 *  - "Binary Kernel Design" (onnx-light-cpu) -- "Operators and traversal":
 *    right-aligned broadcasting, empty dimensions doing no work, the Mod
 *    opset-28 sign rules, FLOAT16/BFLOAT16 through float conversion.
 *  - "Binary Kernel Design" -- "Compute, scheduling, and safety": validation of
 *    integer division, modulo and shifts; one byte per BOOL.
 *  - 0verkilll/onnx "ops" package docs -- BatchNormalizationOp (inference
 *    formula, channel axis 1), PReluOp (x >= 0 ? x : slope*x, slope broadcast
 *    to the data), ClipOp (optional min/max bounds), Add/Sub/Mul,
 *    ConvPReluOp (the per-output-channel bias add and PReLU fused into one
 *    pass: here without the convolution, as BiasPRelu), MulAddOp (y = a*b + c
 *    over three inputs broadcast together).  The bias -> PReLU ->
 *    BatchNormalization chain of one pass (BiasPReluBN) joins ConvPReluOp's
 *    epilogue to BatchNormalizationOp's formula.
 *  - ncnn operators.md -- batchnorm, bias, binaryop (operation types MAX,
 *    MIN, RSUB, RDIV; with_scalar), clip.
 * Where the pages are silent the plain reading is taken (IEEE-754 binary32
 * round-to-nearest-even arithmetic without contraction, two's-complement wrap
 * for integers, C99 pow/fmod semantics, ONNX type lists).
 *
 * Compile with -ffp-contract=off and without fast-math: every float operation
 * below must round on its own.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_pins.py
 * against numpy/Python library routines, closed forms, the sign tables that
 * follow from the Mod rules, and brute force over tiny shapes.  Integer Pow
 * with a negative exponent follows a reading the pages leave open (the exact
 * power truncated toward zero, as integer Div truncates), pinned by brute
 * force against exact rational arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---- the oracle's own operator and type codes (no shared header) ---- */
enum {
    OR_ADD = 0, OR_SUB, OR_MUL, OR_DIV, OR_MOD, OR_POW,
    OR_EQUAL, OR_LESS, OR_GREATER, OR_LESS_EQUAL, OR_GREATER_EQUAL,
    OR_AND, OR_OR, OR_XOR,
    OR_BITWISE_AND, OR_BITWISE_OR, OR_BITWISE_XOR,
    OR_BITSHIFT, OR_PRELU,
    OR_BATCHNORM, OR_CLIP,
    OR_MAX, OR_MIN, OR_RSUB, OR_RDIV,
    OR_BIAS_PRELU, OR_MULADD, OR_BIAS_PRELU_BN,
    OR_NUM_OPS
};
enum { OT_F32 = 0, OT_F16, OT_BF16, OT_I32, OT_I64, OT_U8, OT_U32, OT_BOOL,
       OT_I8, OT_I16, OT_U16, OT_U64, OT_F64, OT_NUM };

/* return codes */
enum { OR_OK = 0, OR_SHAPES = 1, OR_ARGS = 2, OR_TYPE = 3, OR_ATTR = 4 };
/* per-element validation findings, OR-ed into *status */
enum { OR_ST_DIV_BY_ZERO = 1u, OR_ST_SHIFT_RANGE = 2u };

#define OR_MAX_RANK 8

static int size_of(int t)
{
    switch (t) {
    case OT_F32: case OT_I32: case OT_U32: return 4;
    case OT_F16: case OT_BF16: case OT_I16: case OT_U16: return 2;
    case OT_I64: case OT_U64: case OT_F64: return 8;
    case OT_U8: case OT_BOOL: case OT_I8: return 1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* half and bfloat16 <-> float, written out from the IEEE-754 binary16 and   */
/* bfloat16 encodings.  Widening is exact; narrowing rounds to nearest, ties */
/* to even, overflows to infinity and keeps NaN a NaN.                       */
/* ------------------------------------------------------------------------ */
static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

float oracle_half_to_float(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t exp = (h >> 10) & 0x1F;
    uint32_t man = h & 0x3FF;
    if (exp == 0) {
        /* zero or subnormal: man * 2^-24, exact in binary32 */
        float v = (float)man * 5.9604644775390625e-08f;
        return sign ? -v : v;
    }
    if (exp == 31) return bits_to_f32(sign | 0x7F800000u | (man << 13));
    return bits_to_f32(sign | ((exp - 15 + 127) << 23) | (man << 13));
}

/* shift a positive integer right by s bits, rounding to nearest, ties to even */
static uint32_t shift_round_even(uint32_t m, int s)
{
    if (s <= 0) return m;
    if (s > 31) return 0;
    uint32_t q = m >> s;
    uint32_t rem = m & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1;
    return q;
}

uint16_t oracle_float_to_half(float f)
{
    uint32_t x = f32_to_bits(f);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return sign | 0x7E00u;           /* NaN stays NaN */
    if (ax == 0x7F800000u) return sign | 0x7C00u;          /* infinity */
    int e = (int)(ax >> 23) - 127;                          /* unbiased exponent */
    uint32_t m = (ax & 0x7FFFFFu) | (ax >= 0x00800000u ? 0x800000u : 0u);
    if (ax < 0x00800000u) e = -126;                          /* binary32 subnormal */
    if (e >= -14) {
        /* half normal range: keep 10 fraction bits, round the other 13 */
        uint32_t q = shift_round_even(m, 13);                /* 11-bit significand, may carry */
        int he = e + 15;
        if (q == 0x800u) { q = 0x400u; he += 1; }            /* carry into the exponent */
        if (he >= 31) return sign | 0x7C00u;                 /* overflow -> infinity */
        return sign | (uint16_t)((uint32_t)he << 10) | (uint16_t)(q & 0x3FFu);
    }
    /* half subnormal range: value = q * 2^-24, q = m * 2^(e-23) * 2^24 */
    int s = 13 + (-14 - e);                                  /* extra shift below 2^-14 */
    uint32_t q = shift_round_even(m, s);                     /* q <= 0x400 */
    return sign | (uint16_t)q;                               /* 0x400 is the smallest normal */
}

float oracle_bf16_to_float(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

uint16_t oracle_float_to_bf16(float f)
{
    uint32_t x = f32_to_bits(f);
    if ((x & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((x >> 16) | 0x0040u);   /* NaN */
    uint32_t hi = x >> 16;
    uint32_t lo = x & 0xFFFFu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1;   /* carries reach inf */
    return (uint16_t)hi;
}

/* ------------------------------------------------------------------------ */
/* element access                                                            */
/* ------------------------------------------------------------------------ */
/* binary32 and the 16-bit types computed through it; binary64 is separate */
static int is_float_type(int t) { return t == OT_F32 || t == OT_F16 || t == OT_BF16; }
static int is_fp(int t) { return is_float_type(t) || t == OT_F64; }

static double load_double(const void *p, int64_t i) { return ((const double *)p)[i]; }
static void store_double(void *p, int64_t i, double v) { ((double *)p)[i] = v; }
static int is_signed_int(int t)
{
    return t == OT_I32 || t == OT_I64 || t == OT_I8 || t == OT_I16;
}
static int is_int_type(int t)
{
    return is_signed_int(t) || t == OT_U8 || t == OT_U16 || t == OT_U32 || t == OT_U64;
}

static float load_float(const void *p, int t, int64_t i)
{
    if (t == OT_F32) return ((const float *)p)[i];
    if (t == OT_F16) return oracle_half_to_float(((const uint16_t *)p)[i]);
    return oracle_bf16_to_float(((const uint16_t *)p)[i]);
}

static void store_float(void *p, int t, int64_t i, float v)
{
    if (t == OT_F32) ((float *)p)[i] = v;
    else if (t == OT_F16) ((uint16_t *)p)[i] = oracle_float_to_half(v);
    else ((uint16_t *)p)[i] = oracle_float_to_bf16(v);
}

/* integers travel as their value in int64 (every unsigned type up to 32 bits
   fits); uint64 travels as its bit pattern and is compared and divided
   unsigned (see int_cmp and int_op); wrapped on store */
static int64_t load_int(const void *p, int t, int64_t i)
{
    switch (t) {
    case OT_I32: return ((const int32_t *)p)[i];
    case OT_I64: return ((const int64_t *)p)[i];
    case OT_U8: case OT_BOOL: return ((const uint8_t *)p)[i];
    case OT_U32: return ((const uint32_t *)p)[i];
    case OT_I8: return ((const int8_t *)p)[i];
    case OT_I16: return ((const int16_t *)p)[i];
    case OT_U16: return ((const uint16_t *)p)[i];
    case OT_U64: return (int64_t)((const uint64_t *)p)[i];
    }
    return 0;
}

static void store_int(void *p, int t, int64_t i, uint64_t v)
{
    switch (t) {
    case OT_I32: ((uint32_t *)p)[i] = (uint32_t)v; break;
    case OT_I64: ((uint64_t *)p)[i] = v; break;
    case OT_U8: case OT_BOOL: ((uint8_t *)p)[i] = (uint8_t)v; break;
    case OT_U32: ((uint32_t *)p)[i] = (uint32_t)v; break;
    case OT_I8: ((uint8_t *)p)[i] = (uint8_t)v; break;
    case OT_I16: case OT_U16: ((uint16_t *)p)[i] = (uint16_t)v; break;
    case OT_U64: ((uint64_t *)p)[i] = v; break;
    }
}

/* a < b on values of type t */
static int int_less(int t, int64_t a, int64_t b)
{
    return t == OT_U64 ? (uint64_t)a < (uint64_t)b : a < b;
}

static int bits_of(int t) { return 8 * size_of(t); }

/* reinterpret a wrapped bit pattern of width w as a signed value */
static int64_t as_signed(uint64_t v, int w)
{
    if (w == 64) return (int64_t)v;
    uint64_t m = (1ull << w) - 1ull;
    v &= m;
    if (v >> (w - 1)) return (int64_t)(v | ~m);
    return (int64_t)v;
}

/* ------------------------------------------------------------------------ */
/* descriptor rules (which operator accepts which type; attribute checks)    */
/* ------------------------------------------------------------------------ */
int oracle_type_allowed(int op, int t)
{
    switch (op) {
    case OR_ADD: case OR_SUB: case OR_MUL: case OR_DIV: case OR_MOD:
    case OR_LESS: case OR_GREATER: case OR_LESS_EQUAL: case OR_GREATER_EQUAL:
    case OR_CLIP: case OR_MAX: case OR_MIN: case OR_RSUB: case OR_RDIV: case OR_MULADD:
        return t != OT_BOOL && t >= 0 && t < OT_NUM;
    case OR_POW:
        return is_fp(t) || t == OT_I32 || t == OT_I64;
    case OR_EQUAL:
        return t >= 0 && t < OT_NUM;
    case OR_AND: case OR_OR: case OR_XOR:
        return t == OT_BOOL;
    case OR_BITWISE_AND: case OR_BITWISE_OR: case OR_BITWISE_XOR:
        return is_int_type(t);
    case OR_BITSHIFT:
        return t == OT_U8 || t == OT_U16 || t == OT_U32 || t == OT_U64;
    case OR_PRELU:
        return is_fp(t) || t == OT_I32 || t == OT_I64 || t == OT_U32 || t == OT_U64;
    case OR_BATCHNORM: case OR_BIAS_PRELU: case OR_BIAS_PRELU_BN:
        return is_fp(t);
    }
    return 0;
}

int oracle_output_type(int op, int t)
{
    if (op >= OR_EQUAL && op <= OR_XOR) return OT_BOOL;
    return t;
}

/*
 * Descriptor check.  Mod: opset 10..28; floating inputs need fmod=1 before
 * opset 28 ("Binary Kernel Design", Operators and traversal); fmod in {0,1}.
 * BitShift: direction 0 (LEFT) or 1 (RIGHT).
 */
int oracle_check_descriptor(int op, int opset, int fmod, int direction, int ta, int tb)
{
    if (op < 0 || op >= OR_NUM_OPS) return OR_ARGS;
    if (ta != tb) return OR_TYPE;
    if (!oracle_type_allowed(op, ta)) return OR_TYPE;
    if (op == OR_MOD) {
        if (opset < 10 || opset > 28) return OR_ATTR;
        if (fmod != 0 && fmod != 1) return OR_ATTR;
        if (is_fp(ta) && fmod == 0 && opset < 28) return OR_ATTR;
    }
    if (op == OR_BITSHIFT && direction != 0 && direction != 1) return OR_ATTR;
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* scalar semantics                                                          */
/* ------------------------------------------------------------------------ */
static float float_mod(float a, float b, int fmod_flag)
{
    float r = fmodf(a, b);                 /* exact truncated remainder, sign of a */
    if (fmod_flag) return r;
    /* floor remainder: a nonzero result takes the divisor's sign by adding b,
       an exact zero takes the divisor's sign */
    if (r == 0.0f) return copysignf(0.0f, b);
    if (signbit(r) != signbit(b)) r = r + b;
    return r;
}

/*
 * ncnn binaryop MAX / MIN (operation types 4 and 5).  The page names the
 * operations only; read as IEEE 754-2019 maximum / minimum: a NaN operand
 * gives NaN, and +0 counts as larger than -0.
 */
static float float_max(float a, float b)
{
    if (isnan(a) || isnan(b)) return a + b;            /* a NaN */
    if (a == b) return signbit(a) ? b : a;             /* equal, or +0 / -0 */
    return a > b ? a : b;
}

static float float_min(float a, float b)
{
    if (isnan(a) || isnan(b)) return a + b;
    if (a == b) return signbit(a) ? a : b;
    return a < b ? a : b;
}

static float float_op(int op, float a, float b, int fmod_flag)
{
    switch (op) {
    case OR_MAX: return float_max(a, b);
    case OR_MIN: return float_min(a, b);
    case OR_RSUB: return b - a;                         /* ncnn RSUB: B - A */
    case OR_RDIV: return b / a;                         /* ncnn RDIV: B / A */
    case OR_ADD: return a + b;
    case OR_SUB: return a - b;
    case OR_MUL: return a * b;
    case OR_DIV: return a / b;
    case OR_MOD: return float_mod(a, b, fmod_flag);
    case OR_POW: return (float)pow((double)a, (double)b);
    case OR_PRELU: return (a >= 0.0f) ? a : b * a;      /* slope * x below zero */
    }
    return 0.0f;
}

/* binary64 (DOUBLE): the same operators natively in binary64, each rounded
   on its own; Pow is C pow in binary64 */
static double double_max(double a, double b)
{
    if (isnan(a) || isnan(b)) return a + b;
    if (a == b) return signbit(a) ? b : a;
    return a > b ? a : b;
}

static double double_min(double a, double b)
{
    if (isnan(a) || isnan(b)) return a + b;
    if (a == b) return signbit(a) ? a : b;
    return a < b ? a : b;
}

static double double_op(int op, double a, double b, int fmod_flag)
{
    switch (op) {
    case OR_ADD: return a + b;
    case OR_SUB: return a - b;
    case OR_MUL: return a * b;
    case OR_DIV: return a / b;
    case OR_MOD: {
        double r = fmod(a, b);
        if (fmod_flag) return r;
        if (r == 0.0) return copysign(0.0, b);
        if (signbit(r) != signbit(b)) r = r + b;
        return r;
    }
    case OR_POW: return pow(a, b);
    case OR_PRELU: return (a >= 0.0) ? a : b * a;
    case OR_MAX: return double_max(a, b);
    case OR_MIN: return double_min(a, b);
    case OR_RSUB: return b - a;
    case OR_RDIV: return b / a;
    }
    return 0.0;
}

static int double_cmp(int op, double a, double b)
{
    switch (op) {
    case OR_EQUAL: return a == b;
    case OR_LESS: return a < b;
    case OR_GREATER: return a > b;
    case OR_LESS_EQUAL: return a <= b;
    case OR_GREATER_EQUAL: return a >= b;
    }
    return 0;
}

static int float_cmp(int op, float a, float b)
{
    switch (op) {
    case OR_EQUAL: return a == b;
    case OR_LESS: return a < b;
    case OR_GREATER: return a > b;
    case OR_LESS_EQUAL: return a <= b;
    case OR_GREATER_EQUAL: return a >= b;
    }
    return 0;
}

static int int_cmp(int op, int t, int64_t a, int64_t b)
{
    switch (op) {
    case OR_EQUAL: return a == b;
    case OR_LESS: return int_less(t, a, b);
    case OR_GREATER: return int_less(t, b, a);
    case OR_LESS_EQUAL: return !int_less(t, b, a);
    case OR_GREATER_EQUAL: return !int_less(t, a, b);
    }
    return 0;
}

/* integer operator on values a, b of type t; returns the wrapped bit pattern */
static uint64_t int_op(int op, int t, int64_t a, int64_t b, int fmod_flag, int direction,
                       uint32_t *status)
{
    int w = bits_of(t);
    int sgn = is_signed_int(t);
    uint64_t ua = (uint64_t)a, ub = (uint64_t)b;
    switch (op) {
    case OR_ADD: return ua + ub;
    case OR_SUB: return ua - ub;
    case OR_MUL: return ua * ub;
    case OR_DIV:
        if (b == 0) { *status |= OR_ST_DIV_BY_ZERO; return 0; }
        if (!sgn) return ua / ub;                              /* unsigned (uint64 too) */
        if (b == -1) return 0ull - ua;                         /* INT_MIN / -1 wraps */
        return (uint64_t)(a / b);                              /* C truncation */
    case OR_MOD: {
        if (b == 0) { *status |= OR_ST_DIV_BY_ZERO; return 0; }
        if (!sgn) return ua % ub;
        if (b == -1) return 0;
        int64_t r = a % b;                                     /* truncated, sign of a */
        if (!fmod_flag && r != 0 && ((r < 0) != (b < 0))) r += b;   /* floor: sign of b */
        return (uint64_t)r;
    }
    case OR_POW: {
        if (b < 0) {
            if (a == 0) { *status |= OR_ST_DIV_BY_ZERO; return 0; }
            if (a == 1) return 1;
            if (a == -1) return (b & 1) ? (uint64_t)-1 : 1;
            return 0;                                          /* trunc(1 / a^|b|) */
        }
        uint64_t result = 1, base = ua;
        uint64_t e = ub;
        while (e) {                                            /* square and multiply */
            if (e & 1u) result *= base;
            base *= base;
            e >>= 1;
        }
        return result;
    }
    case OR_BITWISE_AND: return ua & ub;
    case OR_BITWISE_OR: return ua | ub;
    case OR_BITWISE_XOR: return ua ^ ub;
    case OR_BITSHIFT: {
        uint64_t s = ub;
        if (s >= (uint64_t)w) { *status |= OR_ST_SHIFT_RANGE; return 0; }
        uint64_t mask = (w == 64) ? ~0ull : ((1ull << w) - 1ull);
        return direction == 0 ? ((ua << s) & mask) : ((ua & mask) >> s);
    }
    case OR_PRELU:                                             /* x >= 0 ? x : slope * x */
        return (!sgn || as_signed(ua, w) >= 0) ? ua : ub * ua;
    case OR_MAX: return int_less(t, b, a) ? ua : ub;          /* values, not bit patterns */
    case OR_MIN: return int_less(t, a, b) ? ua : ub;
    case OR_RSUB: return ub - ua;
    case OR_RDIV:                                              /* B / A, truncated */
        if (a == 0) { *status |= OR_ST_DIV_BY_ZERO; return 0; }
        if (!sgn) return ub / ua;
        if (a == -1) return 0ull - ub;
        return (uint64_t)(b / a);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* broadcasting                                                              */
/* ------------------------------------------------------------------------ */

/*
 * NumPy-style broadcast of two shapes: right-align, then each dimension pair
 * must be equal or contain a 1; the output takes the larger (0 pairs with 1
 * and gives 0).  Rank-0 shapes are scalars.
 */
int oracle_broadcast_shape(const int64_t *sa, int ra, const int64_t *sb, int rb,
                           int64_t *so, int *ro)
{
    if (ra < 0 || rb < 0 || ra > OR_MAX_RANK || rb > OR_MAX_RANK) return OR_ARGS;
    int r = ra > rb ? ra : rb;
    for (int d = 0; d < r; ++d) {
        int ia = d - (r - ra), ib = d - (r - rb);
        int64_t x = ia >= 0 ? sa[ia] : 1;
        int64_t y = ib >= 0 ? sb[ib] : 1;
        if (x < 0 || y < 0) return OR_ARGS;
        if (x == y) so[d] = x;
        else if (x == 1) so[d] = y;
        else if (y == 1) so[d] = x;
        else return OR_SHAPES;
    }
    *ro = r;
    return OR_OK;
}

/* dense row-major strides of `shape` right-aligned into rank r; 0 on size-1 dims */
static void aligned_strides(const int64_t *shape, int rank, int r, int64_t *stride)
{
    int64_t s = 1;
    for (int d = r - 1; d >= 0; --d) {
        int i = d - (r - rank);
        int64_t n = i >= 0 ? shape[i] : 1;
        stride[d] = (n == 1) ? 0 : s;
        s *= n;
    }
}

static int64_t numel(const int64_t *shape, int rank)
{
    int64_t n = 1;
    for (int d = 0; d < rank; ++d) n *= shape[d];
    return n;
}

/* element offsets into A and B of flat output index f (full multi-index) */
static void offsets_of(int64_t f, const int64_t *so, int r, const int64_t *sta,
                       const int64_t *stb, int64_t *oa, int64_t *ob)
{
    int64_t a = 0, b = 0;
    for (int d = r - 1; d >= 0; --d) {
        int64_t idx = f % so[d];
        f /= so[d];
        a += idx * sta[d];
        b += idx * stb[d];
    }
    *oa = a;
    *ob = b;
}

/* channel index (axis 1 of the output) of flat output index f */
static int64_t channel_of(int64_t f, const int64_t *so, int r)
{
    for (int d = r - 1; d > 1; --d) f /= so[d];
    return f % so[1];
}

/* exposed for the planner tests: A and B offsets of each listed output index */
int oracle_offsets(const int64_t *sa, int ra, const int64_t *sb, int rb, const int64_t *idx,
                   int64_t n, int64_t *oa, int64_t *ob)
{
    int64_t so[OR_MAX_RANK], sta[OR_MAX_RANK], stb[OR_MAX_RANK];
    int r;
    int rc = oracle_broadcast_shape(sa, ra, sb, rb, so, &r);
    if (rc) return rc;
    aligned_strides(sa, ra, r, sta);
    aligned_strides(sb, rb, r, stb);
    for (int64_t i = 0; i < n; ++i) offsets_of(idx[i], so, r, sta, stb, &oa[i], &ob[i]);
    return OR_OK;
}

/*
 * Evaluate output elements at the flat indices idx[0..n) (idx == NULL means
 * every element 0..numel-1, in order) and store them densely in out.
 *
 * Operands:
 *  - ordinary ops: A and B of types ta == tb, broadcast against each other;
 *  - PRelu: B (slope) must broadcast to A's shape, out shape == A shape; a
 *    1-D slope of C > 1 elements on data of rank >= 2 is per channel (axis 1;
 *    see prelu_slope_shape);
 *  - BatchNormalization (inference): A = x [N, C, ...] (rank >= 2), B = [4, C]
 *    holding scale, bias, mean, var rows; per element, in binary32 and in the
 *    order written, y = (x - mean) / sqrt(var + eps) * scale + bias;
 *  - Clip: B = [2] holding {min, max}; has_min / has_max say which bound
 *    applies; y = x, then raised to min if below it, then lowered to max if
 *    above it;
 *  - BiasPRelu: A = x [N, C, ...] (rank >= 2), B = [2, C] holding bias and
 *    slope rows; t = x + bias, then y = t when t >= 0 else slope * t, in
 *    binary32, rounded once to x's type;
 *  - BiasPReluBN: the per-channel chain bias add -> PReLU -> inference
 *    BatchNormalization in one pass.  A = x [N, C, ...] (rank >= 2), B = [6, C]
 *    holding bias, slope, scale, bn_bias, mean, var rows; t = x + bias;
 *    t = t >= 0 ? t : slope * t; y = (t - mean) / sqrt(var + eps) * scale +
 *    bn_bias; every step in binary32 in the order written, one rounding to
 *    x's type at the end (no rounding to x's type between the three).
 * Out shape: see oracle_output_shape.
 */
/*
 * PRelu's slope as it broadcasts (0verkilll/onnx ops, PReluOp: the slope is
 * broadcast against the data across the channel dimension; a scalar, a 1-D
 * [C], or a shape whose product is C with 1 everywhere but the channel axis
 * are the per-channel forms).  A 1-D slope of more than one element on data
 * of rank >= 2 is indexed by the channel, axis 1: it is read as the shape
 * [C, 1, ..., 1] of rank ra - 1, which right-aligns onto axis 1.  (ONNX's own
 * PRelu right-aligns a 1-D slope onto the last axis; the page's per-channel
 * reading is followed.)  Every other slope shape keeps its own shape and
 * broadcasts right-aligned.  Writes the shape into lb, its rank into *rlb.
 */
static void prelu_slope_shape(const int64_t *sa, int ra, const int64_t *sb, int rb,
                              int64_t *lb, int *rlb)
{
    (void)sa;
    if (ra >= 2 && rb == 1 && sb[0] != 1) {
        lb[0] = sb[0];
        for (int d = 1; d < ra - 1; ++d) lb[d] = 1;
        *rlb = ra - 1;
        return;
    }
    for (int d = 0; d < rb; ++d) lb[d] = sb[d];
    *rlb = rb;
}

int oracle_output_shape(int op, const int64_t *sa, int ra, const int64_t *sb, int rb,
                        int64_t *so, int *ro)
{
    int64_t lb[OR_MAX_RANK];
    if (op == OR_PRELU && rb >= 0 && rb <= OR_MAX_RANK && ra >= 0 && ra <= OR_MAX_RANK) {
        prelu_slope_shape(sa, ra, sb, rb, lb, &rb);
        sb = lb;
    }
    if (op == OR_BATCHNORM || op == OR_BIAS_PRELU || op == OR_BIAS_PRELU_BN) {
        const int64_t rows = op == OR_BATCHNORM ? 4 : op == OR_BIAS_PRELU ? 2 : 6;
        if (ra < 2 || rb != 2 || sb[0] != rows || sb[1] != sa[1]) return OR_SHAPES;
        for (int d = 0; d < ra; ++d) so[d] = sa[d];
        *ro = ra;
        return OR_OK;
    }
    if (op == OR_CLIP) {
        if (!(rb == 1 && sb[0] == 2)) return OR_SHAPES;
        for (int d = 0; d < ra; ++d) so[d] = sa[d];
        *ro = ra;
        return OR_OK;
    }
    int rc = oracle_broadcast_shape(sa, ra, sb, rb, so, ro);
    if (rc) return rc;
    if (op == OR_PRELU) {
        /* slope broadcasts one way only: the output keeps the data's shape */
        if (*ro != ra) return OR_SHAPES;
        for (int d = 0; d < ra; ++d)
            if (so[d] != sa[d]) return OR_SHAPES;
    }
    return OR_OK;
}

/* A parameter of type tp, widened to binary64 (exactly). */
static double load_param(const void *B, int tp, int64_t i)
{
    return tp == OT_F64 ? load_double(B, i) : (double)load_float(B, tp, i);
}

/* The evaluation behind oracle_eval and oracle_eval_params: tp is the element
   type of BatchNormalization's, BiasPRelu's and BiasPReluBN's parameter block
   (t for every other operator). */
static int eval2(int op, int t, int tp, int fmod_flag, int direction, float eps, int has_min,
                 int has_max, const int64_t *sa, int ra, const int64_t *sb, int rb,
                 const void *A, const void *B, void *out,
                 const int64_t *idx, int64_t n_idx, uint32_t *status)
{
    int64_t so[OR_MAX_RANK], sta[OR_MAX_RANK], stb[OR_MAX_RANK], lb[OR_MAX_RANK];
    int r;
    *status = 0;
    if (op < 0 || op >= OR_NUM_OPS || !oracle_type_allowed(op, t)) return OR_TYPE;
    if (op == OR_MULADD) return OR_ARGS;              /* three inputs: oracle_eval3 */
    if (ra < 0 || rb < 0 || ra > OR_MAX_RANK || rb > OR_MAX_RANK) return OR_ARGS;
    if (op == OR_PRELU) {                             /* a 1-D slope is per channel */
        prelu_slope_shape(sa, ra, sb, rb, lb, &rb);
        sb = lb;
    }
    int rc = oracle_output_shape(op, sa, ra, sb, rb, so, &r);
    if (rc) return rc;
    int64_t total = numel(so, r);
    int64_t count = idx ? n_idx : total;
    int to = oracle_output_type(op, t);
    aligned_strides(sa, ra, r, sta);
    if (op != OR_BATCHNORM && op != OR_CLIP && op != OR_BIAS_PRELU && op != OR_BIAS_PRELU_BN)
        aligned_strides(sb, rb, r, stb);
    else
        for (int d = 0; d < r; ++d) stb[d] = 0;

    for (int64_t k = 0; k < count; ++k) {
        int64_t f = idx ? idx[k] : k;
        if (f < 0 || f >= total) return OR_ARGS;
        int64_t oa, ob;
        offsets_of(f, so, r, sta, stb, &oa, &ob);

        if (op == OR_BATCHNORM && t == OT_F64) {     /* the same formula in binary64 */
            int64_t C = sb[1], c = channel_of(f, so, r);
            double x = load_double(A, oa);
            double scale = load_param(B, tp, 0 * C + c), bias = load_param(B, tp, 1 * C + c);
            double mean = load_param(B, tp, 2 * C + c), var = load_param(B, tp, 3 * C + c);
            store_double(out, k, (x - mean) / sqrt(var + (double)eps) * scale + bias);
            continue;
        }
        if (op == OR_BIAS_PRELU && t == OT_F64) {
            int64_t C = sb[1], c = channel_of(f, so, r);
            double y = load_double(A, oa) + load_param(B, tp, c);
            if (!(y >= 0.0)) y = load_param(B, tp, C + c) * y;
            store_double(out, k, y);
            continue;
        }
        if (op == OR_BIAS_PRELU_BN && t == OT_F64) {
            int64_t C = sb[1], c = channel_of(f, so, r);
            double y = load_double(A, oa) + load_param(B, tp, c);
            if (!(y >= 0.0)) y = load_param(B, tp, C + c) * y;
            double scale = load_param(B, tp, 2 * C + c), bn_bias = load_param(B, tp, 3 * C + c);
            double mean = load_param(B, tp, 4 * C + c), var = load_param(B, tp, 5 * C + c);
            store_double(out, k, (y - mean) / sqrt(var + (double)eps) * scale + bn_bias);
            continue;
        }
        if (op == OR_CLIP && t == OT_F64) {
            double y = load_double(A, oa);
            if (has_min) { double lo = load_double(B, 0); if (y < lo) y = lo; }
            if (has_max) { double hi = load_double(B, 1); if (y > hi) y = hi; }
            store_double(out, k, y);
            continue;
        }
        if (op == OR_BATCHNORM) {
            int64_t C = sb[1], c = channel_of(f, so, r);
            float x = load_float(A, t, oa);
            float scale = load_float(B, tp, 0 * C + c);
            float bias = load_float(B, tp, 1 * C + c);
            float mean = load_float(B, tp, 2 * C + c);
            float var = load_float(B, tp, 3 * C + c);
            float y = (x - mean) / sqrtf(var + eps) * scale + bias;
            store_float(out, t, k, y);
            continue;
        }
        if (op == OR_BIAS_PRELU) {
            /* y = x + bias[c]; y >= 0 ? y : slope[c] * y; binary32 steps, one
               rounding to x's type at the end */
            int64_t C = sb[1], c = channel_of(f, so, r);
            float y = load_float(A, t, oa) + load_float(B, tp, c);
            if (!(y >= 0.0f)) y = load_float(B, tp, C + c) * y;
            store_float(out, t, k, y);
            continue;
        }
        if (op == OR_BIAS_PRELU_BN) {
            /* bias add, PReLU, then the BatchNormalization formula, binary32
               steps in the order written; one rounding to x's type */
            int64_t C = sb[1], c = channel_of(f, so, r);
            float y = load_float(A, t, oa) + load_float(B, tp, c);
            if (!(y >= 0.0f)) y = load_float(B, tp, C + c) * y;
            float scale = load_float(B, tp, 2 * C + c);
            float bn_bias = load_float(B, tp, 3 * C + c);
            float mean = load_float(B, tp, 4 * C + c);
            float var = load_float(B, tp, 5 * C + c);
            y = (y - mean) / sqrtf(var + eps) * scale + bn_bias;
            store_float(out, t, k, y);
            continue;
        }
        if (op == OR_CLIP) {
            if (is_float_type(t)) {
                float y = load_float(A, t, oa);
                if (has_min) { float lo = load_float(B, t, 0); if (y < lo) y = lo; }
                if (has_max) { float hi = load_float(B, t, 1); if (y > hi) y = hi; }
                store_float(out, t, k, y);
            } else {
                int64_t y = load_int(A, t, oa);
                if (has_min) { int64_t lo = load_int(B, t, 0); if (int_less(t, y, lo)) y = lo; }
                if (has_max) { int64_t hi = load_int(B, t, 1); if (int_less(t, hi, y)) y = hi; }
                store_int(out, t, k, (uint64_t)y);
            }
            continue;
        }
        if (to == OT_BOOL) {
            int v;
            if (op == OR_AND || op == OR_OR || op == OR_XOR) {
                int x = load_int(A, t, oa) != 0, y = load_int(B, t, ob) != 0;
                v = op == OR_AND ? (x && y) : op == OR_OR ? (x || y) : (x != y);
            } else if (t == OT_F64) {
                v = double_cmp(op, load_double(A, oa), load_double(B, ob));
            } else if (is_float_type(t)) {
                v = float_cmp(op, load_float(A, t, oa), load_float(B, t, ob));
            } else if (t == OT_BOOL) {
                v = int_cmp(op, t, load_int(A, t, oa) != 0, load_int(B, t, ob) != 0);
            } else {
                v = int_cmp(op, t, load_int(A, t, oa), load_int(B, t, ob));
            }
            ((uint8_t *)out)[k] = (uint8_t)(v ? 1 : 0);
            continue;
        }
        if (t == OT_F64) {
            store_double(out, k, double_op(op, load_double(A, oa), load_double(B, ob), fmod_flag));
        } else if (is_float_type(t)) {
            float y = float_op(op, load_float(A, t, oa), load_float(B, t, ob), fmod_flag);
            store_float(out, t, k, y);
        } else {
            uint64_t y = int_op(op, t, load_int(A, t, oa), load_int(B, t, ob), fmod_flag,
                                direction, status);
            store_int(out, t, k, y);
        }
    }
    return OR_OK;
}

int oracle_eval(int op, int t, int fmod_flag, int direction, float eps, int has_min, int has_max,
                const int64_t *sa, int ra, const int64_t *sb, int rb,
                const void *A, const void *B, void *out,
                const int64_t *idx, int64_t n_idx, uint32_t *status)
{
    return eval2(op, t, t, fmod_flag, direction, eps, has_min, has_max, sa, ra, sb, rb, A, B, out,
                 idx, n_idx, status);
}

/*
 * BatchNormalization, BiasPRelu and BiasPReluBN with the parameter block in
 * binary32 while x is fp16, bf16 or binary64 (the block is "in x's dtype or
 * fp32").  Reading: each parameter enters the compute type as it is -- exactly,
 * since binary32 widens exactly into binary32 and binary64 -- so the result is
 * the same-type formula with the parameters not first rounded to x's type.
 * tp == t is the same-type operator.  Other operators or types: OR_TYPE.
 */
int oracle_eval_params(int op, int t, int tp, float eps, const int64_t *sa, int ra,
                       const int64_t *sb, int rb, const void *A, const void *B, void *out,
                       const int64_t *idx, int64_t n_idx, uint32_t *status)
{
    *status = 0;
    if (op != OR_BATCHNORM && op != OR_BIAS_PRELU && op != OR_BIAS_PRELU_BN) return OR_TYPE;
    if (tp != t && !(tp == OT_F32 && (t == OT_F16 || t == OT_BF16 || t == OT_F64)))
        return OR_TYPE;
    return eval2(op, t, tp, 0, 0, eps, 1, 1, sa, ra, sb, rb, A, B, out, idx, n_idx, status);
}

/*
 * Pow with an exponent of another type ("Binary Kernel Design", Compute,
 * scheduling, and safety: legal signatures other than the same-type ones run
 * through typed scalar adapters; ONNX Pow takes base T and exponent T1).
 * Base types: the Pow types; exponent types: every non-BOOL type.  Reading:
 *  - floating base: the same-type floating Pow with the exponent converted to
 *    binary64 (exact for the 16- and 32-bit types; int64 above 2^53 rounds);
 *  - integer base, integer exponent: the same-type integer Pow (exponent as a
 *    64-bit value);
 *  - integer base, floating exponent: pow in binary64, truncated toward zero
 *    into the base type, saturating at its bounds; NaN gives 0; no status.
 * Output type: the base's.  Same broadcasting and element-by-element
 * evaluation as oracle_eval.
 */
static double exponent_as_double(const void *B, int tb, int64_t i)
{
    if (tb == OT_F64) return load_double(B, i);
    if (is_float_type(tb)) return (double)load_float(B, tb, i);
    if (tb == OT_U64) return (double)(uint64_t)load_int(B, tb, i);
    return (double)load_int(B, tb, i);
}

int oracle_eval_pow_mixed(int ta, int tb, const int64_t *sa, int ra, const int64_t *sb, int rb,
                          const void *A, const void *B, void *out, const int64_t *idx,
                          int64_t n_idx, uint32_t *status)
{
    int64_t so[OR_MAX_RANK], sta[OR_MAX_RANK], stb[OR_MAX_RANK];
    int r;
    *status = 0;
    if (!oracle_type_allowed(OR_POW, ta) || tb == OT_BOOL || tb < 0 || tb >= OT_NUM)
        return OR_TYPE;
    int rc = oracle_broadcast_shape(sa, ra, sb, rb, so, &r);
    if (rc) return rc;
    aligned_strides(sa, ra, r, sta);
    aligned_strides(sb, rb, r, stb);
    int64_t total = numel(so, r);
    int64_t count = idx ? n_idx : total;
    for (int64_t k = 0; k < count; ++k) {
        int64_t f = idx ? idx[k] : k;
        if (f < 0 || f >= total) return OR_ARGS;
        int64_t oa, ob;
        offsets_of(f, so, r, sta, stb, &oa, &ob);
        if (ta == OT_F64) {
            store_double(out, k, pow(load_double(A, oa), exponent_as_double(B, tb, ob)));
        } else if (is_float_type(ta)) {
            double x = (double)load_float(A, ta, oa);
            store_float(out, ta, k, (float)pow(x, exponent_as_double(B, tb, ob)));
        } else if (!is_fp(tb)) {
            int64_t e = load_int(B, tb, ob);
            if (tb == OT_U64 && e < 0) {                       /* an exponent of 2^63 or more */
                uint64_t result = 1, base = (uint64_t)load_int(A, ta, oa), k2 = (uint64_t)e;
                while (k2) {
                    if (k2 & 1u) result *= base;
                    base *= base;
                    k2 >>= 1;
                }
                store_int(out, ta, k, result);
            } else {
                store_int(out, ta, k, int_op(OR_POW, ta, load_int(A, ta, oa), e, 0, 0, status));
            }
        } else {
            double y = pow((double)load_int(A, ta, oa), exponent_as_double(B, tb, ob));
            int64_t v;
            if (isnan(y)) v = 0;
            else if (ta == OT_I32) v = y >= 2147483647.0 ? 2147483647 :
                                       y <= -2147483648.0 ? -2147483647 - 1 : (int64_t)y;
            else v = y >= 9223372036854775807.0 ? INT64_MAX :
                     y <= -9223372036854775808.0 ? INT64_MIN : (int64_t)y;
            store_int(out, ta, k, (uint64_t)v);
        }
    }
    return OR_OK;
}

/*
 * MulAdd (0verkilll/onnx ops, MulAddOp): y = (a * b) + c.  The shapes follow
 * the unfused pair: the product has shape broadcast(A, B) and the output
 * broadcast(broadcast(A, B), C).  Each output element is computed from its full
 * multi-index: a binary32 product and a binary32 sum, each rounded on its own,
 * then one rounding to a 16-bit type; integers wrap.  Elements at the flat
 * indices idx[0..n) (all when idx == NULL) are stored densely in out.
 */
int oracle_eval3(int op, int t, const int64_t *sa, int ra, const int64_t *sb, int rb,
                 const int64_t *sc, int rc, const void *A, const void *B, const void *C,
                 void *out, const int64_t *idx, int64_t n_idx)
{
    int64_t sab[OR_MAX_RANK], so[OR_MAX_RANK];
    int64_t sta[OR_MAX_RANK], stb[OR_MAX_RANK], stc[OR_MAX_RANK];
    int rab, r;
    if (op != OR_MULADD || !oracle_type_allowed(op, t)) return OR_TYPE;
    int rcode = oracle_broadcast_shape(sa, ra, sb, rb, sab, &rab);
    if (rcode) return rcode;
    rcode = oracle_broadcast_shape(sab, rab, sc, rc, so, &r);
    if (rcode) return rcode;
    aligned_strides(sa, ra, r, sta);
    aligned_strides(sb, rb, r, stb);
    aligned_strides(sc, rc, r, stc);
    int64_t total = numel(so, r);
    int64_t count = idx ? n_idx : total;
    for (int64_t k = 0; k < count; ++k) {
        int64_t f = idx ? idx[k] : k;
        if (f < 0 || f >= total) return OR_ARGS;
        int64_t oa, ob, oc, unused;
        offsets_of(f, so, r, sta, stb, &oa, &ob);
        offsets_of(f, so, r, stc, stc, &oc, &unused);
        if (t == OT_F64) {
            double p = load_double(A, oa) * load_double(B, ob);
            store_double(out, k, p + load_double(C, oc));
        } else if (is_float_type(t)) {
            float p = load_float(A, t, oa) * load_float(B, t, ob);
            float y = p + load_float(C, t, oc);
            store_float(out, t, k, y);
        } else {
            uint64_t y = (uint64_t)load_int(A, t, oa) * (uint64_t)load_int(B, t, ob) +
                         (uint64_t)load_int(C, t, oc);
            store_int(out, t, k, y);
        }
    }
    return OR_OK;
}

/* output shape of a three-input operator: broadcast(broadcast(A, B), C) */
int oracle_output_shape3(const int64_t *sa, int ra, const int64_t *sb, int rb,
                         const int64_t *sc, int rc, int64_t *so, int *ro)
{
    int64_t sab[OR_MAX_RANK];
    int rab;
    int rcode = oracle_broadcast_shape(sa, ra, sb, rb, sab, &rab);
    if (rcode) return rcode;
    return oracle_broadcast_shape(sab, rab, sc, rc, so, ro);
}

/* bulk forms of the conversions above, for the pin tests */
void oracle_f32_to_f16_n(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_float_to_half(x[i]);
}
void oracle_f32_to_bf16_n(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_float_to_bf16(x[i]);
}
void oracle_f16_to_f32_n(const uint16_t *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_half_to_float(x[i]);
}
void oracle_bf16_to_f32_n(const uint16_t *x, float *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16_to_float(x[i]);
}
