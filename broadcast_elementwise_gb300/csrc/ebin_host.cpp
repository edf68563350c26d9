// Host side of the ebin C ABI: descriptors, the broadcast planner, the
// 8-entry plan LRU, execution (alias check, family dispatch, launch) and the
// per-stream device status word.
//
// Follows "Binary Kernel Design" (onnx-light-cpu):
//   Prepared execution      -- descriptor built once per node; plans cached in
//                              a bounded 8-entry LRU keyed on a monotonic
//                              descriptor id, the types and both shapes; a miss
//                              builds and validates a fresh plan.
//   Operators and traversal -- right-align, zero strides for broadcast dims,
//                              drop unit dims, coalesce, pick a loop family;
//                              empty dims do no work.
//   Compute, scheduling, and safety -- validation before the math; one byte
//                              per BOOL; aliasing only when type and shape equal
//                              the output's.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <list>
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ebin.h"
#include "ebin_launch.h"
#include "ebin_plan.h"

using ebin::Fam;
using ebin::Geom;
using ebin::kMaxRank;

// ------------------------------------------------------------------ types
namespace {

int dt_class(ebin_dtype t) {
    switch (t) {
    case EBIN_FLOAT32: return ebin::DT_F32;
    case EBIN_FLOAT16: return ebin::DT_F16;
    case EBIN_BFLOAT16: return ebin::DT_BF16;
    case EBIN_INT32: return ebin::DT_I32;
    case EBIN_INT64: return ebin::DT_I64;
    case EBIN_UINT8: return ebin::DT_U8;
    case EBIN_UINT32: return ebin::DT_U32;
    case EBIN_BOOL: return ebin::DT_BOOL;
    case EBIN_INT8: return ebin::DT_I8;
    case EBIN_INT16: return ebin::DT_I16;
    case EBIN_UINT16: return ebin::DT_U16;
    case EBIN_UINT64: return ebin::DT_U64;
    case EBIN_DOUBLE: return ebin::DT_F64;
    }
    return -1;
}

// floating types (binary32 and the 16-bit types computed through it, and binary64)
bool is_float(ebin_dtype t) {
    return t == EBIN_FLOAT32 || t == EBIN_FLOAT16 || t == EBIN_BFLOAT16 || t == EBIN_DOUBLE;
}
bool is_int(ebin_dtype t) {
    return t == EBIN_INT32 || t == EBIN_INT64 || t == EBIN_UINT8 || t == EBIN_UINT32 ||
           t == EBIN_INT8 || t == EBIN_INT16 || t == EBIN_UINT16 || t == EBIN_UINT64;
}
bool is_signed_int(ebin_dtype t) {
    return t == EBIN_INT32 || t == EBIN_INT64 || t == EBIN_INT8 || t == EBIN_INT16;
}

// Type manifest: which element type each operator accepts (A and B share it).
bool type_legal(int op, ebin_dtype t) {
    if (dt_class(t) < 0) return false;
    switch (op) {
    case EBIN_OP_ADD: case EBIN_OP_SUB: case EBIN_OP_MUL: case EBIN_OP_DIV: case EBIN_OP_MOD:
    case EBIN_OP_LESS: case EBIN_OP_GREATER: case EBIN_OP_LESS_OR_EQUAL:
    case EBIN_OP_GREATER_OR_EQUAL: case EBIN_OP_CLIP:
    case EBIN_OP_MAX: case EBIN_OP_MIN: case EBIN_OP_RSUB: case EBIN_OP_RDIV:
    case EBIN_OP_MULADD:
        return is_float(t) || is_int(t);
    case EBIN_OP_POW: return is_float(t) || t == EBIN_INT32 || t == EBIN_INT64;  // ONNX Pow T
    case EBIN_OP_EQUAL: return true;
    case EBIN_OP_AND: case EBIN_OP_OR: case EBIN_OP_XOR: return t == EBIN_BOOL;
    case EBIN_OP_BITWISE_AND: case EBIN_OP_BITWISE_OR: case EBIN_OP_BITWISE_XOR: return is_int(t);
    case EBIN_OP_BITSHIFT:
        return t == EBIN_UINT8 || t == EBIN_UINT16 || t == EBIN_UINT32 || t == EBIN_UINT64;
    case EBIN_OP_PRELU:   // ONNX PRelu T
        return is_float(t) || t == EBIN_INT32 || t == EBIN_INT64 || t == EBIN_UINT32 ||
               t == EBIN_UINT64;
    case EBIN_OP_BATCHNORM: case EBIN_OP_BIAS_PRELU: case EBIN_OP_BIAS_PRELU_BN:
        return is_float(t);
    }
    return false;
}

ebin_dtype output_type(int op, ebin_dtype t) {
    return (op >= EBIN_OP_EQUAL && op <= EBIN_OP_XOR) ? EBIN_BOOL : t;
}

// Operators whose kernels can meet invalid elements and report them.
bool validates(int op, ebin_dtype t) {
    if ((op == EBIN_OP_DIV || op == EBIN_OP_MOD || op == EBIN_OP_RDIV) && is_int(t)) return true;
    if (op == EBIN_OP_POW && (t == EBIN_INT32 || t == EBIN_INT64)) return true;
    return op == EBIN_OP_BITSHIFT;
}

// Operators that accept ncnn binaryop's with_scalar (operators.md, binaryop:
// operation types ADD, SUB, MUL, DIV, MAX, MIN, POW, RSUB, RDIV).
bool scalar_attr_op(int op) {
    switch (op) {
    case EBIN_OP_ADD: case EBIN_OP_SUB: case EBIN_OP_MUL: case EBIN_OP_DIV: case EBIN_OP_POW:
    case EBIN_OP_MAX: case EBIN_OP_MIN: case EBIN_OP_RSUB: case EBIN_OP_RDIV:
        return true;
    }
    return false;
}

// B is an ordinary broadcast tensor (not the BN parameter block or Clip bounds).
bool plain_b(int op) {
    return op != EBIN_OP_BATCHNORM && op != EBIN_OP_CLIP && op != EBIN_OP_BIAS_PRELU &&
           op != EBIN_OP_BIAS_PRELU_BN;
}

// B is a per-channel parameter block of rows of C (BatchNormalization,
// BiasPRelu, BiasPReluBN).
bool param_block(int op) {
    return op == EBIN_OP_BATCHNORM || op == EBIN_OP_BIAS_PRELU || op == EBIN_OP_BIAS_PRELU_BN;
}

// Operators with three inputs (planned by ebin_plan_create3).
bool ternary(int op) { return op == EBIN_OP_MULADD; }

// Output keeps A's shape: B broadcasts one way.
bool one_way(int op) {
    return op == EBIN_OP_PRELU || op == EBIN_OP_BATCHNORM || op == EBIN_OP_CLIP ||
           op == EBIN_OP_BIAS_PRELU || op == EBIN_OP_BIAS_PRELU_BN;
}

std::atomic<uint64_t> g_next_id{1};
std::atomic<uint64_t> g_launches{0};

}  // namespace

struct ebin_descriptor_s {
    uint64_t id;
    int op;
    int opset;
    ebin_attrs attrs;
    ebin_dtype dt;
    ebin_dtype dt_b;       // B's type: dt, except for Pow with another exponent type
    ebin_dtype out_dt;
};


// ------------------------------------------------------------------ descriptor
extern "C" ebin_status ebin_descriptor_create(ebin_op op, int opset, const ebin_attrs *attrs,
                                              ebin_dtype dtype_a, ebin_dtype dtype_b,
                                              ebin_descriptor_t *out) {
    if (!out) return EBIN_ERR_INVALID_ARG;
    *out = nullptr;
    if ((int)op < 0 || (int)op >= EBIN_OP_COUNT) return EBIN_ERR_UNSUPPORTED_OP;
    ebin_attrs a{0, 0, EBIN_DEFAULT_EPSILON, 1, 1, 0, 0.0f};
    if (attrs) a = *attrs;
    // A and B share a type, except Pow's exponent, which may be any non-BOOL
    // type ("typed scalar adapters" for the other legal signatures), and the
    // parameter block of BatchNormalization, BiasPRelu and BiasPReluBN, which
    // may be binary32 beside a 16-bit or binary64 x
    if (!type_legal(op, dtype_a)) return EBIN_ERR_UNSUPPORTED_TYPE;
    if (dtype_a != dtype_b &&
        !(op == EBIN_OP_POW && dt_class(dtype_b) >= 0 && dtype_b != EBIN_BOOL) &&
        !(param_block(op) && dtype_b == EBIN_FLOAT32 && is_float(dtype_a)))
        return EBIN_ERR_UNSUPPORTED_TYPE;
    if (op == EBIN_OP_MOD) {
        // "Mod tracks schema version 28 while retaining minimum opset 10";
        // floating fmod=0 (floor remainder) only from opset 28.
        if (opset < 10 || opset > 28) return EBIN_ERR_INVALID_ATTR;
        if (a.fmod != 0 && a.fmod != 1) return EBIN_ERR_INVALID_ATTR;
        if (is_float(dtype_a) && a.fmod == 0 && opset < 28) return EBIN_ERR_INVALID_ATTR;
    }
    if (op == EBIN_OP_BITSHIFT && a.direction != 0 && a.direction != 1)
        return EBIN_ERR_INVALID_ATTR;
    if (a.with_scalar != 0 && a.with_scalar != 1) return EBIN_ERR_INVALID_ATTR;
    if (a.with_scalar && (!scalar_attr_op(op) || !is_float(dtype_a))) return EBIN_ERR_INVALID_ATTR;
    if (!a.with_scalar) a.scalar_b = 0.0f;
    auto *d = new ebin_descriptor_s;
    d->id = g_next_id.fetch_add(1);
    d->op = op;
    d->opset = opset;
    d->attrs = a;
    d->dt = dtype_a;
    d->dt_b = dtype_b;
    d->out_dt = output_type(op, dtype_a);
    *out = d;
    return EBIN_OK;
}

extern "C" ebin_status ebin_descriptor_output_dtype(ebin_descriptor_t desc, ebin_dtype *out) {
    if (!desc || !out) return EBIN_ERR_INVALID_ARG;
    *out = desc->out_dt;
    return EBIN_OK;
}

extern "C" ebin_status ebin_descriptor_id(ebin_descriptor_t desc, uint64_t *id) {
    if (!desc || !id) return EBIN_ERR_INVALID_ARG;
    *id = desc->id;
    return EBIN_OK;
}

// ------------------------------------------------------------------ planner
namespace {

// Element counts and view spans stay below 2^60, so that every element
// offset, byte offset and byte size (elements of at most 8 bytes) fits in
// int64_t; a larger shape is refused before any arithmetic on it.
constexpr int64_t kMaxElems = EBIN_MAX_ELEMENTS;

// Number of elements of a shape: 0 when an extent is 0 (whatever the others
// are), -1 when the count reaches kMaxElems.
int64_t elem_count(const int64_t *s, int r) {
    for (int i = 0; i < r; ++i)
        if (s[i] == 0) return 0;
    int64_t n = 1;
    for (int i = 0; i < r; ++i)
        if (__builtin_mul_overflow(n, s[i], &n) || n >= kMaxElems) return -1;
    return n;
}

// Loop family for a coalesced geometry, or EBIN_ERR_FAMILY through *ok when a
// forced family cannot traverse it.
int family_of(const ebin_plan_s &p, int forced, bool *ok) {
    *ok = true;
    if (p.numel == 0) return ebin::FAM_EMPTY;
    const Geom &g = p.g;
    const int r = g.rank;
    const int64_t G = 16 / (int64_t)ebin_dtype_size(p.dt);
    const int64_t inner = g.n[r - 1];
    const bool contig = r == 1 && g.sa[0] == 1 && g.sb[0] == 1;
    const bool left = r == 1 && g.sa[0] == 0 && g.sb[0] == 1 && plain_b(p.op);
    const bool right = r == 1 && g.sa[0] == 1 && g.sb[0] == 0;
    const int64_t ia = g.sa[r - 1], ib = g.sb[r - 1];
    // an input read in 16-byte packs along the rows needs every row to start on
    // a pack boundary: its outer strides are multiples of G (always true of
    // dense inputs; strided views may break it)
    bool rows_aligned = true;
    for (int i = 0; i + 1 < r; ++i)
        rows_aligned = rows_aligned && (ia != 1 || g.sa[i] % G == 0) &&
                       (ib != 1 || g.sb[i] % G == 0);
    // REPEATED_BLOCK: one input dense, the other a row block reused (0,1) or
    // one value per row (1,0), any row length (rows that are not a whole
    // number of 16-byte packs run the periodic flat kernel)
    bool block = false;
    if (r == 2) {
        const bool a_dense = g.sa[0] == inner && g.sa[1] == 1;
        const bool b_dense = g.sb[0] == inner && g.sb[1] == 1;
        auto bcast = [](const int64_t *s) {
            return (s[0] == 1 && s[1] == 0) || (s[0] == 0 && s[1] == 1);
        };
        block = (a_dense && bcast(g.sb)) || (b_dense && bcast(g.sa) && plain_b(p.op));
    }
    const bool inner_ok = inner % G == 0 && (ia == 0 || ia == 1) && (ib == 0 || ib == 1) &&
                          (ia == 1 || ib == 1) && (ia == 1 || plain_b(p.op)) && rows_aligned;
    switch (forced) {
    case EBIN_FAMILY_AUTO:
        if (contig) return ebin::FAM_CONTIGUOUS;
        if (left) return ebin::FAM_LEFT_SCALAR;
        if (right) return ebin::FAM_RIGHT_SCALAR;
        if (block) return ebin::FAM_REPEATED_BLOCK;
        if (inner_ok && inner >= 64) return ebin::FAM_INNER_VECTOR_OUTER;
        return ebin::FAM_GENERAL_STRIDED;
    case EBIN_FAMILY_CONTIGUOUS: *ok = contig; return forced;
    case EBIN_FAMILY_LEFT_SCALAR: *ok = left; return forced;
    case EBIN_FAMILY_RIGHT_SCALAR: *ok = right; return forced;
    case EBIN_FAMILY_REPEATED_BLOCK: *ok = block; return forced;
    case EBIN_FAMILY_INNER_VECTOR_OUTER: *ok = inner_ok; return forced;
    case EBIN_FAMILY_GENERAL_STRIDED: return forced;
    default: *ok = false; return forced;
    }
}

// Element strides of a view, or nullptr when they are the dense row-major ones
// (dims of extent 1 or 0 place no constraint).  Negative strides: *bad.
const int64_t *view_strides(const int64_t *shape, const int64_t *st, int rank, bool *bad) {
    *bad = false;
    if (!st) return nullptr;
    bool dense = true;
    int64_t acc = 1;
    for (int i = rank - 1; i >= 0; --i) {
        if (st[i] < 0) *bad = true;
        if (shape[i] > 1 && st[i] != acc) dense = false;
        // saturates: a shape this large is refused by its element count
        if (__builtin_mul_overflow(acc, shape[i], &acc)) acc = INT64_MAX;
    }
    return dense ? nullptr : st;
}

// Storage extent of a view in elements: largest offset + 1 (0 when empty, -1
// when it reaches kMaxElems).
int64_t view_span(const int64_t *shape, const int64_t *st, int rank) {
    for (int i = 0; i < rank; ++i)
        if (shape[i] == 0) return 0;
    int64_t span = 1;
    for (int i = 0; i < rank; ++i) {
        int64_t t;
        if (__builtin_mul_overflow(shape[i] - 1, st[i], &t) ||
            __builtin_add_overflow(span, t, &span) || span >= kMaxElems)
            return -1;
    }
    return span;
}

// The traversal of a plan without output elements: nothing is read, so no
// stride is formed (an empty input's extents may overflow any product).
Geom empty_geometry() {
    Geom g{};
    g.rank = 1;
    return g;
}

// Steps 2-4 of planning a non-empty two-input broadcast: element strides
// (dense, or the view's ta / tb), zero on broadcast dims; output dims of extent
// 1 dropped; adjacent dims merged where both inputs continue across them.
// so: output shape; xa / xb: each input right-aligned to rank r (rank ra / rb
// before alignment).  Every product stays below the element-count bound.
Geom coalesce2(const int64_t *so, const int64_t *xa, const int64_t *xb, int r, int ra, int rb,
               const int64_t *ta, const int64_t *tb) {
    int64_t st_a[kMaxRank], st_b[kMaxRank];
    int64_t acc_a = 1, acc_b = 1;
    for (int i = r - 1; i >= 0; --i) {
        const int ja = i - (r - ra), jb = i - (r - rb);
        st_a[i] = xa[i] == 1 ? 0 : (ta ? ta[ja] : acc_a);
        st_b[i] = xb[i] == 1 ? 0 : (tb ? tb[jb] : acc_b);
        acc_a *= xa[i];
        acc_b *= xb[i];
    }
    Geom g{};
    int k = 0;
    for (int i = 0; i < r; ++i) {
        if (so[i] == 1) continue;
        if (k > 0 && g.sa[k - 1] == st_a[i] * so[i] && g.sb[k - 1] == st_b[i] * so[i]) {
            // the previous (outer) dim continues this one: fold it in
            g.n[k - 1] *= so[i];
            g.sa[k - 1] = st_a[i];
            g.sb[k - 1] = st_b[i];
            continue;
        }
        g.n[k] = so[i];
        g.sa[k] = st_a[i];
        g.sb[k] = st_b[i];
        ++k;
    }
    if (k == 0) {  // a single element
        g.n[0] = 1;
        g.sa[0] = 1;
        g.sb[0] = 1;
        k = 1;
    }
    g.rank = k;
    return g;
}

ebin_status build_plan(const ebin_descriptor_s &d, const int64_t *sa, int ra, const int64_t *sb,
                       int rb, int forced, ebin_plan_s **out, const int64_t *ta = nullptr,
                       const int64_t *tb = nullptr) {
    if (ra < 0 || rb < 0) return EBIN_ERR_INVALID_ARG;
    if (ra > kMaxRank || rb > kMaxRank) return EBIN_ERR_RANK_TOO_LARGE;
    if ((ra > 0 && !sa) || (rb > 0 && !sb)) return EBIN_ERR_INVALID_ARG;
    for (int i = 0; i < ra; ++i)
        if (sa[i] < 0) return EBIN_ERR_INVALID_ARG;
    for (int i = 0; i < rb; ++i)
        if (sb[i] < 0) return EBIN_ERR_INVALID_ARG;
    // strided views: A always; B only where it is an ordinary tensor
    bool bad_a = false, bad_b = false;
    ta = view_strides(sa, ta, ra, &bad_a);
    tb = d.attrs.with_scalar ? nullptr : view_strides(sb, tb, rb, &bad_b);
    if (bad_a || bad_b || (tb && !plain_b(d.op))) return EBIN_ERR_INVALID_ARG;

    // The logical shape B broadcasts with.  BatchNormalization: B = [4, C]
    // holds four parameter rows of C and broadcasts as [1, C, 1, ...] along
    // x's channel axis 1.  Clip: B = [2] holds {min, max}, a scalar pair.
    int64_t lb[kMaxRank], lt[kMaxRank];
    int rlb = rb;
    int64_t plane = 0;
    if (d.op == EBIN_OP_BATCHNORM || d.op == EBIN_OP_BIAS_PRELU ||
        d.op == EBIN_OP_BIAS_PRELU_BN) {
        // parameter rows of C: BN scale, bias, mean, var; BiasPRelu bias,
        // slope; BiasPReluBN bias, slope, scale, bn_bias, mean, var
        const int64_t rows = d.op == EBIN_OP_BATCHNORM ? 4 : d.op == EBIN_OP_BIAS_PRELU ? 2 : 6;
        if (ra < 2 || rb != 2 || sb[0] != rows || sb[1] != sa[1])
            return EBIN_ERR_INCOMPATIBLE_SHAPES;
        rlb = ra;
        for (int i = 0; i < ra; ++i) lb[i] = (i == 1) ? sa[1] : 1;
        plane = sa[1];
    } else if (d.op == EBIN_OP_CLIP) {
        if (rb != 1 || sb[0] != 2) return EBIN_ERR_INCOMPATIBLE_SHAPES;
        rlb = 0;
    } else if (d.attrs.with_scalar) {
        rlb = 0;               // B is the attribute value: a scalar
    } else if (d.op == EBIN_OP_PRELU && ra >= 2 && rb == 1 && sb[0] != 1) {
        // 0verkilll/onnx ops, PReluOp: a 1-D slope [C] is per channel, broadcast
        // across the channel dimension (axis 1), read as [C, 1, ..., 1]; its
        // view stride, if any, moves along C and the unit dims take none
        rlb = ra - 1;
        lb[0] = sb[0];
        for (int i = 1; i < rlb; ++i) lb[i] = 1;
        if (tb) {
            lt[0] = tb[0];
            for (int i = 1; i < rlb; ++i) lt[i] = 0;
            tb = lt;
        }
    } else {
        for (int i = 0; i < rb; ++i) lb[i] = sb[i];
    }

    // 1. right-align and broadcast
    const int r = std::max(ra, rlb);
    int64_t so[kMaxRank], xa[kMaxRank], xb[kMaxRank];
    for (int i = 0; i < r; ++i) {
        const int ia = i - (r - ra), ib = i - (r - rlb);
        xa[i] = ia >= 0 ? sa[ia] : 1;
        xb[i] = ib >= 0 ? lb[ib] : 1;
        if (xa[i] == xb[i]) so[i] = xa[i];
        else if (xa[i] == 1) so[i] = xb[i];
        else if (xb[i] == 1) so[i] = xa[i];
        else return EBIN_ERR_INCOMPATIBLE_SHAPES;
    }
    if (one_way(d.op)) {
        if (r != ra) return EBIN_ERR_INCOMPATIBLE_SHAPES;
        for (int i = 0; i < r; ++i)
            if (so[i] != sa[i]) return EBIN_ERR_INCOMPATIBLE_SHAPES;
    }
    const int64_t numel = elem_count(so, r), numel_a = elem_count(sa, ra);
    const int64_t numel_b = d.attrs.with_scalar ? 0 : elem_count(sb, rb);
    const int64_t span_a = ta ? view_span(sa, ta, ra) : numel_a;
    const int64_t span_b = tb ? view_span(sb, tb, rb) : numel_b;
    if (numel < 0 || numel_a < 0 || numel_b < 0 || span_a < 0 || span_b < 0)
        return EBIN_ERR_INVALID_ARG;

    auto *p = new ebin_plan_s;
    p->desc_id = d.id;
    p->dt = d.dt;
    p->rank_a = ra;
    p->rank_b = rb;
    for (int i = 0; i < ra; ++i) p->shape_a[i] = sa[i];
    for (int i = 0; i < rb; ++i) p->shape_b[i] = sb[i];
    p->op = d.op;
    p->attrs = d.attrs;
    p->out_dt = d.out_dt;
    p->dt_b = d.dt_b;
    p->rank_out = r;
    for (int i = 0; i < r; ++i) p->shape_out[i] = so[i];
    p->numel = numel;
    p->numel_a = numel_a;
    p->numel_b = numel_b;
    p->strided_a = ta != nullptr;
    p->strided_b = tb != nullptr;
    for (int i = 0; ta && i < ra; ++i) p->strides_a[i] = ta[i];
    for (int i = 0; tb && i < rb; ++i) p->strides_b[i] = tb[i];
    p->span_a = span_a;
    p->span_b = span_b;
    p->plane = plane;
    p->g = empty_geometry();
    if (numel > 0) p->g = coalesce2(so, xa, xb, r, ra, rlb, ta, tb);

    // 5. loop family (a with_scalar plan runs its own family or the general one;
    // a mixed-type Pow only the general one)
    bool ok = true;
    p->family = family_of(*p, forced, &ok);
    if (ok && d.op == EBIN_OP_POW && p->dt_b != p->dt && p->numel > 0) {
        ok = forced == EBIN_FAMILY_AUTO || forced == EBIN_FAMILY_GENERAL_STRIDED;
        p->family = ebin::FAM_GENERAL_STRIDED;
    }
    if (ok && d.attrs.with_scalar && forced != EBIN_FAMILY_AUTO &&
        forced != EBIN_FAMILY_GENERAL_STRIDED) {
        bool nat_ok = true;
        ok = forced == family_of(*p, EBIN_FAMILY_AUTO, &nat_ok);
    }
    if (!ok) {
        delete p;
        return EBIN_ERR_FAMILY;
    }
    *out = p;
    return EBIN_OK;
}

// Loop family of a three-input plan: one row traversal for inner strides in
// {0, 1}, labelled by its shape; else the general kernel.
int family_of3(const ebin_plan_s &p, int forced, bool *ok) {
    *ok = true;
    if (p.numel == 0) return ebin::FAM_EMPTY;
    const Geom &g = p.g;
    const int r = g.rank;
    const int64_t G = 16 / (int64_t)ebin_dtype_size(p.dt);
    const int64_t inner = g.n[r - 1];
    const int64_t ia = g.sa[r - 1], ib = g.sb[r - 1], ic = g.sc[r - 1];
    auto unit = [](int64_t v) { return v == 0 || v == 1; };
    const bool vec = inner % G == 0 && unit(ia) && unit(ib) && unit(ic) &&
                     (ia == 1 || ib == 1 || ic == 1) && (r == 1 || inner >= 64);
    const int natural = !vec ? ebin::FAM_GENERAL_STRIDED
                        : r > 1 ? ebin::FAM_INNER_VECTOR_OUTER
                        : (ia == 1 && ib == 1 && ic == 1) ? ebin::FAM_CONTIGUOUS
                                                          : ebin::FAM_RIGHT_SCALAR;
    if (forced == EBIN_FAMILY_AUTO) return natural;
    if (forced == EBIN_FAMILY_GENERAL_STRIDED) return forced;
    *ok = forced == natural;
    return forced;
}

// Steps 2-4 of planning a non-empty three-input broadcast: dense strides,
// zero on broadcast dims; output dims of extent 1 dropped; adjacent dims
// merged where all three inputs continue across them.  so: output shape;
// x[k]: input k right-aligned to rank r.
Geom coalesce3(const int64_t *so, const int64_t (*x)[kMaxRank], int r) {
    int64_t st[3][kMaxRank];
    for (int k = 0; k < 3; ++k) {
        int64_t acc = 1;
        for (int i = r - 1; i >= 0; --i) {
            st[k][i] = x[k][i] == 1 ? 0 : acc;
            acc *= x[k][i];
        }
    }
    Geom g{};
    int n = 0;
    for (int i = 0; i < r; ++i) {
        if (so[i] == 1) continue;
        if (n > 0 && g.sa[n - 1] == st[0][i] * so[i] && g.sb[n - 1] == st[1][i] * so[i] &&
            g.sc[n - 1] == st[2][i] * so[i]) {
            g.n[n - 1] *= so[i];
            g.sa[n - 1] = st[0][i];
            g.sb[n - 1] = st[1][i];
            g.sc[n - 1] = st[2][i];
            continue;
        }
        g.n[n] = so[i];
        g.sa[n] = st[0][i];
        g.sb[n] = st[1][i];
        g.sc[n] = st[2][i];
        ++n;
    }
    if (n == 0) {  // a single element
        g.n[0] = 1;
        g.sa[0] = g.sb[0] = g.sc[0] = 1;
        n = 1;
    }
    g.rank = n;
    return g;
}

ebin_status build_plan3(const ebin_descriptor_s &d, const int64_t *sa, int ra, const int64_t *sb,
                        int rb, const int64_t *sc, int rc, int forced, ebin_plan_s **out) {
    if (ra < 0 || rb < 0 || rc < 0) return EBIN_ERR_INVALID_ARG;
    if (ra > kMaxRank || rb > kMaxRank || rc > kMaxRank) return EBIN_ERR_RANK_TOO_LARGE;
    if ((ra > 0 && !sa) || (rb > 0 && !sb) || (rc > 0 && !sc)) return EBIN_ERR_INVALID_ARG;
    const int64_t *shp[3] = {sa, sb, sc};
    const int rk[3] = {ra, rb, rc};
    for (int k = 0; k < 3; ++k)
        for (int i = 0; i < rk[k]; ++i)
            if (shp[k][i] < 0) return EBIN_ERR_INVALID_ARG;

    // 1. right-align and broadcast all three (NumPy rules)
    const int r = std::max(ra, std::max(rb, rc));
    int64_t so[kMaxRank], x[3][kMaxRank];
    for (int i = 0; i < r; ++i) {
        int64_t o = 1;
        for (int k = 0; k < 3; ++k) {
            const int j = i - (r - rk[k]);
            x[k][i] = j >= 0 ? shp[k][j] : 1;
            if (x[k][i] == o || x[k][i] == 1) continue;
            if (o != 1) return EBIN_ERR_INCOMPATIBLE_SHAPES;
            o = x[k][i];
        }
        so[i] = o;
    }

    const int64_t numel = elem_count(so, r), numel_a = elem_count(sa, ra),
                  numel_b = elem_count(sb, rb), numel_c = elem_count(sc, rc);
    if (numel < 0 || numel_a < 0 || numel_b < 0 || numel_c < 0) return EBIN_ERR_INVALID_ARG;

    auto *p = new ebin_plan_s;
    p->desc_id = d.id;
    p->dt = d.dt;
    p->dt_b = d.dt_b;
    p->rank_a = ra;
    p->rank_b = rb;
    p->rank_c = rc;
    for (int i = 0; i < ra; ++i) p->shape_a[i] = sa[i];
    for (int i = 0; i < rb; ++i) p->shape_b[i] = sb[i];
    for (int i = 0; i < rc; ++i) p->shape_c[i] = sc[i];
    p->op = d.op;
    p->attrs = d.attrs;
    p->out_dt = d.out_dt;
    p->rank_out = r;
    for (int i = 0; i < r; ++i) p->shape_out[i] = so[i];
    p->numel = numel;
    p->numel_a = numel_a;
    p->numel_b = numel_b;
    p->numel_c = numel_c;
    p->span_a = numel_a;
    p->span_b = numel_b;
    p->g = empty_geometry();
    if (numel > 0) p->g = coalesce3(so, x, r);
    bool ok = true;
    p->family = family_of3(*p, forced, &ok);
    if (!ok) {
        delete p;
        return EBIN_ERR_FAMILY;
    }
    *out = p;
    return EBIN_OK;
}

// ------------------------------------------------------------------ plan cache
std::mutex g_cache_mu;
std::list<ebin_plan_s *> g_cache;  // most recently used first
uint64_t g_hits = 0, g_misses = 0;

void plan_unref(ebin_plan_s *p) {
    if (p && p->refs.fetch_sub(1) == 1) delete p;
}

// ta / tb: the view strides as normalised by view_strides (nullptr = dense).
bool key_equal(const ebin_plan_s &p, uint64_t id, const int64_t *sa, int ra, const int64_t *sb,
               int rb, const int64_t *sc = nullptr, int rc = -1, const int64_t *ta = nullptr,
               const int64_t *tb = nullptr) {
    if (p.desc_id != id || p.rank_a != ra || p.rank_b != rb || p.rank_c != rc) return false;
    if (p.strided_a != (ta != nullptr) || p.strided_b != (tb != nullptr)) return false;
    for (int i = 0; i < ra; ++i)
        if (p.shape_a[i] != sa[i] || (ta && p.strides_a[i] != ta[i])) return false;
    for (int i = 0; i < rb; ++i)
        if (p.shape_b[i] != sb[i] || (tb && p.strides_b[i] != tb[i])) return false;
    for (int i = 0; i < rc; ++i)
        if (p.shape_c[i] != sc[i]) return false;
    return true;
}

}  // namespace

extern "C" void ebin_descriptor_destroy(ebin_descriptor_t desc) {
    if (!desc) return;
    std::list<ebin_plan_s *> dropped;
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        for (auto it = g_cache.begin(); it != g_cache.end();) {
            if ((*it)->desc_id == desc->id) {
                dropped.push_back(*it);
                it = g_cache.erase(it);
            } else {
                ++it;
            }
        }
    }
    for (auto *p : dropped) plan_unref(p);
    delete desc;
}

namespace {

// LRU lookup, or build and insert (two-input plans: rc = -1).
ebin_status cached_plan(const ebin_descriptor_s &d, const int64_t *sa, int ra, const int64_t *sb,
                        int rb, const int64_t *sc, int rc, ebin_plan_t *out,
                        const int64_t *ta = nullptr, const int64_t *tb = nullptr) {
    // the key holds the normalised strides (dense views share the dense plans)
    bool bad = false;
    const int64_t *ka = view_strides(sa, ta, ra, &bad);
    const int64_t *kb = d.attrs.with_scalar ? nullptr : view_strides(sb, tb, rb, &bad);
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        for (auto it = g_cache.begin(); !bad && it != g_cache.end(); ++it) {
            if (key_equal(**it, d.id, sa, ra, sb, rb, sc, rc, ka, kb)) {
                ebin_plan_s *p = *it;
                g_cache.splice(g_cache.begin(), g_cache, it);
                p->refs.fetch_add(1);
                ++g_hits;
                *out = p;
                return EBIN_OK;
            }
        }
        ++g_misses;
    }
    ebin_plan_s *p = nullptr;
    const ebin_status st = rc < 0
        ? build_plan(d, sa, ra, sb, rb, EBIN_FAMILY_AUTO, &p, ta, tb)
        : build_plan3(d, sa, ra, sb, rb, sc, rc, EBIN_FAMILY_AUTO, &p);
    if (st != EBIN_OK) return st;
    ebin_plan_s *evicted = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        // another thread may have inserted the same key while this one built
        // its plan: the cache keeps one entry per key, so take that one
        for (auto it = g_cache.begin(); it != g_cache.end(); ++it) {
            if (key_equal(**it, d.id, sa, ra, sb, rb, sc, rc, ka, kb)) {
                evicted = p;   // never shared: freed below
                p = *it;
                g_cache.splice(g_cache.begin(), g_cache, it);
                p->refs.fetch_add(1);
                break;
            }
        }
        if (!evicted) {
            p->refs.fetch_add(1);  // the cache's reference
            g_cache.push_front(p);
            if ((int)g_cache.size() > EBIN_PLAN_CACHE_CAPACITY) {
                evicted = g_cache.back();
                g_cache.pop_back();
            }
        }
    }
    plan_unref(evicted);
    *out = p;
    return EBIN_OK;
}

}  // namespace

extern "C" ebin_status ebin_plan_create(ebin_descriptor_t desc, const int64_t *shape_a,
                                        int rank_a, const int64_t *shape_b, int rank_b,
                                        ebin_plan_t *out) {
    if (!desc || !out) return EBIN_ERR_INVALID_ARG;
    *out = nullptr;
    if (ternary(desc->op)) return EBIN_ERR_INVALID_ARG;   // three inputs: ebin_plan_create3
    if (desc->attrs.with_scalar) rank_b = 0;   // shape B is not read
    if (rank_a < 0 || rank_b < 0) return EBIN_ERR_INVALID_ARG;
    if (rank_a > kMaxRank || rank_b > kMaxRank) return EBIN_ERR_RANK_TOO_LARGE;
    if ((rank_a > 0 && !shape_a) || (rank_b > 0 && !shape_b)) return EBIN_ERR_INVALID_ARG;
    return cached_plan(*desc, shape_a, rank_a, shape_b, rank_b, nullptr, -1, out);
}

extern "C" ebin_status ebin_plan_create_forced(ebin_descriptor_t desc, const int64_t *shape_a,
                                               int rank_a, const int64_t *shape_b, int rank_b,
                                               ebin_family family, ebin_plan_t *out) {
    if (!desc || !out) return EBIN_ERR_INVALID_ARG;
    *out = nullptr;
    if (ternary(desc->op)) return EBIN_ERR_INVALID_ARG;
    if (desc->attrs.with_scalar) rank_b = 0;
    ebin_plan_s *p = nullptr;
    const ebin_status st = build_plan(*desc, shape_a, rank_a, shape_b, rank_b, (int)family, &p);
    if (st != EBIN_OK) return st;
    *out = p;
    return EBIN_OK;
}

extern "C" ebin_status ebin_plan_create_strided(ebin_descriptor_t desc, const int64_t *shape_a,
                                                const int64_t *strides_a, int rank_a,
                                                const int64_t *shape_b, const int64_t *strides_b,
                                                int rank_b, ebin_family family,
                                                ebin_plan_t *out) {
    if (!desc || !out) return EBIN_ERR_INVALID_ARG;
    *out = nullptr;
    if (ternary(desc->op)) return EBIN_ERR_INVALID_ARG;
    if (desc->attrs.with_scalar) {
        rank_b = 0;
        strides_b = nullptr;
    }
    if (rank_a < 0 || rank_b < 0) return EBIN_ERR_INVALID_ARG;
    if (rank_a > kMaxRank || rank_b > kMaxRank) return EBIN_ERR_RANK_TOO_LARGE;
    if ((rank_a > 0 && !shape_a) || (rank_b > 0 && !shape_b)) return EBIN_ERR_INVALID_ARG;
    if (family == EBIN_FAMILY_AUTO)
        return cached_plan(*desc, shape_a, rank_a, shape_b, rank_b, nullptr, -1, out, strides_a,
                           strides_b);
    ebin_plan_s *p = nullptr;
    const ebin_status st = build_plan(*desc, shape_a, rank_a, shape_b, rank_b, (int)family, &p,
                                      strides_a, strides_b);
    if (st != EBIN_OK) return st;
    *out = p;
    return EBIN_OK;
}

extern "C" ebin_status ebin_plan_create3(ebin_descriptor_t desc, const int64_t *shape_a,
                                         int rank_a, const int64_t *shape_b, int rank_b,
                                         const int64_t *shape_c, int rank_c, ebin_plan_t *out) {
    if (!desc || !out) return EBIN_ERR_INVALID_ARG;
    *out = nullptr;
    if (!ternary(desc->op)) return EBIN_ERR_INVALID_ARG;
    if (rank_a < 0 || rank_b < 0 || rank_c < 0) return EBIN_ERR_INVALID_ARG;
    if (rank_a > kMaxRank || rank_b > kMaxRank || rank_c > kMaxRank) return EBIN_ERR_RANK_TOO_LARGE;
    if ((rank_a > 0 && !shape_a) || (rank_b > 0 && !shape_b) || (rank_c > 0 && !shape_c))
        return EBIN_ERR_INVALID_ARG;
    return cached_plan(*desc, shape_a, rank_a, shape_b, rank_b, shape_c, rank_c, out);
}

extern "C" ebin_status ebin_plan_create3_forced(ebin_descriptor_t desc, const int64_t *shape_a,
                                                int rank_a, const int64_t *shape_b, int rank_b,
                                                const int64_t *shape_c, int rank_c,
                                                ebin_family family, ebin_plan_t *out) {
    if (!desc || !out) return EBIN_ERR_INVALID_ARG;
    *out = nullptr;
    if (!ternary(desc->op)) return EBIN_ERR_INVALID_ARG;
    ebin_plan_s *p = nullptr;
    const ebin_status st =
        build_plan3(*desc, shape_a, rank_a, shape_b, rank_b, shape_c, rank_c, (int)family, &p);
    if (st != EBIN_OK) return st;
    *out = p;
    return EBIN_OK;
}

extern "C" ebin_status ebin_plan_output_shape(ebin_plan_t plan, int64_t *shape, int *rank) {
    if (!plan || !shape || !rank) return EBIN_ERR_INVALID_ARG;
    *rank = plan->rank_out;
    for (int i = 0; i < plan->rank_out; ++i) shape[i] = plan->shape_out[i];
    return EBIN_OK;
}

extern "C" ebin_status ebin_plan_numel(ebin_plan_t plan, int64_t *numel) {
    if (!plan || !numel) return EBIN_ERR_INVALID_ARG;
    *numel = plan->numel;
    return EBIN_OK;
}

extern "C" ebin_status ebin_plan_family(ebin_plan_t plan, ebin_family *family) {
    if (!plan || !family) return EBIN_ERR_INVALID_ARG;
    *family = (ebin_family)plan->family;
    return EBIN_OK;
}

extern "C" ebin_status ebin_plan_geometry(ebin_plan_t plan, int *rank, int64_t *n,
                                          int64_t *stride_a, int64_t *stride_b) {
    if (!plan || !rank || !n || !stride_a || !stride_b) return EBIN_ERR_INVALID_ARG;
    *rank = plan->g.rank;
    for (int i = 0; i < plan->g.rank; ++i) {
        n[i] = plan->g.n[i];
        stride_a[i] = plan->g.sa[i];
        stride_b[i] = plan->g.sb[i];
    }
    return EBIN_OK;
}

extern "C" void ebin_plan_release(ebin_plan_t plan) { plan_unref(plan); }

extern "C" ebin_status ebin_plan_cache_stats(uint64_t *hits, uint64_t *misses, int *size) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    if (hits) *hits = g_hits;
    if (misses) *misses = g_misses;
    if (size) *size = (int)g_cache.size();
    return EBIN_OK;
}

extern "C" void ebin_plan_cache_clear(void) {
    std::list<ebin_plan_s *> dropped;
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        dropped.swap(g_cache);
        g_hits = 0;
        g_misses = 0;
    }
    for (auto *p : dropped) plan_unref(p);
}

// ------------------------------------------------------------------ execution
namespace {

std::mutex g_dev_mu;
std::map<std::pair<int, uintptr_t>, uint32_t *> g_status_words;
std::atomic<int> g_sm_count[128];   // 0 until looked up (host threads race to fill it)

int sm_count(int dev) {
    const bool slot = dev >= 0 && dev < 128;
    if (slot) {
        const int n = g_sm_count[dev].load(std::memory_order_relaxed);
        if (n > 0) return n;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (slot) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

// The status word of (device, stream), allocated and zeroed (stream-ordered)
// on first use.
uint32_t *status_word(int dev, cudaStream_t stream, bool create) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    const auto key = std::make_pair(dev, (uintptr_t)stream);
    auto it = g_status_words.find(key);
    if (it != g_status_words.end()) return it->second;
    if (!create) return nullptr;
    uint32_t *w = nullptr;
    if (cudaMalloc(&w, sizeof(uint32_t)) != cudaSuccess) return nullptr;
    if (cudaMemsetAsync(w, 0, sizeof(uint32_t), stream) != cudaSuccess) {
        cudaFree(w);
        return nullptr;
    }
    g_status_words[key] = w;
    return w;
}

bool overlaps(const void *p, int64_t pb, const void *q, int64_t qb) {
    const uintptr_t a = (uintptr_t)p, b = (uintptr_t)q;
    return pb > 0 && qb > 0 && a < b + (uintptr_t)qb && b < a + (uintptr_t)pb;
}

}  // namespace

cudaError_t ebin::launch(const Launch &L) {
#define EBIN_PICK(g)                                                                      \
    switch (L.dt) {                                                                       \
    case 0: return launch_##g##_0(L);                                                     \
    case 1: return launch_##g##_1(L);                                                     \
    case 2: return launch_##g##_2(L);                                                     \
    case 3: return launch_##g##_3(L);                                                     \
    case 4: return launch_##g##_4(L);                                                     \
    case 5: return launch_##g##_5(L);                                                     \
    case 6: return launch_##g##_6(L);                                                     \
    case 7: return launch_##g##_7(L);                                                     \
    case 8: return launch_##g##_8(L);                                                     \
    case 9: return launch_##g##_9(L);                                                     \
    case 10: return launch_##g##_10(L);                                                   \
    case 11: return launch_##g##_11(L);                                                   \
    case 12: return launch_##g##_12(L);                                                   \
    default: return cudaErrorInvalidValue;                                                \
    }
    switch (L.op) {
    case EBIN_OP_ADD: case EBIN_OP_SUB: case EBIN_OP_MUL: case EBIN_OP_DIV: EBIN_PICK(arith)
    case EBIN_OP_MOD: EBIN_PICK(mod)
    case EBIN_OP_POW:
        if (L.dt_b != L.dt) EBIN_PICK(powmix)
        EBIN_PICK(pow)
    case EBIN_OP_EQUAL: case EBIN_OP_LESS: case EBIN_OP_GREATER: case EBIN_OP_LESS_OR_EQUAL:
    case EBIN_OP_GREATER_OR_EQUAL: EBIN_PICK(cmp)
    case EBIN_OP_AND: case EBIN_OP_OR: case EBIN_OP_XOR: case EBIN_OP_BITWISE_AND:
    case EBIN_OP_BITWISE_OR: case EBIN_OP_BITWISE_XOR: case EBIN_OP_BITSHIFT: EBIN_PICK(logic)
    case EBIN_OP_PRELU: case EBIN_OP_BATCHNORM: case EBIN_OP_CLIP: case EBIN_OP_BIAS_PRELU:
    case EBIN_OP_BIAS_PRELU_BN:
        EBIN_PICK(chan)
    case EBIN_OP_MAX: case EBIN_OP_MIN: case EBIN_OP_RSUB: case EBIN_OP_RDIV: EBIN_PICK(ext)
    case EBIN_OP_MULADD: EBIN_PICK(tern)
    default: return cudaErrorInvalidValue;
    }
#undef EBIN_PICK
}

// Checks and launch description shared by the execute entry points (the
// no-allocation one included): the buffer, alias and alignment rules of
// ebin_execute, and the status word -- the stream's own, allocated on first
// use, or `status` when the caller supplies one.
ebin_status ebin::prepare_launch(const ebin_plan_s &p, const void *A, const void *B, void *out,
                                 cudaStream_t s, uint32_t *status, ebin::Launch &L) {
    const bool b_needed = !(p.op == EBIN_OP_CLIP && !p.attrs.clip_has_min && !p.attrs.clip_has_max) &&
                          !p.attrs.with_scalar;
    if (!A || !out || (b_needed && !B)) return EBIN_ERR_INVALID_ARG;
    if (p.attrs.with_scalar) B = nullptr;   // never read

    // Aliasing: an input may share storage with out only as the identical
    // buffer of the output's type and element count; a broadcast input or a
    // parameter block is never overwritten in place.
    // (a strided view may be in place only where its layout is the output's:
    // never, so any overlap with out is ALIAS)
    const int64_t isz = (int64_t)ebin_dtype_size(p.dt);
    const int64_t isz_b = (int64_t)ebin_dtype_size(p.dt_b);
    const int64_t out_bytes = p.numel * (int64_t)ebin_dtype_size(p.out_dt);
    if (overlaps(A, p.span_a * isz, out, out_bytes)) {
        if (!(A == out && !p.strided_a && p.numel_a == p.numel && p.dt == p.out_dt))
            return EBIN_ERR_ALIAS;
    }
    if (B && overlaps(B, p.span_b * isz_b, out, out_bytes)) {
        if (!(plain_b(p.op) && B == out && !p.strided_b && p.numel_b == p.numel &&
              p.dt_b == p.out_dt))
            return EBIN_ERR_ALIAS;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EBIN_ERR_CUDA;
    L = ebin::Launch{};
    L.op = p.op;
    L.dt = dt_class(p.dt);
    L.dt_b = dt_class(p.dt_b);
    L.family = p.family;
    L.g = p.g;
    L.numel = p.numel;
    L.A = A;
    L.B = B;
    L.out = out;
    L.args.fmod = p.attrs.fmod;
    L.args.direction = p.attrs.direction;
    L.args.eps = p.attrs.epsilon;
    L.args.has_min = p.attrs.clip_has_min;
    L.args.has_max = p.attrs.clip_has_max;
    L.args.plane = p.plane;
    L.args.with_scalar = p.attrs.with_scalar;
    L.args.scalar_b = p.attrs.scalar_b;
    L.args.one = 1.0f;
    L.stream = s;
    L.num_sms = sm_count(dev);
    L.status = nullptr;
    if (validates(p.op, p.dt)) {
        L.status = status ? status : status_word(dev, s, true);
        if (!L.status) return EBIN_ERR_CUDA;
    }
    // The vector families move 16-byte packs: pointers off that alignment
    // take the general kernel, which reads element by element.
    if (L.family != ebin::FAM_GENERAL_STRIDED) {
        const uintptr_t G = 16 / (uintptr_t)isz;
        const uintptr_t out_align = G * (uintptr_t)ebin_dtype_size(p.out_dt);
        const bool aligned = ((uintptr_t)A % 16 == 0) && (!B || (uintptr_t)B % 16 == 0) &&
                             ((uintptr_t)out % out_align == 0);
        if (!aligned) L.family = ebin::FAM_GENERAL_STRIDED;
    }
    return EBIN_OK;
}

namespace {

using ebin::prepare_launch;

ebin_status launch_counted(const ebin::Launch &L) {
    const cudaError_t e = ebin::launch(L);
    g_launches.fetch_add(1);
    return e == cudaSuccess ? EBIN_OK : EBIN_ERR_CUDA;
}

}  // namespace

extern "C" ebin_status ebin_execute(ebin_plan_t plan, const void *A, const void *B, void *out,
                                    void *stream) {
    if (!plan || plan->rank_c >= 0) return EBIN_ERR_INVALID_ARG;
    const ebin_plan_s &p = *plan;
    if (p.numel == 0) return EBIN_OK;  // empty dims: no work, nothing read
    ebin::Launch L;
    const ebin_status st = prepare_launch(p, A, B, out, static_cast<cudaStream_t>(stream), nullptr, L);
    if (st != EBIN_OK) return st;
    return launch_counted(L);
}

extern "C" ebin_status ebin_execute3(ebin_plan_t plan, const void *A, const void *B,
                                     const void *C, void *out, void *stream) {
    if (!plan || plan->rank_c < 0) return EBIN_ERR_INVALID_ARG;
    const ebin_plan_s &p = *plan;
    if (p.numel == 0) return EBIN_OK;
    if (!A || !B || !C || !out) return EBIN_ERR_INVALID_ARG;
    // an input may be out only as the identical buffer of the output's size
    const int64_t isz = (int64_t)ebin_dtype_size(p.dt);
    const int64_t out_bytes = p.numel * (int64_t)ebin_dtype_size(p.out_dt);
    const void *in[3] = {A, B, C};
    const int64_t cnt[3] = {p.numel_a, p.numel_b, p.numel_c};
    for (int k = 0; k < 3; ++k)
        if (overlaps(in[k], cnt[k] * isz, out, out_bytes) &&
            !(in[k] == out && cnt[k] == p.numel && p.dt == p.out_dt))
            return EBIN_ERR_ALIAS;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EBIN_ERR_CUDA;
    ebin::Launch L{};
    L.op = p.op;
    L.dt = dt_class(p.dt);
    L.dt_b = L.dt;
    L.family = p.family;
    L.g = p.g;
    L.numel = p.numel;
    L.A = A;
    L.B = B;
    L.C = C;
    L.out = out;
    L.stream = static_cast<cudaStream_t>(stream);
    L.num_sms = sm_count(dev);
    L.status = nullptr;
    if (L.family != ebin::FAM_GENERAL_STRIDED) {
        bool aligned = (uintptr_t)out % 16 == 0;
        for (int k = 0; k < 3; ++k) aligned = aligned && (uintptr_t)in[k] % 16 == 0;
        if (!aligned) L.family = ebin::FAM_GENERAL_STRIDED;
    }
    return launch_counted(L);
}

namespace {

// Host-buffer pipeline of one device: an input-copy and an output-copy stream
// beside the caller's, and reusable events.  Created on first use, kept until
// the process exits; `mu` makes one call's enqueue sequence atomic.
constexpr int kPipeChunks = 32;                 // at most this many chunks per call
constexpr int64_t kPipeMinChunk = int64_t(1) << 20;   // elements
constexpr int64_t kPipeGrain = 4096;            // chunk sizes are multiples of this
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t copied[kPipeChunks] = {}, computed[kPipeChunks] = {};
};
HostPipe g_pipes[128];

HostPipe *host_pipe(int dev) {
    if (dev < 0 || dev >= 128) return nullptr;
    HostPipe &h = g_pipes[dev];
    std::lock_guard<std::mutex> lk(h.mu);
    if (h.ready) return &h;
    const unsigned ev = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.start, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&h.done, ev) == cudaSuccess;
    for (int c = 0; ok && c < kPipeChunks; ++c)
        ok = cudaEventCreateWithFlags(&h.copied[c], ev) == cudaSuccess &&
             cudaEventCreateWithFlags(&h.computed[c], ev) == cudaSuccess;
    if (!ok) return nullptr;   // partially created handles stay unused
    h.ready = true;
    return &h;
}

// Copies in, kernel, copies out, one after the other on the caller's stream.
ebin_status host_serial(const ebin_plan_s &p, const ebin::Launch &L, const void *host_a,
                        const void *host_b, void *host_out, void *dev_a, void *dev_b,
                        void *dev_out, cudaStream_t s) {
    const size_t isz = ebin_dtype_size(p.dt);
    // the inputs' whole storage extents (a strided view's span)
    if (cudaMemcpyAsync(dev_a, host_a, (size_t)p.span_a * isz, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return EBIN_ERR_CUDA;
    if (host_b && dev_b && p.span_b > 0) {
        if (cudaMemcpyAsync(dev_b, host_b, (size_t)p.span_b * ebin_dtype_size(p.dt_b),
                            cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
            return EBIN_ERR_CUDA;
    }
    const ebin_status st = launch_counted(L);
    if (st != EBIN_OK) return st;
    if (cudaMemcpyAsync(host_out, dev_out, (size_t)p.numel * ebin_dtype_size(p.out_dt),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return EBIN_ERR_CUDA;
    return EBIN_OK;
}

}  // namespace

extern "C" ebin_status ebin_execute_host(ebin_plan_t plan, const void *host_a, const void *host_b,
                                         void *host_out, void *dev_a, void *dev_b, void *dev_out,
                                         void *stream) {
    if (!plan || plan->rank_c >= 0) return EBIN_ERR_INVALID_ARG;
    const ebin_plan_s &p = *plan;
    if (p.numel == 0) return EBIN_OK;
    if (!host_a || !host_out || !dev_a || !dev_out) return EBIN_ERR_INVALID_ARG;
    if (host_b && !dev_b) return EBIN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ebin::Launch L;
    ebin_status st = prepare_launch(p, dev_a, host_b ? dev_b : nullptr, dev_out, s, nullptr, L);
    if (st != EBIN_OK) return st;

    // Streaming families whose output range [o, o+n) reads only the same range
    // of each dense operand (and all of a scalar one) run as a pipeline of
    // chunks: chunk c+1 is copied in while chunk c computes and chunk c-1 is
    // copied out, on two copy streams beside the caller's.
    const bool streaming = (L.family == ebin::FAM_CONTIGUOUS ||
                            L.family == ebin::FAM_LEFT_SCALAR ||
                            L.family == ebin::FAM_RIGHT_SCALAR) &&
                           !p.strided_a && !p.strided_b;
    int dev = 0;
    HostPipe *hp = nullptr;
    if (streaming && p.numel >= 2 * kPipeMinChunk && cudaGetDevice(&dev) == cudaSuccess)
        hp = host_pipe(dev);
    if (!hp) return host_serial(p, L, host_a, host_b, host_out, dev_a, dev_b, dev_out, s);

    const size_t isz = ebin_dtype_size(p.dt), osz = ebin_dtype_size(p.out_dt);
    const size_t isz_b = ebin_dtype_size(p.dt_b);   // binary32 parameters beside 16-bit x
    // An operand with stride 1 moves with the output: chunk c reads its range
    // [off, off + n).  A plain one is copied chunk by chunk; a parameter block
    // (rows of C, plane elements apart, each moving with the output) is copied
    // whole, first, and each chunk's kernel starts off elements into it.  An
    // operand with stride 0 is a scalar, copied whole, first.
    const bool a_moves = L.g.sa[0] != 0, b_moves = L.B && L.g.sb[0] != 0;
    const bool b_chunked = b_moves && plain_b(p.op);
    const int64_t want = std::max(kPipeMinChunk, (p.numel + kPipeChunks - 1) / kPipeChunks);
    const int64_t chunk = (want + kPipeGrain - 1) / kPipeGrain * kPipeGrain;
    const int nchunks = (int)((p.numel + chunk - 1) / chunk);

    std::lock_guard<std::mutex> lk(hp->mu);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // the copy streams start after everything already queued on the caller's
    if (!ok(cudaEventRecord(hp->start, s)) || !ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) ||
        !ok(cudaStreamWaitEvent(hp->out, hp->start, 0)))
        return EBIN_ERR_CUDA;
    if (!a_moves && !ok(cudaMemcpyAsync(dev_a, host_a, (size_t)p.numel_a * isz,
                                        cudaMemcpyHostToDevice, hp->in)))
        return EBIN_ERR_CUDA;
    if (L.B && !b_chunked && p.numel_b > 0 &&
        !ok(cudaMemcpyAsync(dev_b, host_b, (size_t)p.numel_b * isz_b, cudaMemcpyHostToDevice,
                            hp->in)))
        return EBIN_ERR_CUDA;
    for (int c = 0; c < nchunks; ++c) {
        const int64_t off = (int64_t)c * chunk;
        const int64_t n = std::min(chunk, p.numel - off);
        const size_t ib = (size_t)off * isz, nb = (size_t)n * isz;
        const size_t ib_b = (size_t)off * isz_b, nb_b = (size_t)n * isz_b;
        if (a_moves && !ok(cudaMemcpyAsync((char *)dev_a + ib, (const char *)host_a + ib, nb,
                                           cudaMemcpyHostToDevice, hp->in)))
            return EBIN_ERR_CUDA;
        if (b_chunked &&
            !ok(cudaMemcpyAsync((char *)dev_b + ib_b, (const char *)host_b + ib_b, nb_b,
                                cudaMemcpyHostToDevice, hp->in)))
            return EBIN_ERR_CUDA;
        if (!ok(cudaEventRecord(hp->copied[c], hp->in)) ||
            !ok(cudaStreamWaitEvent(s, hp->copied[c], 0)))
            return EBIN_ERR_CUDA;
        ebin::Launch Lc = L;
        Lc.numel = n;
        if (Lc.g.rank == 1) Lc.g.n[0] = n;   // the chunk's own extent
        Lc.A = a_moves ? (const void *)((const char *)dev_a + ib) : dev_a;
        Lc.B = b_moves ? (const void *)((const char *)dev_b + ib_b) : L.B;
        Lc.out = (char *)dev_out + (size_t)off * osz;
        if ((st = launch_counted(Lc)) != EBIN_OK) return st;
        if (!ok(cudaEventRecord(hp->computed[c], s)) ||
            !ok(cudaStreamWaitEvent(hp->out, hp->computed[c], 0)) ||
            !ok(cudaMemcpyAsync((char *)host_out + (size_t)off * osz,
                                (const char *)dev_out + (size_t)off * osz, (size_t)n * osz,
                                cudaMemcpyDeviceToHost, hp->out)))
            return EBIN_ERR_CUDA;
    }
    // the caller's stream completes only after the last output copy
    if (!ok(cudaEventRecord(hp->done, hp->out)) || !ok(cudaStreamWaitEvent(s, hp->done, 0)))
        return EBIN_ERR_CUDA;
    return EBIN_OK;
}

namespace {

// cuPointerGetAttribute, looked up through the runtime (no link against the
// driver library), or null.
using PointerAttrFn = CUresult (*)(void *, CUpointer_attribute, CUdeviceptr);

PointerAttrFn pointer_attr_fn() {
    static const PointerAttrFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (PointerAttrFn) nullptr;
        }
        return reinterpret_cast<PointerAttrFn>(f);
    }();
    return fn;
}

// Device address of the host range [p, p + bytes) when all of it lies in one
// pinned allocation mapped into the device's address space (first and last
// byte in host memory, with the same allocation id and a contiguous device
// mapping); else null.
const void *mapped_range(const void *p, size_t bytes) {
    if (!p || bytes == 0) return nullptr;
    const char *first = static_cast<const char *>(p);
    const char *last = first + (bytes - 1);
    cudaPointerAttributes a0{}, a1{};
    if (cudaPointerGetAttributes(&a0, first) != cudaSuccess ||
        cudaPointerGetAttributes(&a1, last) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a0.type != cudaMemoryTypeHost || a1.type != cudaMemoryTypeHost || !a0.devicePointer ||
        static_cast<const char *>(a1.devicePointer) !=
            static_cast<const char *>(a0.devicePointer) + (bytes - 1))
        return nullptr;
    const PointerAttrFn fn = pointer_attr_fn();
    unsigned long long id0 = 0, id1 = 0;
    if (!fn || fn(&id0, CU_POINTER_ATTRIBUTE_BUFFER_ID, (CUdeviceptr)(uintptr_t)first) != CUDA_SUCCESS ||
        fn(&id1, CU_POINTER_ATTRIBUTE_BUFFER_ID, (CUdeviceptr)(uintptr_t)last) != CUDA_SUCCESS ||
        id0 != id1)
        return nullptr;
    return a0.devicePointer;
}

}  // namespace

extern "C" ebin_status ebin_execute_mapped(ebin_plan_t plan, const void *host_a,
                                           const void *host_b, void *host_out, void *stream) {
    if (!plan || plan->rank_c >= 0) return EBIN_ERR_INVALID_ARG;
    const ebin_plan_s &p = *plan;
    if (p.numel == 0) return EBIN_OK;
    if (!host_a || !host_out) return EBIN_ERR_INVALID_ARG;
    const void *da = mapped_range(host_a, (size_t)p.span_a * ebin_dtype_size(p.dt));
    const void *db = nullptr;
    if (host_b && p.span_b > 0) {
        db = mapped_range(host_b, (size_t)p.span_b * ebin_dtype_size(p.dt_b));
        if (!db) return EBIN_ERR_INVALID_ARG;
    }
    void *dout = const_cast<void *>(
        mapped_range(host_out, (size_t)p.numel * ebin_dtype_size(p.out_dt)));
    if (!da || !dout) return EBIN_ERR_INVALID_ARG;
    ebin::Launch L;
    const ebin_status st = prepare_launch(p, da, db, dout, static_cast<cudaStream_t>(stream), nullptr, L);
    if (st != EBIN_OK) return st;
    return launch_counted(L);
}

extern "C" ebin_status ebin_execute3_mapped(ebin_plan_t plan, const void *host_a,
                                            const void *host_b, const void *host_c,
                                            void *host_out, void *stream) {
    if (!plan || plan->rank_c < 0) return EBIN_ERR_INVALID_ARG;
    const ebin_plan_s &p = *plan;
    if (p.numel == 0) return EBIN_OK;
    if (!host_a || !host_b || !host_c || !host_out) return EBIN_ERR_INVALID_ARG;
    const size_t isz = ebin_dtype_size(p.dt);
    const void *da = mapped_range(host_a, (size_t)p.numel_a * isz);
    const void *db = mapped_range(host_b, (size_t)p.numel_b * isz);
    const void *dc = mapped_range(host_c, (size_t)p.numel_c * isz);
    void *dout = const_cast<void *>(
        mapped_range(host_out, (size_t)p.numel * ebin_dtype_size(p.out_dt)));
    if (!da || !db || !dc || !dout) return EBIN_ERR_INVALID_ARG;
    return ebin_execute3(plan, da, db, dc, dout, stream);
}

extern "C" ebin_status ebin_get_device_status(void *stream, uint32_t *bits) {
    if (!bits) return EBIN_ERR_INVALID_ARG;
    *bits = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EBIN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *w = status_word(dev, s, false);
    if (!w) return cudaStreamSynchronize(s) == cudaSuccess ? EBIN_OK : EBIN_ERR_CUDA;
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, w, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return EBIN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return EBIN_ERR_CUDA;
    if (cudaMemsetAsync(w, 0, sizeof(uint32_t), s) != cudaSuccess) return EBIN_ERR_CUDA;
    *bits = h;
    return EBIN_OK;
}

extern "C" uint64_t ebin_launch_count(void) { return g_launches.load(); }

void ebin::count_launch() { g_launches.fetch_add(1); }

extern "C" size_t ebin_dtype_size(ebin_dtype t) {
    switch (t) {
    case EBIN_FLOAT32: case EBIN_INT32: case EBIN_UINT32: return 4;
    case EBIN_FLOAT16: case EBIN_BFLOAT16: case EBIN_INT16: case EBIN_UINT16: return 2;
    case EBIN_INT64: case EBIN_UINT64: case EBIN_DOUBLE: return 8;
    case EBIN_UINT8: case EBIN_BOOL: case EBIN_INT8: return 1;
    }
    return 0;
}

extern "C" const char *ebin_status_string(ebin_status s) {
    switch (s) {
    case EBIN_OK: return "ok";
    case EBIN_ERR_INVALID_ARG: return "invalid argument";
    case EBIN_ERR_UNSUPPORTED_OP: return "unsupported operator";
    case EBIN_ERR_UNSUPPORTED_TYPE: return "unsupported type";
    case EBIN_ERR_INVALID_ATTR: return "invalid attribute";
    case EBIN_ERR_INCOMPATIBLE_SHAPES: return "incompatible shapes";
    case EBIN_ERR_RANK_TOO_LARGE: return "rank too large";
    case EBIN_ERR_ALIAS: return "input aliases the output";
    case EBIN_ERR_CUDA: return "CUDA error";
    case EBIN_ERR_FAMILY: return "loop family cannot traverse this plan";
    }
    return "unknown status";
}
