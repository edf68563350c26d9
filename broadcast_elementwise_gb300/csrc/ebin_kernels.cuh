// Loop-family kernels of the broadcast binary engine for sm_103a, and the
// per-operator launcher that picks one from the plan's family.
//
// Families ("Binary Kernel Design", section "Operators and traversal",
// loop-family table), each a kernel template instantiated per operator and
// element type:
//   k_contiguous        A, B and out advance together          (Contiguous)
//   k_scalar            one operand is a single value          (Left / right scalar)
//   k_rows<NOPREFIX>    rank-2 plans: one value per row, or one row block
//                       reused by every row                    (Repeated contiguous block)
//   k_rows<G>           vectorised inner rows, outer offsets advanced by
//                       constant steps                          (Inner-vector / outer broadcast)
//   k_rows<G=1, any>    any coalesced strides, element by element (General strided)
//
// GB300 design points (all measured on the part):
//  * One tile per CTA ("one-shot" grid): a grid-stride persistent loop reached
//    ~6.5 TB/s on the contiguous fp32 stream, one tile per CTA ~7.1 TB/s.
//  * Dense streams move as 16-byte vectors: ld.global.nc.L1::no_allocate for
//    inputs read once, st.global.cs (evict-first) for outputs.  A warp touches
//    512 consecutive bytes per access (16 sectors per request).
//  * Row traversal: a tile is (outer prefix index, a run of rows along the
//    dimension next to the inner one, a chunk of columns).  A thread owns one
//    column group and walks its rows with constant offset steps -- "offsets
//    advance incrementally; division and modulo are not performed for every
//    output element".  The tile index is split with precomputed
//    Granlund-Montgomery divisors (multiply-high and shifts), once per thread.
//    An operand whose run stride is 0 (a row block reused by every row) stays
//    in registers for the whole run.
//
// Validation ("Compute, scheduling, and safety"): operators that can meet an
// invalid element (integer division by zero, shift counts) write 0 for it and
// OR a bit into the stream's status word once per thread.  There is no trap,
// no assert and no waiting in any kernel.
#pragma once

#include <cstring>
#include <type_traits>

#include "ebin_ops.cuh"

namespace ebin {

constexpr int kThreads = 256;

// A pack of G elements is aligned to its size when that is a power of two up to
// 16 bytes (so it moves as one vector access); other packs (parameter blocks)
// keep the element's natural alignment.
template <class T, int G> constexpr size_t pack_align() {
    constexpr size_t n = sizeof(T) * G;
    return (n <= 16 && (n & (n - 1)) == 0) ? n : alignof(T);
}

template <class T, int G> struct alignas(pack_align<T, G>()) Pack {
    T v[G];
};

// 16-byte read-once load, kept out of L1.
template <class T, int G>
__device__ __forceinline__ Pack<T, G> ld_stream(const T *p) {
    static_assert(sizeof(T) * G == 16, "16-byte vectors only");
    uint32_t r0, r1, r2, r3;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "l"(p));
    const uint32_t w[4] = {r0, r1, r2, r3};
    Pack<T, G> out;
    memcpy(&out, w, 16);
    return out;
}

// Streaming (evict-first) store of a pack of 1..16 bytes.
template <class T, int G>
__device__ __forceinline__ void st_stream(T *p, const Pack<T, G> &v) {
    constexpr int kBytes = (int)sizeof(T) * G;
    if constexpr (kBytes == 16) {
        uint32_t w[4];
        memcpy(w, &v, 16);
        asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
    } else if constexpr (kBytes == 8) {
        uint32_t w[2];
        memcpy(w, &v, 8);
        asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(w[0]), "r"(w[1])
                     : "memory");
    } else if constexpr (kBytes == 4) {
        uint32_t w;
        memcpy(&w, &v, 4);
        asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(w) : "memory");
    } else if constexpr (kBytes == 2) {
        uint16_t w;
        memcpy(&w, &v, 2);
        asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(w) : "memory");
    } else {
        static_assert(kBytes == 1, "pack size");
        uint32_t w = 0;
        memcpy(&w, &v, 1);
        asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(w) : "memory");
    }
}

// Programmatic dependent launch.  Every kernel first lets the next grid on its
// stream be scheduled (it is launched once all CTAs of this grid have started),
// then waits until the grids it depends on have finished and their memory is
// visible, before its first global access.  The next kernel's launch then
// overlaps this kernel's last wave instead of following its completion.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The same split in two, for kernels with index arithmetic to do first: the
// arithmetic between pdl_launch and pdl_wait reads kernel parameters only
// and overlaps the tail of the grid this one depends on.
__device__ __forceinline__ void pdl_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <class Op>
__device__ __forceinline__ void flush_err(uint32_t *status, uint32_t err) {
    if constexpr (Op::kValidates) {
        if (err) atomicOr(status, err);
    }
}

// Operators with a whole-group form (Op::kPack) use it for groups of a multiple of 4.
template <class Op, class = void> struct HasPack : std::false_type {};
template <class Op>
struct HasPack<Op, std::void_t<decltype(Op::kPack)>> : std::bool_constant<Op::kPack> {};

// Operators that prepare a B shared by many elements (Op::kPrep, Op::prep,
// Op::apply_prep_group) -- e.g. the reciprocal of a Mod divisor.
template <class Op, class = void> struct HasPrep : std::false_type {};
// The fewest rows a thread of the row kernel walks (Op::kMinRows, default 1):
// operators with costly per-row parameters amortise the thread's setup.
template <class Op, class = void> struct MinRowsOf : std::integral_constant<int, 1> {};
template <class Op>
struct MinRowsOf<Op, std::void_t<decltype(Op::kMinRows)>>
    : std::integral_constant<int, Op::kMinRows> {};
template <class Op>
struct HasPrep<Op, std::void_t<decltype(Op::kPrep)>> : std::bool_constant<Op::kPrep> {};

// Operators with a form for a group of elements that share one B value
// (Op::kGroup, Op::apply_group) -- e.g. BatchNormalization's prepared division.
template <class Op, class = void> struct HasGroup : std::false_type {};
template <class Op>
struct HasGroup<Op, std::void_t<decltype(Op::kGroup)>> : std::bool_constant<Op::kGroup> {};

struct PrepNone {
    using PB = int;
};

// B's element type: Op::BIn where it differs from A's (mixed-type Pow), else In.
template <class Op, class = void> struct BInOf {
    using type = typename Op::In;
};
template <class Op> struct BInOf<Op, std::void_t<typename Op::BIn>> {
    using type = typename Op::BIn;
};

// o[k] = op(a[k], b[k]) for one group of G elements.  SA / SB: the operand is
// one value for the whole group (a[0] / b[0]), not G values.
template <class Op, int G, bool SA = false, bool SB = false>
__device__ __forceinline__ void compute_group(const typename Op::In *a, const typename Op::BV *b,
                                              typename Op::Out *o, const OpArgs &args,
                                              uint32_t &err) {
    if constexpr (SB && HasPrep<Op>::value) {
        const typename Op::PB pb = Op::prep(b[0]);
        Op::template apply_prep_group<G, SA>(a, pb, o, args, err);
    } else if constexpr (SB && HasGroup<Op>::value) {
        Op::template apply_group<G, SA>(a, b[0], o, args, err);
    } else if constexpr (HasPack<Op>::value && G % 4 == 0) {
        if constexpr (SA || SB) {
            typename Op::In ta[G], tb[G];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                ta[k] = a[SA ? 0 : k];
                tb[k] = b[SB ? 0 : k];
            }
            Op::template apply_pack<G>(ta, tb, o);
        } else {
            Op::template apply_pack<G>(a, b, o);
        }
    } else {
#pragma unroll
        for (int k = 0; k < G; ++k) o[k] = Op::apply(a[SA ? 0 : k], b[SB ? 0 : k], args, err);
    }
}

// Everything a kernel needs, passed by value.
struct KArgs {
    const void *A;
    const void *B;
    const void *C;       // three-input kernels only
    void *out;
    int64_t numel;
    OpArgs args;
    uint32_t *status;
};

// ---------------------------------------------------------------- invariant division
// n / d for 0 <= n < 2^32 and 1 <= d < 2^32 with one multiply-high, a
// subtract, an add and two shifts: the unsigned method of Granlund and
// Montgomery, "Division by invariant integers using multiplication" (PLDI
// 1994), section 4: l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
// q = (t + ((n - t) >> min(l,1))) >> max(l-1,0) with t = mulhi(m, n).
struct FastDiv {
    uint32_t m;
    uint32_t s1;
    uint32_t s2;
};

inline FastDiv make_fastdiv(uint64_t d) {
    FastDiv f{1, 0, 0};
    if (d == 0 || d >= (1ull << 32)) return f;  // unused: the wide path divides directly
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
    f.s1 = l < 1 ? l : 1;
    f.s2 = l > 0 ? l - 1 : 0;
    return f;
}

__device__ __forceinline__ uint32_t fastdiv(uint32_t n, const FastDiv &f) {
    const uint32_t t = __umulhi(f.m, n);
    return (t + ((n - t) >> f.s1)) >> f.s2;
}

// q = n / d; 32-bit fast path unless `wide` (some index may reach 2^32).
__device__ __forceinline__ int64_t udiv(int64_t n, int64_t d, const FastDiv &f, bool wide) {
    if (!wide) return (int64_t)fastdiv((uint32_t)n, f);
    return n / d;
}

// ---------------------------------------------------------------- Contiguous
// One tile of kThreads*U groups of G elements per CTA; a ragged tail of
// numel % G elements is finished element by element.
template <class Op, int U>
__global__ void __launch_bounds__(kThreads) k_contiguous(KArgs p) {
    pdl_enter();
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BV = typename Op::BV;
    using BIn = typename BInOf<Op>::type;
    static_assert(!Op::kPlainB || std::is_same_v<BIn, In>, "packed B shares A's type");
    constexpr int G = 16 / sizeof(In);
    const In *A = static_cast<const In *>(p.A);
    const BIn *B = static_cast<const BIn *>(p.B);
    Out *O = static_cast<Out *>(p.out);
    const int64_t ng = p.numel / G;
    uint32_t err = 0;
    const int64_t step = (int64_t)gridDim.x * (kThreads * U);
    for (int64_t base = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x; base < ng;
         base += step) {
        Pack<In, G> a[U];
        Pack<In, G> bp[U];   // plain B: one 16-byte pack per group
        BV bv[Op::kPlainB ? 1 : U][G];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) {
                a[u] = ld_stream<In, G>(A + g * G);
                if constexpr (Op::kPlainB) {
                    bp[u] = ld_stream<In, G>(B + g * G);
                } else {
#pragma unroll
                    for (int k = 0; k < G; ++k) bv[u][k] = Op::loadB(B, g * G + k, p.args);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) {
                Pack<Out, G> o;
                if constexpr (Op::kPlainB) compute_group<Op, G>(a[u].v, bp[u].v, o.v, p.args, err);
                else compute_group<Op, G>(a[u].v, bv[u], o.v, p.args, err);
                st_stream<Out, G>(O + g * G, o);
            }
        }
    }
    for (int64_t e = ng * G + (int64_t)blockIdx.x * kThreads + threadIdx.x; e < p.numel;
         e += (int64_t)gridDim.x * kThreads)
        O[e] = Op::apply(A[e], Op::loadB(B, e, p.args), p.args, err);
    flush_err<Op>(p.status, err);
}

// ---------------------------------------------------------------- Left / right scalar
// SCALAR_A: A is the single value (left scalar); otherwise B is (right scalar).
// The scalar is read once per thread (a warp-uniform address) and kept in
// registers; operand order is preserved.
template <class Op, bool SCALAR_A, int U>
__global__ void __launch_bounds__(kThreads) k_scalar(KArgs p) {
    pdl_enter();
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BV = typename Op::BV;
    using BIn = typename BInOf<Op>::type;
    static_assert(!SCALAR_A || std::is_same_v<BIn, In>, "a left scalar B shares A's type");
    constexpr int G = 16 / sizeof(In);
    const In *A = static_cast<const In *>(p.A);
    const BIn *B = static_cast<const BIn *>(p.B);
    Out *O = static_cast<Out *>(p.out);
    const In *D = SCALAR_A ? static_cast<const In *>(p.B) : A;
    In sa{};
    BV sb{};
    if constexpr (SCALAR_A) sa = A[0];
    else sb = Op::loadB(B, 0, p.args);
    // a right scalar that the operator can prepare is prepared once per thread
    using PrepT = typename std::conditional_t<HasPrep<Op>::value, Op, PrepNone>::PB;
    PrepT pb{};
    if constexpr (!SCALAR_A && HasPrep<Op>::value) pb = Op::prep(sb);
    const int64_t ng = p.numel / G;
    uint32_t err = 0;
    const int64_t step = (int64_t)gridDim.x * (kThreads * U);
    for (int64_t base = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x; base < ng;
         base += step) {
        Pack<In, G> d[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) d[u] = ld_stream<In, G>(D + g * G);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) {
                Pack<Out, G> o;
                if constexpr (SCALAR_A) {
                    compute_group<Op, G, true, false>(&sa, d[u].v, o.v, p.args, err);
                } else if constexpr (HasPrep<Op>::value) {
                    Op::template apply_prep_group<G, false>(d[u].v, pb, o.v, p.args, err);
                } else {
                    compute_group<Op, G, false, true>(d[u].v, &sb, o.v, p.args, err);
                }
                st_stream<Out, G>(O + g * G, o);
            }
        }
    }
    for (int64_t e = ng * G + (int64_t)blockIdx.x * kThreads + threadIdx.x; e < p.numel;
         e += (int64_t)gridDim.x * kThreads) {
        if constexpr (SCALAR_A) O[e] = Op::apply(sa, D[e], p.args, err);
        else O[e] = Op::apply(D[e], sb, p.args, err);
    }
    flush_err<Op>(p.status, err);
}

// ---------------------------------------------------------------- Row traversal
//
// The coalesced dims split into: prefix digits (dims 0..rank-3), the run dim
// (rank-2, extent M, strides smA/smB) and the inner row (rank-1, L elements =
// cols groups of G).  A CTA of tpr*rs threads handles one tile:
// (prefix index, run index, column chunk).  rs rows advance in parallel; each
// thread covers V column groups of its rows (tpr groups apart, so a warp's
// accesses stay contiguous) and walks kr of its rows, rs apart.
struct RowArgs {
    int64_t L;            // inner elements per row
    int64_t cols;         // groups per row = L / G
    int64_t M;            // extent of the run dim (1 for rank-1 plans)
    int64_t smA, smB;     // A and B strides along the run dim
    int64_t ia, ib;       // inner element strides (general kernel)
    int64_t smC, ic;      // the same for a third input (three-input kernels)
    int32_t tpr;          // threads per row
    int32_t rs;           // rows in parallel (threads = tpr * rs)
    int32_t kr;           // rows per thread per tile
    int32_t wide;         // an index may reach 2^32: divide in 64 bits
    int64_t cc;           // column chunks per row = ceil(cols / (tpr * V))
    int64_t runs;         // run tiles per prefix index = ceil(M / (rs * kr))
    int32_t nprefix;      // prefix digits (rank - 2, at least 0)
    int32_t pack_ok;      // rows are a whole number of V*G packs: pack stores stay aligned
    int64_t pn[kMaxRank];
    int64_t psa[kMaxRank];
    int64_t psb[kMaxRank];
    int64_t psc[kMaxRank];
    FastDiv f_cc, f_runs, f_tpr, f_rs;
    FastDiv f_pn[kMaxRank];
};

// IA / IB: 1 = the operand advances along the row (vector loads), 0 = it is
// constant along the row (one value per row), 2 = any inner stride (G == 1).
// NOPREFIX: rank <= 2, no prefix digits to decode.  V: column groups per
// thread per row.  PACKED: the V groups are adjacent and their outputs form
// one store of V*G*sizeof(Out) <= 16 bytes (outputs narrower than inputs,
// e.g. comparisons writing BOOL); otherwise they are tpr groups apart.
// Pointers advance by constant steps from row to row.
template <class Op, int G, int IA, int IB, bool NOPREFIX, int V, bool PACKED>
__global__ void __launch_bounds__(kThreads) k_rows(KArgs p, RowArgs r) {
    pdl_launch();
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BV = typename Op::BV;
    static_assert(G == 1 || (IA != 2 && IB != 2), "runtime inner strides need G == 1");
    static_assert(!PACKED || V * G * (int)sizeof(Out) <= 16, "packed output fits one store");
    constexpr bool kVecA = IA == 1 && G > 1;
    constexpr bool kVecB = IB == 1 && G > 1;
    constexpr bool kBElem = kVecB && !Op::kPlainB;   // per-element parameter blocks

    const int t = threadIdx.x;
    if (t >= r.tpr * r.rs) return;
    const bool wide = r.wide != 0;
    // tile -> (prefix index, run index, column chunk), the column chunk fastest
    const int64_t tile = blockIdx.x;
    const int64_t q1 = udiv(tile, r.cc, r.f_cc, wide);
    const int64_t ci = tile - q1 * r.cc;
    const int64_t pi = udiv(q1, r.runs, r.f_runs, wide);
    const int64_t ri = q1 - pi * r.runs;
    const int rsub = r.rs == 1 ? 0 : (int)fastdiv((uint32_t)t, r.f_tpr);
    const int64_t lane = ci * (int64_t)r.tpr + (t - rsub * r.tpr);
    // first column group of this thread, and the distance between its groups
    const int64_t c0 = PACKED ? lane * V : lane + (ci * (int64_t)r.tpr) * (V - 1);
    const int64_t cstep = PACKED ? 1 : r.tpr;
    if (c0 >= r.cols) return;
    const int64_t m0 = ri * (int64_t)(r.rs * r.kr) + rsub;
    if (m0 >= r.M) return;
    bool ok[V];
#pragma unroll
    for (int v = 0; v < V; ++v) ok[v] = c0 + v * cstep < r.cols;

    int64_t baseA = 0, baseB = 0;
    if constexpr (!NOPREFIX) {
        int64_t rem = pi;
#pragma unroll
        for (int d = kMaxRank - 1; d >= 0; --d) {
            if (d < r.nprefix) {
                const int64_t q = udiv(rem, r.pn[d], r.f_pn[d], wide);
                const int64_t digit = rem - q * r.pn[d];
                rem = q;
                baseA += digit * r.psa[d];
                baseB += digit * r.psb[d];
            }
        }
    }
    // element distance between the thread's groups v and v+1
    const int64_t vstepA = IA == 1 ? cstep * G : IA == 2 ? cstep * r.ia : 0;
    const int64_t vstepB = IB == 1 ? cstep * G : IB == 2 ? cstep * r.ib : 0;
    const int64_t vstepO = cstep * G;
    const In *pa = static_cast<const In *>(p.A) + baseA + m0 * r.smA +
                   (IA == 1 ? c0 * G : IA == 2 ? c0 * r.ia : 0);
    using BIn = typename BInOf<Op>::type;
    const BIn *pb = static_cast<const BIn *>(p.B) + baseB + m0 * r.smB +
                    (IB == 1 ? c0 * G : IB == 2 ? c0 * r.ib : 0);
    Out *po = static_cast<Out *>(p.out) + (pi * r.M + m0) * r.L + c0 * G;
    const int64_t stepA = (int64_t)r.rs * r.smA;
    const int64_t stepB = (int64_t)r.rs * r.smB;
    const int64_t stepO = (int64_t)r.rs * r.L;
    // this thread's rows in the run: ceil((M - m0) / rs), at most kr
    const int64_t rows_left = r.M - m0 + r.rs - 1;
    const int64_t left = wide ? rows_left / r.rs : (int64_t)fastdiv((uint32_t)rows_left, r.f_rs);
    const int n = (int)(left < r.kr ? left : r.kr);

    // Dense operands stay 16-byte packs; an operand constant along the row is
    // one value.  An operand whose run stride is 0 is read once and kept.
    using APack = std::conditional_t<kVecA, Pack<In, G>, Pack<In, 1>>;
    using BPack = std::conditional_t<kVecB && Op::kPlainB, Pack<In, G>, Pack<BV, kBElem ? G : 1>>;
    constexpr int VA = (IA == 0) ? 1 : V;   // a row-constant operand is the same for all v
    constexpr int VB = (IB == 0) ? 1 : V;
    const bool reloadA = stepA != 0, reloadB = stepB != 0;
    auto load_a = [&](const In *q) {
        APack x;
        if constexpr (kVecA) x = ld_stream<In, G>(q);
        else x.v[0] = *q;
        return x;
    };
    auto load_b = [&](const BIn *q) {
        BPack x;
        if constexpr (kVecB && Op::kPlainB) {
            x = ld_stream<In, G>(q);
        } else if constexpr (kBElem) {
#pragma unroll
            for (int k = 0; k < G; ++k) x.v[k] = Op::loadB(q, k, p.args);
        } else {
            x.v[0] = Op::loadB(q, 0, p.args);
        }
        return x;
    };
    APack a[VA];
    BPack b[VB];
    uint32_t err = 0;
    pdl_wait();   // the index arithmetic above touched no global memory
    // Not unrolled: an unrolled row loop holds two rows' registers (64 against
    // 40 for bf16 Add), costing a third of the resident CTAs (per-channel bf16
    // Add 25.9 -> 22.6 us, Greater fp16 -> BOOL 149 -> 141 us on GB300).
#pragma unroll 1
    for (int j = 0; j < n; ++j) {
        if (j == 0 || reloadA) {
#pragma unroll
            for (int v = 0; v < VA; ++v)
                if (ok[v]) a[v] = load_a(pa + v * vstepA);
        }
        if (j == 0 || reloadB) {
#pragma unroll
            for (int v = 0; v < VB; ++v)
                if (ok[v]) b[v] = load_b(pb + v * vstepB);
        }
        if constexpr (PACKED) {
            Pack<Out, V * G> o;
#pragma unroll
            for (int v = 0; v < V; ++v)
                compute_group<Op, G, !kVecA, !kVecB>(a[IA == 0 ? 0 : v].v, b[IB == 0 ? 0 : v].v,
                                                    o.v + v * G, p.args, err);
            if (r.pack_ok && ok[V - 1]) {
                st_stream<Out, V * G>(po, o);
            } else {
                // rows that are not a whole number of packs: one aligned store per group
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    if (ok[v]) {
                        Pack<Out, G> og;
#pragma unroll
                        for (int k = 0; k < G; ++k) og.v[k] = o.v[v * G + k];
                        st_stream<Out, G>(po + v * G, og);
                    }
                }
            }
        } else {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (ok[v]) {
                    Pack<Out, G> o;
                    compute_group<Op, G, !kVecA, !kVecB>(a[IA == 0 ? 0 : v].v,
                                                        b[IB == 0 ? 0 : v].v, o.v, p.args, err);
                    if constexpr (G > 1) st_stream<Out, G>(po + v * vstepO, o);
                    else po[v * vstepO] = o.v[0];
                }
            }
        }
        pa += stepA;
        pb += stepB;
        po += stepO;
    }
    flush_err<Op>(p.status, err);
}

// ---------------------------------------------------------------- short rows
//
// Plans whose rows are short or off the 16-byte pack width: a channels-last
// per-channel operand of 3 or 4 channels, rows of 13, and the general shapes
// [a, 1, k] x [1, b, k] and [a, 1] x [1, k] with small k.  The output is
// streamed flat in packs of G elements, as in k_scalar.  After coalescing the
// plan is [n0,] n1, n2: an optional outer index over blocks of Lb = n1 n2
// elements, and in each block rows of P = n2.  For output element e, with
// (i0, f) = (e / Lb, e mod Lb) and (q, r) = (f / P, f mod P), each input is
// read at i0 s0 + one of
//   DENSE     f   (dense within the block; read in 16-byte packs),
//   ROWVAL    q   (one value per row),
//   ROWBLOCK  r   (one row of P values reused by every row).
// The position (i0, f, q, r) is decoded once per pack and stepped with
// selects; a pack never crosses a block (Lb is a multiple of G when there is
// an outer index).  Indices are 32-bit: the launcher sends plans of 2^31
// elements or more to the row kernel.
enum PMode { PM_DENSE = 0, PM_ROWVAL = 1, PM_ROWBLOCK = 2 };

struct PeriodicArgs {
    int32_t P;          // row length (innermost extent)
    int32_t Lb;         // block length (numel when there is no outer index)
    int32_t sa0, sb0;   // A's and B's element strides along the outer index
    FastDiv fP, fLb;
};

template <class Op, int MA, int MB, int U>
__global__ void __launch_bounds__(kThreads) k_periodic(KArgs p, PeriodicArgs a) {
    pdl_launch();
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BIn = typename BInOf<Op>::type;
    using BV = typename Op::BV;
    static_assert(!(MA == PM_DENSE && MB == PM_DENSE), "one input at least repeats");
    static_assert(MB != PM_DENSE || Op::kPlainB, "a dense B is read in packs of A's type");
    constexpr int G = 16 / sizeof(In);
    const In *A = static_cast<const In *>(p.A);
    const BIn *B = static_cast<const BIn *>(p.B);
    Out *O = static_cast<Out *>(p.out);
    const int64_t ng = p.numel / G;
    const int64_t step = (int64_t)gridDim.x * (kThreads * U);
    uint32_t err = 0;
    // offsets of element e = i0 Lb + f
    auto decode = [&](int32_t e, int32_t &i0, int32_t &f) {
        i0 = (int32_t)fastdiv((uint32_t)e, a.fLb);
        f = e - i0 * a.Lb;
    };
    pdl_wait();
    for (int64_t base = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x; base < ng;
         base += step) {
        Pack<In, G> da[MA == PM_DENSE ? U : 1];
        Pack<In, G> db[MB == PM_DENSE ? U : 1];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) {
                int32_t i0, f;
                decode((int32_t)(g * G), i0, f);
                if constexpr (MA == PM_DENSE) da[u] = ld_stream<In, G>(A + i0 * a.sa0 + f);
                if constexpr (MB == PM_DENSE)
                    db[u] = ld_stream<In, G>(reinterpret_cast<const In *>(B) + i0 * a.sb0 + f);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) {
                const int32_t e0 = (int32_t)(g * G);
                int32_t i0, f;
                decode(e0, i0, f);
                int32_t q = (int32_t)fastdiv((uint32_t)f, a.fP);
                int32_t r = f - q * a.P;
                const In *pa = A + i0 * a.sa0;
                const BIn *pb = B + i0 * a.sb0;
                Pack<Out, G> o;
#pragma unroll
                for (int k = 0; k < G; ++k) {
                    In xa;
                    if constexpr (MA == PM_DENSE) xa = da[u].v[k];
                    else xa = pa[MA == PM_ROWVAL ? q : r];
                    BV xb;
                    if constexpr (MB == PM_DENSE) xb = db[u].v[k];
                    else xb = Op::loadB(pb, MB == PM_ROWVAL ? q : r, p.args);
                    o.v[k] = Op::apply(xa, xb, p.args, err);
                    const bool wrap = ++r == a.P;
                    r = wrap ? 0 : r;
                    q += wrap ? 1 : 0;
                }
                st_stream<Out, G>(O + e0, o);
            }
        }
    }
    // the last numel % G elements, one by one
    for (int64_t e = ng * G + (int64_t)blockIdx.x * kThreads + threadIdx.x; e < p.numel;
         e += (int64_t)gridDim.x * kThreads) {
        int32_t i0, f;
        decode((int32_t)e, i0, f);
        const int32_t q = (int32_t)fastdiv((uint32_t)f, a.fP);
        const int32_t r = f - q * a.P;
        const int32_t oa = i0 * a.sa0 + (MA == PM_DENSE ? f : MA == PM_ROWVAL ? q : r);
        const int32_t ob = i0 * a.sb0 + (MB == PM_DENSE ? f : MB == PM_ROWVAL ? q : r);
        O[e] = Op::apply(A[oa], Op::loadB(B, ob, p.args), p.args, err);
    }
    flush_err<Op>(p.status, err);
}

// ---------------------------------------------------------------- a short row reused in blocks
//
// The k_periodic pattern with one input X a row of P <= kBlockRowMaxP values
// reused by every row of a block (ROWBLOCK) and the other, D, dense in the
// block: [a, 1, k] x [1, b, k], [n, k] x [k].  The 16-byte pack of X that an
// output pack needs depends only on the row position r0 = f mod P where the
// pack starts, so each CTA first lays out in shared memory, for the (at most
// two) blocks its tile touches, the P rotations of the row:
//   pat[s][r0][j] = X[(i0 + s) sx0 + (r0 + j) mod P],  j < G,
// behind one barrier; then each output pack is one 16-byte shared load of X,
// one 16-byte load of D and one 16-byte store.  One tile of kThreads x U
// packs per CTA; a block holds at least that many elements (the launcher
// checks), so a tile spans at most two blocks.  X_IS_A: X is A (else B).
constexpr int kBlockRowMaxP = 32;

struct BlockRowArgs {
    int32_t P;          // row length
    int32_t Lb;         // block length, a multiple of P (numel when there is no outer index)
    int32_t n0;         // blocks
    int32_t sx0, sd0;   // X's and D's element strides along the outer index
    int32_t dr;         // (kThreads * G) mod P: the row position's step between a thread's packs
    FastDiv fP, fLb;
};

template <class Op, bool X_IS_A, int U>
__global__ void __launch_bounds__(kThreads) k_blockrow(KArgs p, BlockRowArgs a) {
    pdl_launch();
    using In = typename Op::In;
    using Out = typename Op::Out;
    static_assert(Op::kPlainB, "both inputs are plain tensors of one type");
    constexpr int G = 16 / sizeof(In);
    __shared__ Pack<In, G> pat[2][kBlockRowMaxP];
    const In *X = static_cast<const In *>(X_IS_A ? p.A : p.B);
    const In *D = static_cast<const In *>(X_IS_A ? p.B : p.A);
    Out *O = static_cast<Out *>(p.out);
    const int64_t ng = p.numel / G;
    const int64_t tile0 = (int64_t)blockIdx.x * (kThreads * U);
    // the tile's first block ib; packs from pb on lie in block ib + 1 (Lb is a
    // multiple of G when there is an outer index; else pb >= ng)
    const int32_t ib = (int32_t)fastdiv((uint32_t)(tile0 * G), a.fLb);
    const int64_t pb = (int64_t)(ib + 1) * a.Lb / G;
    // D's element index of output element e in block i0 is i0 (sd0 - Lb) + e
    const int64_t off0 = (int64_t)ib * (a.sd0 - a.Lb), off1 = off0 + (a.sd0 - a.Lb);
    pdl_wait();
    // the rotations of the row of blocks ib and ib + 1
    for (int idx = threadIdx.x; idx < 2 * a.P * G; idx += kThreads) {
        const int s = idx / (a.P * G), rem = idx - s * (a.P * G);
        const int r0 = rem / G, j = rem - r0 * G;
        if (ib + s < a.n0) {
            int rj = r0 + j;
            while (rj >= a.P) rj -= a.P;   // (r0 + j) mod P, at most G / P + 1 steps
            pat[s][r0].v[j] = X[(ib + s) * a.sx0 + rj];
        }
    }
    __syncthreads();
    uint32_t err = 0;
    Pack<In, G> d[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t g = tile0 + (int64_t)u * kThreads + threadIdx.x;
        if (g < ng) d[u] = ld_stream<In, G>(D + ((g >= pb ? off1 : off0) + g * G));
    }
    // the row position of the thread's first pack (Lb is a multiple of P, so
    // it does not depend on the block), then stepped by dr from pack to pack
    const int32_t e_first = (int32_t)((tile0 + threadIdx.x) * G);
    int32_t r = e_first - (int32_t)fastdiv((uint32_t)e_first, a.fP) * a.P;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t g = tile0 + (int64_t)u * kThreads + threadIdx.x;
        if (g < ng) {
            const Pack<In, G> x = pat[g >= pb ? 1 : 0][r];
            Pack<Out, G> o;
            if constexpr (X_IS_A) compute_group<Op, G>(x.v, d[u].v, o.v, p.args, err);
            else compute_group<Op, G>(d[u].v, x.v, o.v, p.args, err);
            st_stream<Out, G>(O + g * G, o);
        }
        r += a.dr;
        r -= r >= a.P ? a.P : 0;
    }
    // the last numel % G elements, one per thread (rank-2 plans only: with an
    // outer index the element count is a multiple of G)
    for (int64_t e = ng * G + (int64_t)blockIdx.x * kThreads + threadIdx.x; e < p.numel;
         e += (int64_t)gridDim.x * kThreads) {
        const int32_t i0 = (int32_t)fastdiv((uint32_t)e, a.fLb);
        const int32_t f = (int32_t)e - i0 * a.Lb;
        const int32_t rr = f - (int32_t)fastdiv((uint32_t)f, a.fP) * a.P;
        const In xv = X[i0 * a.sx0 + rr], dv = D[i0 * a.sd0 + f];
        O[e] = X_IS_A ? Op::apply(xv, dv, p.args, err) : Op::apply(dv, xv, p.args, err);
    }
    flush_err<Op>(p.status, err);
}

// ---------------------------------------------------------------- rows with one value each
//
// Inner-vector / repeated-block plans whose dense input covers the whole output
// in order (x[N, C, H, W] against a per-channel operand, [M, L] against
// [M, 1]) and whose other input is one value per row of L elements, L a
// multiple of the pack width G.  The rows are not walked one by one: the
// output is streamed flat, and each CTA takes `iters` consecutive runs of
// kThreads x U packs (one contiguous chunk), so that a thread meets few row
// boundaries.  A thread keeps the value of its current row (the parameters,
// prepared where the operator prepares them) and reloads it only when a pack
// lies outside that row; the row value's offset is decoded from the row
// index only then.  A run whose packs all lie in bounds and in the cached row
// (nearly every run) takes no per-pack test.  ROW_A: A is the per-row input
// and B the dense one.  WIDE: pack indices are 64-bit and divide in 64 bits
// (the launcher takes it when some run start would reach 2^31 packs); else
// they are 32-bit.
struct RowConstArgs {
    int64_t lp;                 // packs per row (L / G)
    FastDiv f_lp;
    int32_t nd;                 // outer dims (everything but the inner row)
    int32_t iters;              // runs of kThreads x U packs per CTA
    int64_t on[kMaxRank];       // outer extents, outermost first
    int64_t os[kMaxRank];       // the per-row input's strides along them
    FastDiv f_on[kMaxRank];
};

// The smallest number of resident CTAs per SM asked of the compiler for an
// operator's k_rowconst (0: none asked).  Measured on GB300, bf16
// x[8,64,256,256] against a per-channel operand: BiasPReluBN takes 66
// registers unbounded (three CTAs per SM, 25.9 us) and 53 when asked for four
// (24.1 us), BatchNormalization 22.6 -> 22.3 us; Add 21.0 -> 20.7 us and fp32
// Mod rows 21.7 -> 21.5 us asked for one, while PRelu and BiasPRelu lose 10%
// when asked for one (20.8 -> 22.9 us), so they ask nothing.
template <class Op> struct RowConstMinCtas : std::integral_constant<int, HasGroup<Op>::value ? 4 : 0> {};
template <class T, int K> struct RowConstMinCtas<OpArith<T, K>> : std::integral_constant<int, 1> {};
template <class T> struct RowConstMinCtas<OpMod<T>> : std::integral_constant<int, 1> {};

template <class Op, bool ROW_A, int U, bool WIDE>
__device__ __forceinline__ void rowconst_body(const KArgs &p, const RowConstArgs &r) {
    pdl_launch();
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BV = typename Op::BV;
    using BIn = typename BInOf<Op>::type;
    // pack indices: 32-bit unless a run start of the launch reaches 2^31 packs
    using I = std::conditional_t<WIDE, int64_t, int32_t>;
    constexpr int G = 16 / sizeof(In);
    constexpr bool kPrep = !ROW_A && HasPrep<Op>::value;
    using PrepT = typename std::conditional_t<HasPrep<Op>::value, Op, PrepNone>::PB;
    using RowV = std::conditional_t<ROW_A, In, std::conditional_t<kPrep, PrepT, BV>>;
    const In *D = ROW_A ? static_cast<const In *>(p.B) : static_cast<const In *>(p.A);
    const In *RA = static_cast<const In *>(p.A);
    const BIn *RB = static_cast<const BIn *>(p.B);
    Out *O = static_cast<Out *>(p.out);
    const I np = (I)(p.numel / G);
    const I lp = (I)r.lp;
    const I first = (I)blockIdx.x * (I)r.iters * (I)(kThreads * U) + (I)threadIdx.x;
    // packs [lo, hi) are the row whose value rv holds (none yet)
    I lo = 0, hi = 0;
    RowV rv{};
    uint32_t err = 0;
    auto set_row = [&](I g) {   // the row of pack g becomes the cached one
        const int64_t row = udiv(g, r.lp, r.f_lp, WIDE);
        lo = (I)row * lp;
        hi = lo + lp;
        int64_t rem = row, off = 0;
#pragma unroll
        for (int k = kMaxRank - 1; k >= 0; --k) {
            if (k < r.nd) {
                const int64_t q = udiv(rem, r.on[k], r.f_on[k], WIDE);
                off += (rem - q * r.on[k]) * r.os[k];
                rem = q;
            }
        }
        if constexpr (ROW_A) rv = RA[off];
        else if constexpr (kPrep) rv = Op::prep(Op::loadB(RB, off, p.args));
        else rv = Op::loadB(RB, off, p.args);
    };
    pdl_wait();
#pragma unroll 1
    for (int j = 0; j < r.iters; ++j) {
        const I base = first + (I)j * (I)(kThreads * U);
        if (base >= np) break;
        Pack<In, G> d[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const I g = base + (I)(u * kThreads);
            if (g < np) d[u] = ld_stream<In, G>(D + (int64_t)g * G);
        }
        // the loads are in flight: bring the row of the run's first pack in
        if (base < lo || base >= hi) set_row(base);
        const I last = base + (I)((U - 1) * kThreads);
        if (last < np && last < hi) {
            // the common run: every pack in bounds and in the cached row, so
            // no per-pack test, and the stores are one base plus constants
            Out *dst = O + (int64_t)base * G;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                Pack<Out, G> o;
                if constexpr (ROW_A) compute_group<Op, G, true, false>(&rv, d[u].v, o.v, p.args, err);
                else if constexpr (kPrep)
                    Op::template apply_prep_group<G, false>(d[u].v, rv, o.v, p.args, err);
                else compute_group<Op, G, false, true>(d[u].v, &rv, o.v, p.args, err);
                st_stream<Out, G>(dst + u * kThreads * G, o);
            }
            continue;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const I g = base + (I)(u * kThreads);
            if (g < np) {
                if (g < lo || g >= hi) set_row(g);
                Pack<Out, G> o;
                if constexpr (ROW_A) compute_group<Op, G, true, false>(&rv, d[u].v, o.v, p.args, err);
                else if constexpr (kPrep)
                    Op::template apply_prep_group<G, false>(d[u].v, rv, o.v, p.args, err);
                else compute_group<Op, G, false, true>(d[u].v, &rv, o.v, p.args, err);
                st_stream<Out, G>(O + (int64_t)g * G, o);
            }
        }
    }
    flush_err<Op>(p.status, err);
}

template <class Op, bool ROW_A, int U, bool WIDE>
__global__ void __launch_bounds__(kThreads) k_rowconst(KArgs p, RowConstArgs r) {
    rowconst_body<Op, ROW_A, U, WIDE>(p, r);
}

template <class Op, bool ROW_A, int U, bool WIDE, int MINCTAS>
__global__ void __launch_bounds__(kThreads, MINCTAS) k_rowconst_bounded(KArgs p, RowConstArgs r) {
    rowconst_body<Op, ROW_A, U, WIDE>(p, r);
}

// ---------------------------------------------------------------- a transposed input
//
// GENERAL_STRIDED plans of rank 2 whose one input is dense (strides (N, 1))
// and whose other is a transposed view (strides (1, ld)): output element
// (i, j) reads D[i N + j] and T[i + j ld].  Along the output's rows T is a
// gather with stride ld.  Each CTA instead takes one square tile of TW x TW
// elements: it reads T's part along T's contiguous direction into shared
// memory (rows padded by one element, so that reading it across rows spreads
// over the banks), then walks the output tile along its rows with coalesced
// loads of D and stores.  T_IS_B: B is the transposed input (else A).
//
// Measured on GB300 (Add fp32 [8192,8192] + a transposed [8192,8192] view;
// the row traversal takes 271 us, 0.445 of the measured copy): tiles of 32
// elements 203 us, of 64 elements 183 us (0.66), of 128 bf16 elements 0.25
// against 0.36 at 64; tall tiles (1 KB runs of T by 16 or 32 columns) 206-255
// us, and a diagonal tile order changed nothing, also at 8000 x 8000.  Tiles
// wholly inside the output without bounds tests and with stepped addresses:
// 168 us (0.72), bf16 Mul 167 -> 145 us (0.42).
struct TransArgs {
    int64_t M, N;        // output rows and columns
    int64_t ld;          // the transposed input: element (i, j) at i + j * ld
    uint32_t tiles_n;    // tiles across the output's columns
};

constexpr int kTransTile = 64;         // TW

template <int B> struct BitsOf;
template <> struct BitsOf<1> { using type = uint8_t; };
template <> struct BitsOf<2> { using type = uint16_t; };
template <> struct BitsOf<4> { using type = uint32_t; };
template <> struct BitsOf<8> { using type = uint64_t; };

template <class Op, bool T_IS_B>
__global__ void __launch_bounds__(kThreads) k_transposed(KArgs p, TransArgs a) {
    pdl_launch();
    using In = typename Op::In;
    using Out = typename Op::Out;
    using S = typename BitsOf<sizeof(In)>::type;   // the tile holds raw element bits
    constexpr int TW = kTransTile;
    constexpr int RP = kThreads / TW;              // tile rows per pass of the CTA
    static_assert(TW * RP == kThreads && TW % RP == 0, "tile shape");
    __shared__ S tile[TW][TW + 1];
    static_assert(sizeof(tile) <= 48 * 1024, "static shared memory");
    const int tx = (int)threadIdx.x % TW, ty = (int)threadIdx.x / TW;
    const uint32_t bi = blockIdx.x / a.tiles_n, bj = blockIdx.x - bi * a.tiles_n;
    const int64_t i0 = (int64_t)bi * TW, j0 = (int64_t)bj * TW;
    const In *T = static_cast<const In *>(T_IS_B ? p.B : p.A);
    const In *D = static_cast<const In *>(T_IS_B ? p.A : p.B);
    Out *O = static_cast<Out *>(p.out);
    uint32_t err = 0;
    // a tile wholly inside the output takes no bounds test, and each pass
    // steps its addresses from one base
    const bool whole = i0 + TW <= a.M && j0 + TW <= a.N;
    pdl_wait();
    // tile[c][r] = T(i0 + r, j0 + c), read along r (T's contiguous direction)
    if (whole) {
        const In *tp = T + (i0 + tx) + (j0 + ty) * a.ld;
        const int64_t step = (int64_t)RP * a.ld;
#pragma unroll
        for (int k = 0; k < TW / RP; ++k) {
            const In t = tp[k * step];
            memcpy(&tile[ty + k * RP][tx], &t, sizeof(S));
        }
    } else {
#pragma unroll
        for (int c = ty; c < TW; c += RP) {
            const int64_t i = i0 + tx, j = j0 + c;
            if (i < a.M && j < a.N) {
                const In t = T[i + j * a.ld];
                memcpy(&tile[c][tx], &t, sizeof(S));
            }
        }
    }
    __syncthreads();
    if (whole) {
        const int64_t base = (i0 + ty) * a.N + (j0 + tx), step = (int64_t)RP * a.N;
        const In *dp = D + base;
        Out *op = O + base;
#pragma unroll
        for (int k = 0; k < TW / RP; ++k) {
            In t;
            memcpy(&t, &tile[tx][ty + k * RP], sizeof(S));
            const In d = dp[k * step];
            op[k * step] = T_IS_B ? Op::apply(d, t, p.args, err) : Op::apply(t, d, p.args, err);
        }
    } else {
#pragma unroll
        for (int r = ty; r < TW; r += RP) {
            const int64_t i = i0 + r, j = j0 + tx;
            if (i < a.M && j < a.N) {      // the same (i, j) the first pass loaded
                In t;
                memcpy(&t, &tile[tx][r], sizeof(S));
                const In d = D[i * a.N + j];
                O[i * a.N + j] = T_IS_B ? Op::apply(d, t, p.args, err) : Op::apply(t, d, p.args, err);
            }
        }
    }
    flush_err<Op>(p.status, err);
}

// ---------------------------------------------------------------- three inputs, one value per row
//
// k_rowconst for a three-input operator (Op::apply3): two inputs dense over
// the output in order and the third, operand RP (0 = a, 1 = b, 2 = c), one
// value per row of L elements, L a multiple of the pack width G (MulAdd with
// a per-channel multiplier: x[N, C, H, W] * s[1, C, 1, 1] + y).  The same flat
// stream of runs, cached row value and common run as k_rowconst.
template <class Op, int RP, int U, bool WIDE>
__global__ void __launch_bounds__(kThreads) k_rowconst3(KArgs p, RowConstArgs r) {
    pdl_launch();
    using In = typename Op::In;
    using Out = typename Op::Out;
    using I = std::conditional_t<WIDE, int64_t, int32_t>;
    constexpr int G = 16 / sizeof(In);
    const In *A = static_cast<const In *>(p.A);
    const In *B = static_cast<const In *>(p.B);
    const In *C = static_cast<const In *>(p.C);
    const In *D0 = RP == 0 ? B : A;             // the dense inputs, in operand order
    const In *D1 = RP == 2 ? B : C;
    const In *R = RP == 0 ? A : RP == 1 ? B : C;
    Out *O = static_cast<Out *>(p.out);
    const I np = (I)(p.numel / G);
    const I lp = (I)r.lp;
    const I first = (I)blockIdx.x * (I)r.iters * (I)(kThreads * U) + (I)threadIdx.x;
    I lo = 0, hi = 0;                           // packs [lo, hi): the row rv belongs to
    In rv{};
    auto set_row = [&](I g) {
        const int64_t row = udiv(g, r.lp, r.f_lp, WIDE);
        lo = (I)row * lp;
        hi = lo + lp;
        int64_t rem = row, off = 0;
#pragma unroll
        for (int k = kMaxRank - 1; k >= 0; --k) {
            if (k < r.nd) {
                const int64_t q = udiv(rem, r.on[k], r.f_on[k], WIDE);
                off += (rem - q * r.on[k]) * r.os[k];
                rem = q;
            }
        }
        rv = R[off];
    };
    auto compute = [&](const Pack<In, G> &x, const Pack<In, G> &y, Pack<Out, G> &o) {
#pragma unroll
        for (int k = 0; k < G; ++k) {
            if constexpr (RP == 0) o.v[k] = Op::apply3(rv, x.v[k], y.v[k]);
            else if constexpr (RP == 1) o.v[k] = Op::apply3(x.v[k], rv, y.v[k]);
            else o.v[k] = Op::apply3(x.v[k], y.v[k], rv);
        }
    };
    pdl_wait();
#pragma unroll 1
    for (int j = 0; j < r.iters; ++j) {
        const I base = first + (I)j * (I)(kThreads * U);
        if (base >= np) break;
        Pack<In, G> d0[U], d1[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const I g = base + (I)(u * kThreads);
            if (g < np) {
                d0[u] = ld_stream<In, G>(D0 + (int64_t)g * G);
                d1[u] = ld_stream<In, G>(D1 + (int64_t)g * G);
            }
        }
        // the loads are in flight: bring the row of the run's first pack in
        if (base < lo || base >= hi) set_row(base);
        const I last = base + (I)((U - 1) * kThreads);
        if (last < np && last < hi) {           // the common run: no per-pack test
            Out *dst = O + (int64_t)base * G;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                Pack<Out, G> o;
                compute(d0[u], d1[u], o);
                st_stream<Out, G>(dst + u * kThreads * G, o);
            }
            continue;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const I g = base + (I)(u * kThreads);
            if (g < np) {
                if (g < lo || g >= hi) set_row(g);
                Pack<Out, G> o;
                compute(d0[u], d1[u], o);
                st_stream<Out, G>(O + (int64_t)g * G, o);
            }
        }
    }
}

// ---------------------------------------------------------------- three inputs
//
// The row traversal of k_rows for an operator of three inputs (Op::apply3):
// the same tile (prefix index, run of rows, column chunk), V column groups a
// row-width apart per thread, kr rows walked with constant pointer steps.
// IA / IB / IC: 1 = the input advances along the row (16-byte packs when
// G > 1), 0 = one value per row, 2 = any inner stride (G == 1).
template <class In, int G, int I> struct RowOperand {
    static constexpr bool kVec = I == 1 && G > 1;
    using P = std::conditional_t<kVec, Pack<In, G>, Pack<In, 1>>;
    __device__ __forceinline__ static P load(const In *q) {
        P x;
        if constexpr (kVec) x = ld_stream<In, G>(q);
        else x.v[0] = *q;
        return x;
    }
    __device__ __forceinline__ static In at(const P &x, int k) {
        if constexpr (kVec) return x.v[k];
        else return x.v[0];
    }
    // element distance between column groups cstep apart, and to the first group
    __device__ __forceinline__ static int64_t step(int64_t cstep, int64_t inner) {
        return I == 1 ? cstep * G : I == 2 ? cstep * inner : 0;
    }
};

template <class Op, int G, int IA, int IB, int IC, int V>
__global__ void __launch_bounds__(kThreads) k_rows3(KArgs p, RowArgs r) {
    pdl_launch();
    using In = typename Op::In;
    using Out = typename Op::Out;
    static_assert(G == 1 || (IA != 2 && IB != 2 && IC != 2), "runtime strides need G == 1");
    using OA = RowOperand<In, G, IA>;
    using OB = RowOperand<In, G, IB>;
    using OC = RowOperand<In, G, IC>;

    const int t = threadIdx.x;
    if (t >= r.tpr * r.rs) return;
    const bool wide = r.wide != 0;
    const int64_t tile = blockIdx.x;
    const int64_t q1 = udiv(tile, r.cc, r.f_cc, wide);
    const int64_t ci = tile - q1 * r.cc;
    const int64_t pi = udiv(q1, r.runs, r.f_runs, wide);
    const int64_t ri = q1 - pi * r.runs;
    const int rsub = r.rs == 1 ? 0 : (int)fastdiv((uint32_t)t, r.f_tpr);
    const int64_t lane = ci * (int64_t)r.tpr + (t - rsub * r.tpr);
    const int64_t c0 = lane + (ci * (int64_t)r.tpr) * (V - 1);
    const int64_t cstep = r.tpr;
    if (c0 >= r.cols) return;
    const int64_t m0 = ri * (int64_t)(r.rs * r.kr) + rsub;
    if (m0 >= r.M) return;
    bool ok[V];
#pragma unroll
    for (int v = 0; v < V; ++v) ok[v] = c0 + v * cstep < r.cols;

    int64_t baseA = 0, baseB = 0, baseC = 0;
    int64_t rem = pi;
#pragma unroll
    for (int d = kMaxRank - 1; d >= 0; --d) {
        if (d < r.nprefix) {
            const int64_t q = udiv(rem, r.pn[d], r.f_pn[d], wide);
            const int64_t digit = rem - q * r.pn[d];
            rem = q;
            baseA += digit * r.psa[d];
            baseB += digit * r.psb[d];
            baseC += digit * r.psc[d];
        }
    }
    const int64_t vsA = OA::step(cstep, r.ia), vsB = OB::step(cstep, r.ib),
                  vsC = OC::step(cstep, r.ic);
    const In *pa = static_cast<const In *>(p.A) + baseA + m0 * r.smA + OA::step(c0, r.ia);
    const In *pb = static_cast<const In *>(p.B) + baseB + m0 * r.smB + OB::step(c0, r.ib);
    const In *pc = static_cast<const In *>(p.C) + baseC + m0 * r.smC + OC::step(c0, r.ic);
    Out *po = static_cast<Out *>(p.out) + (pi * r.M + m0) * r.L + c0 * G;
    const int64_t stepA = (int64_t)r.rs * r.smA, stepB = (int64_t)r.rs * r.smB,
                  stepC = (int64_t)r.rs * r.smC, stepO = (int64_t)r.rs * r.L;
    const int64_t rows_left = r.M - m0 + r.rs - 1;
    const int64_t left = wide ? rows_left / r.rs : (int64_t)fastdiv((uint32_t)rows_left, r.f_rs);
    const int n = (int)(left < r.kr ? left : r.kr);

    // an input constant along the row is one value for all v
    constexpr int VA = IA == 0 ? 1 : V, VB = IB == 0 ? 1 : V, VC = IC == 0 ? 1 : V;
    typename OA::P a[VA];
    typename OB::P b[VB];
    typename OC::P c[VC];
    pdl_wait();   // the index arithmetic above touched no global memory
#pragma unroll 1
    for (int j = 0; j < n; ++j) {
        if (j == 0 || stepA != 0) {
#pragma unroll
            for (int v = 0; v < VA; ++v)
                if (ok[v]) a[v] = OA::load(pa + v * vsA);
        }
        if (j == 0 || stepB != 0) {
#pragma unroll
            for (int v = 0; v < VB; ++v)
                if (ok[v]) b[v] = OB::load(pb + v * vsB);
        }
        if (j == 0 || stepC != 0) {
#pragma unroll
            for (int v = 0; v < VC; ++v)
                if (ok[v]) c[v] = OC::load(pc + v * vsC);
        }
#pragma unroll
        for (int v = 0; v < V; ++v) {
            if (ok[v]) {
                Pack<Out, G> o;
#pragma unroll
                for (int k = 0; k < G; ++k)
                    o.v[k] = Op::apply3(OA::at(a[IA == 0 ? 0 : v], k),
                                        OB::at(b[IB == 0 ? 0 : v], k),
                                        OC::at(c[IC == 0 ? 0 : v], k));
                if constexpr (G > 1) st_stream<Out, G>(po + v * cstep * G, o);
                else po[v * cstep] = o.v[0];
            }
        }
        pa += stepA;
        pb += stepB;
        pc += stepC;
        po += stepO;
    }
}

// Three inputs at rank 1: each dense (I = 1, 16-byte packs) or one value (I = 0,
// read once per thread), one tile of kThreads x U groups per CTA as in
// k_contiguous; a ragged tail of numel % G elements element by element.
template <class Op, int IA, int IB, int IC, int U>
__global__ void __launch_bounds__(kThreads) k_flat3(KArgs p) {
    pdl_enter();
    using In = typename Op::In;
    using Out = typename Op::Out;
    constexpr int G = 16 / sizeof(In);
    const In *A = static_cast<const In *>(p.A);
    const In *B = static_cast<const In *>(p.B);
    const In *C = static_cast<const In *>(p.C);
    Out *O = static_cast<Out *>(p.out);
    const In sa = IA == 0 ? A[0] : In{}, sb = IB == 0 ? B[0] : In{}, sc = IC == 0 ? C[0] : In{};
    const int64_t ng = p.numel / G;
    const int64_t base = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x;
    Pack<In, G> a[IA ? U : 1], b[IB ? U : 1], c[IC ? U : 1];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t g = base + (int64_t)u * kThreads;
        if (g < ng) {
            if constexpr (IA) a[u] = ld_stream<In, G>(A + g * G);
            if constexpr (IB) b[u] = ld_stream<In, G>(B + g * G);
            if constexpr (IC) c[u] = ld_stream<In, G>(C + g * G);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t g = base + (int64_t)u * kThreads;
        if (g < ng) {
            Pack<Out, G> o;
#pragma unroll
            for (int k = 0; k < G; ++k)
                o.v[k] = Op::apply3(IA ? a[IA ? u : 0].v[k] : sa, IB ? b[IB ? u : 0].v[k] : sb,
                                    IC ? c[IC ? u : 0].v[k] : sc);
            st_stream<Out, G>(O + g * G, o);
        }
    }
    for (int64_t e = ng * G + (int64_t)blockIdx.x * kThreads + threadIdx.x; e < p.numel;
         e += (int64_t)gridDim.x * kThreads)
        O[e] = Op::apply3(IA ? A[e] : sa, IB ? B[e] : sb, IC ? C[e] : sc);
}

// ---------------------------------------------------------------- launch helpers
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <class Op>
KArgs kargs(const Launch &L) {
    KArgs k;
    k.A = L.A;
    k.B = L.B;
    k.C = L.C;
    k.out = L.out;
    k.numel = L.numel;
    k.args = L.args;
    k.status = L.status;
    return k;
}

// Launch with programmatic stream serialization (see pdl_enter).
template <class... KParams, class... Args>
cudaError_t launch_pdl(void (*kernel)(KParams...), int64_t grid, int block, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kUnrollFlat = 2;
constexpr int64_t kMaxGrid = 0x7FFFFFFF;

template <class Op>
cudaError_t run_contiguous(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    const int64_t ng = L.numel / G;
    int64_t grid = ceil_div(ng > 0 ? ng : 1, (int64_t)kThreads * kUnrollFlat);
    grid = std::min<int64_t>(grid, kMaxGrid);
    return launch_pdl(k_contiguous<Op, kUnrollFlat>, grid, kThreads, L.stream, kargs<Op>(L));
}

template <class Op, bool ROW_A> cudaError_t run_rowconst(const Launch &L);

template <class Op, bool SCALAR_A>
cudaError_t run_scalar(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    if constexpr (HasPrep<Op>::value && !SCALAR_A) {
        // a prepared right scalar over a whole number of packs is one row of
        // the per-row flat kernel, the divisor prepared once per thread (fp32
        // Mod fmod0 vs a scalar, A[4096,4096]: 21.98 -> 21.42 us on GB300)
        if (L.numel % G == 0) return run_rowconst<Op, false>(L);
    }
    // an operator that prepares the scalar (Mod's divisor) spreads the
    // preparation over four packs per thread (fp32 Mod fmod0 vs a scalar:
    // 23.7 -> 22.2 us on GB300; one pack 30.7 us, eight 21.8 but int32 worse)
    constexpr int U = HasPrep<Op>::value ? 4 : kUnrollFlat;
    const int64_t ng = L.numel / G;
    int64_t grid = ceil_div(ng > 0 ? ng : 1, (int64_t)kThreads * U);
    grid = std::min<int64_t>(grid, kMaxGrid);
    return launch_pdl(k_scalar<Op, SCALAR_A, U>, grid, kThreads, L.stream, kargs<Op>(L));
}

// Tile shape for a row traversal with rows of `cols` groups and V groups per
// thread per row: threads per row, rows in parallel and rows per thread,
// aiming at enough CTAs for several waves.
// min_kr: the fewest rows a thread walks (operators that prepare a divisor
// per row amortise the thread's setup over at least two).
inline RowArgs row_args(const Geom &g, int G, int V, int num_sms, int64_t min_kr = 1) {
    RowArgs r{};
    const int rank = g.rank;
    r.L = g.n[rank - 1];
    r.cols = r.L / G;
    r.ia = g.sa[rank - 1];
    r.ib = g.sb[rank - 1];
    r.ic = g.sc[rank - 1];
    if (rank >= 2) {
        r.M = g.n[rank - 2];
        r.smA = g.sa[rank - 2];
        r.smB = g.sb[rank - 2];
        r.smC = g.sc[rank - 2];
    } else {
        r.M = 1;
        r.smA = 0;
        r.smB = 0;
        r.smC = 0;
    }
    r.nprefix = rank >= 2 ? rank - 2 : 0;
    int64_t P = 1;
    for (int i = 0; i < r.nprefix; ++i) {
        r.pn[i] = g.n[i];
        r.psa[i] = g.sa[i];
        r.psb[i] = g.sb[i];
        r.psc[i] = g.sc[i];
        r.f_pn[i] = make_fastdiv((uint64_t)g.n[i]);
        P *= g.n[i];
    }
    const int64_t per_thread_cols = ceil_div(r.cols, V);
    if (per_thread_cols >= kThreads) {
        r.tpr = kThreads;
        r.rs = 1;
    } else {
        r.tpr = (int32_t)per_thread_cols;
        r.rs = (int32_t)(kThreads / per_thread_cols);
        if (r.rs > r.M) r.rs = (int32_t)r.M;
    }
    r.cc = ceil_div(r.cols, (int64_t)r.tpr * V);
    r.pack_ok = (r.L % ((int64_t)V * G) == 0) ? 1 : 0;
    // rows per thread: keep >= ~16 CTAs per SM in flight, at most 16 rows each
    const int64_t groups = P * r.M * r.cols;
    const int64_t per_cta = (int64_t)r.tpr * r.rs * V;
    int64_t kr = groups / (per_cta * (int64_t)num_sms * 16);
    kr = std::max<int64_t>(min_kr, std::min<int64_t>(16, kr));
    kr = std::min<int64_t>(kr, ceil_div(r.M, r.rs));
    r.kr = (int32_t)kr;
    r.runs = ceil_div(r.M, (int64_t)r.rs * r.kr);
    r.f_cc = make_fastdiv((uint64_t)r.cc);
    r.f_runs = make_fastdiv((uint64_t)r.runs);
    r.f_tpr = make_fastdiv((uint64_t)r.tpr);
    r.f_rs = make_fastdiv((uint64_t)r.rs);
    const int64_t tiles = P * r.runs * r.cc;
    r.wide = tiles >= (1ll << 31) ? 1 : 0;
    for (int i = 0; i < r.nprefix; ++i)
        if (r.pn[i] >= (1ll << 32)) r.wide = 1;
    if (r.cc >= (1ll << 32) || r.runs >= (1ll << 32) || r.M + r.rs >= (1ll << 32)) r.wide = 1;
    return r;
}

inline int64_t row_tiles(const RowArgs &r) {
    int64_t P = 1;
    for (int i = 0; i < r.nprefix; ++i) P *= r.pn[i];
    return P * r.runs * r.cc;
}

template <class Op, int G, int IA, int IB, bool NOPREFIX, int V, bool PACKED>
cudaError_t run_rows_kernel(const Launch &L) {
    const RowArgs r = row_args(L.g, G, V, L.num_sms, MinRowsOf<Op>::value);
    const int64_t tiles = row_tiles(r);
    if (tiles > kMaxGrid) return cudaErrorInvalidConfiguration;
    return launch_pdl(k_rows<Op, G, IA, IB, NOPREFIX, V, PACKED>, tiles, r.tpr * r.rs, L.stream,
                      kargs<Op>(L), r);
}

// Column groups per thread per row (V), measured on GB300.  Outputs narrower
// than the inputs (comparisons to BOOL) take adjacent groups whose results make
// one 16-byte store (Greater fp16 -> BOOL [64,32,512,1024]: 7.6 TB/s, against
// 5.1 with groups a row-width apart).  Otherwise two groups a row-width apart
// for a dense A (per-channel bf16: 5.0 TB/s, against 4.4 with one group and
// four rows per iteration) and four when A is one value per row.
template <class Op, int IA, int IB>
struct RowShape {
    using In = typename Op::In;
    using Out = typename Op::Out;
    static constexpr int G = 16 / (int)sizeof(In);
    static constexpr bool kElemB = IB == 1 && !Op::kPlainB;
    static constexpr int kPackV = 16 / (G * (int)sizeof(Out));
    static constexpr bool PACKED = !kElemB && sizeof(Out) < sizeof(In) && kPackV >= 2;
    // a floating divisor prepared per row is spread over 4 groups (Mod fp32
    // against [4096,1]: 25.5 -> 24.5 us; int32 Mod is faster with 2)
    static constexpr bool kFloatPrepRow = HasPrep<Op>::value && IB == 0 && is_float_v<In>;
    static constexpr int V = PACKED ? (kPackV > 4 ? 4 : kPackV)
                             : kElemB ? 1
                             : (IA == 0 || kFloatPrepRow) ? 4 : 2;
};

// Resident CTAs of KERNEL per SM at kThreads threads, looked up once per
// kernel (the kernel is the template argument: kernels of one signature share
// a pointer type, so a cache keyed on the type would hand every one of them
// the first kernel's count).
template <auto KERNEL> int resident_ctas() {
    static const int n = [] {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, KERNEL, kThreads, 0) != cudaSuccess ||
            b < 1) {
            cudaGetLastError();
            b = 1;
        }
        return b;
    }();
    return n;
}

// The dense input covers the whole output in order (its coalesced strides
// are the dense ones) and the other input is one value per row: the flat
// k_rowconst streams it.  Rows must be a whole number of packs.
inline bool rowconst_fits(const Geom &g, int G, bool row_a) {
    const int r = g.rank;
    if (r < 2) return false;
    const int64_t *sd = row_a ? g.sb : g.sa;      // the dense input
    const int64_t *sr = row_a ? g.sa : g.sb;      // the per-row input
    if (g.n[r - 1] % G != 0 || sd[r - 1] != 1 || sr[r - 1] != 0) return false;
    int64_t acc = g.n[r - 1];
    for (int i = r - 2; i >= 0; --i) {
        if (sd[i] != acc) return false;
        acc *= g.n[i];
    }
    return true;
}

// One CTA per chunk of kThreads x U x iters consecutive packs; `iters` sized
// for about kRowConstWaves waves of resident CTAs (measured on GB300, bf16
// x[8,64,256,256]: per-channel Add 24.6 us at two waves, 21.7 at four, 21.2
// at eight).  A shared-memory staging of the dense input (cp.async, up to
// three runs ahead) and two packs per thread for the costlier operators were
// tried and gave nothing once BatchNormalization's divide was prepared.
constexpr int kRowConstU = 4;
template <class Op> constexpr int kRowConstWaves = HasGroup<Op>::value ? 4 : 8;

// The per-row launch description: rows of g.n[rank - 1] elements (packs of
// G), the outer dims, and the per-row input's strides `sr` along them.
inline RowConstArgs rowconst_args(const Geom &g, int G, const int64_t *sr) {
    RowConstArgs r{};
    const int rank = g.rank;
    r.lp = g.n[rank - 1] / G;
    r.f_lp = make_fastdiv((uint64_t)r.lp);
    r.nd = rank - 1;
    for (int i = 0; i < r.nd; ++i) {
        r.on[i] = g.n[i];
        r.os[i] = sr[i];
        r.f_on[i] = make_fastdiv((uint64_t)g.n[i]);
    }
    return r;
}

// Launch a per-row flat kernel: runs of kThreads x U packs, `iters` of them
// per CTA, for about `waves` waves of resident CTAs.  K32 indexes packs in 32
// bits, K64 in 64: K32 runs when every run start a thread forms, and every
// row bound, stays below 2^31 packs (grid x iters runs of kThreads x U packs
// cover them all), whatever the occupancy behind `iters`.
template <class Op, auto K32, auto K64>
cudaError_t launch_rowconst(const Launch &L, RowConstArgs r, int G, int U, int waves) {
    const int64_t np = L.numel / G;
    const int64_t per_run = (int64_t)kThreads * U;
    const int64_t runs = ceil_div(np, per_run);
    auto shape = [&](int resident, int64_t &iters, int64_t &grid) {
        const int64_t slots = (int64_t)L.num_sms * resident * waves;
        iters = std::max<int64_t>(1, ceil_div(runs, slots));
        grid = ceil_div(runs, iters);
    };
    int64_t iters = 0, grid = 0;
    shape(resident_ctas<K32>(), iters, grid);
    const bool narrow = grid * iters * per_run < (1ll << 31);
    if (!narrow) shape(resident_ctas<K64>(), iters, grid);
    if (iters > 0x7FFFFFFF || grid > kMaxGrid) return cudaErrorInvalidConfiguration;
    r.iters = (int32_t)iters;
    if (narrow) return launch_pdl(K32, grid, kThreads, L.stream, kargs<Op>(L), r);
    return launch_pdl(K64, grid, kThreads, L.stream, kargs<Op>(L), r);
}

template <class Op, bool ROW_A>
cudaError_t run_rowconst(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    constexpr int U = kRowConstU;
    constexpr int kMin = RowConstMinCtas<Op>::value;
    const RowConstArgs r = rowconst_args(L.g, G, ROW_A ? L.g.sa : L.g.sb);
    if constexpr (kMin > 0)
        return launch_rowconst<Op, k_rowconst_bounded<Op, ROW_A, U, false, kMin>,
                               k_rowconst_bounded<Op, ROW_A, U, true, kMin>>(
            L, r, G, U, kRowConstWaves<Op>);
    else
        return launch_rowconst<Op, k_rowconst<Op, ROW_A, U, false>, k_rowconst<Op, ROW_A, U, true>>(
            L, r, G, U, kRowConstWaves<Op>);
}

// Three inputs: operand rp one value per row, the other two dense over the
// output in order (their coalesced strides the dense ones), rows a whole
// number of packs.
inline bool rowconst3_fits(const Geom &g, int G, int rp) {
    const int r = g.rank;
    if (r < 2 || g.n[r - 1] % G != 0) return false;
    const int64_t *st[3] = {g.sa, g.sb, g.sc};
    for (int k = 0; k < 3; ++k)
        if (st[k][r - 1] != (k == rp ? 0 : 1)) return false;
    int64_t acc = g.n[r - 1];
    for (int i = r - 2; i >= 0; --i) {
        for (int k = 0; k < 3; ++k)
            if (k != rp && st[k][i] != acc) return false;
        acc *= g.n[i];
    }
    return true;
}

// two packs of each dense input per thread and run (MulAdd bf16
// x[8,64,256,256] * s[1,64,1,1] + y on GB300: 30.25 us, against 32.08 with
// four packs at 111 registers and 32.27 on the row traversal k_rows3)
constexpr int kRowConst3U = 2;

template <class Op, int RP>
cudaError_t run_rowconst3(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    constexpr int U = kRowConst3U;
    const int64_t *sr = RP == 0 ? L.g.sa : RP == 1 ? L.g.sb : L.g.sc;
    const RowConstArgs r = rowconst_args(L.g, G, sr);
    return launch_rowconst<Op, k_rowconst3<Op, RP, U, false>, k_rowconst3<Op, RP, U, true>>(
        L, r, G, U, 8);
}

template <class Op, bool NOPREFIX>
cudaError_t run_rows_vector(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    const int64_t ia = L.g.sa[L.g.rank - 1], ib = L.g.sb[L.g.rank - 1];
    if (ia == 1 && ib == 0 && rowconst_fits(L.g, G, false)) return run_rowconst<Op, false>(L);
    if constexpr (Op::kPlainB) {
        if (ia == 0 && ib == 1 && rowconst_fits(L.g, G, true)) return run_rowconst<Op, true>(L);
    }
    if (ia == 1 && ib == 1) {
        using S = RowShape<Op, 1, 1>;
        return run_rows_kernel<Op, G, 1, 1, NOPREFIX, S::V, S::PACKED>(L);
    }
    if (ia == 1 && ib == 0) {
        using S = RowShape<Op, 1, 0>;
        return run_rows_kernel<Op, G, 1, 0, NOPREFIX, S::V, S::PACKED>(L);
    }
    if (ia == 0 && ib == 1) {
        using S = RowShape<Op, 0, 1>;
        return run_rows_kernel<Op, G, 0, 1, NOPREFIX, S::V, S::PACKED>(L);
    }
    return cudaErrorInvalidValue;
}

template <class Op>
cudaError_t run_general(const Launch &L) {
    return run_rows_kernel<Op, 1, 2, 2, false, 2, false>(L);
}

// The pattern of one input over the last two coalesced dims (n1, n2), for
// k_periodic: dense (n2, 1), one value per row (1, 0), a reused row (0, 1).
inline int pmode_of(int64_t s1, int64_t s2, int64_t n2) {
    if (s1 == n2 && s2 == 1) return PM_DENSE;
    if (s1 == 1 && s2 == 0) return PM_ROWVAL;
    if (s1 == 0 && s2 == 1) return PM_ROWBLOCK;
    return -1;
}

// Whether k_periodic can stream a plan (rank 2, or rank 3 with an outer
// index), and its arguments: 32-bit indices, one input at least repeating,
// packs that stay inside a block and dense inputs whose packs stay aligned.
// A dense B only for operators whose B is a plain tensor of A's type.
template <class Op>
bool periodic_fits(const Launch &L, int *ma, int *mb, PeriodicArgs *pa) {
    constexpr int64_t G = 16 / sizeof(typename Op::In);
    const Geom &g = L.g;
    if (L.numel >= (1ll << 31) || (g.rank != 2 && g.rank != 3)) return false;
    const int o = g.rank - 2;          // first of the two inner dims
    const int64_t n1 = g.n[o], n2 = g.n[o + 1];
    *ma = pmode_of(g.sa[o], g.sa[o + 1], n2);
    *mb = pmode_of(g.sb[o], g.sb[o + 1], n2);
    if (*ma < 0 || *mb < 0 || (*ma == PM_DENSE && *mb == PM_DENSE)) return false;
    if (*mb == PM_DENSE && !Op::kPlainB) return false;
    const int64_t sa0 = o ? g.sa[0] : 0, sb0 = o ? g.sb[0] : 0;
    if (o && (n1 * n2) % G != 0) return false;
    if ((*ma == PM_DENSE && sa0 % G != 0) || (*mb == PM_DENSE && sb0 % G != 0)) return false;
    pa->P = (int32_t)n2;
    pa->Lb = (int32_t)(o ? n1 * n2 : L.numel);
    pa->sa0 = (int32_t)sa0;
    pa->sb0 = (int32_t)sb0;
    pa->fP = make_fastdiv((uint64_t)pa->P);
    pa->fLb = make_fastdiv((uint64_t)pa->Lb);
    return true;
}

// A reused short row against data dense in the block, in blocks of at least
// one k_blockrow tile: the shared-memory rotations instead of per-element reads.
constexpr int kBlockRowU = 4;

template <class Op, bool X_IS_A>
cudaError_t launch_blockrow(const Launch &L, const PeriodicArgs &pa) {
    constexpr int G = 16 / sizeof(typename Op::In);
    BlockRowArgs b{};
    b.P = pa.P;
    b.Lb = pa.Lb;
    b.n0 = (int32_t)(L.numel / pa.Lb);
    b.sx0 = X_IS_A ? pa.sa0 : pa.sb0;
    b.sd0 = X_IS_A ? pa.sb0 : pa.sa0;
    b.fP = pa.fP;
    b.fLb = pa.fLb;
    b.dr = (int32_t)(((int64_t)kThreads * G) % pa.P);
    const int64_t ng = L.numel / G;
    const int64_t grid = ceil_div(ng > 0 ? ng : 1, (int64_t)kThreads * kBlockRowU);
    if (grid > kMaxGrid) return cudaErrorInvalidConfiguration;
    return launch_pdl(k_blockrow<Op, X_IS_A, kBlockRowU>, grid, kThreads, L.stream, kargs<Op>(L),
                      b);
}

template <class Op, int MA, int MB>
cudaError_t launch_periodic(const Launch &L, const PeriodicArgs &pa) {
    constexpr int G = 16 / sizeof(typename Op::In);
    const int64_t ng = L.numel / G;
    int64_t grid = ceil_div(ng > 0 ? ng : 1, (int64_t)kThreads * kUnrollFlat);
    grid = std::min<int64_t>(grid, kMaxGrid);
    return launch_pdl(k_periodic<Op, MA, MB, kUnrollFlat>, grid, kThreads, L.stream, kargs<Op>(L),
                      pa);
}

// Short rows and general shapes that k_periodic streams, else the row kernel
// (the general traversal).  Pointers off 16-byte alignment never reach here
// (the host sends them to the general family first).
template <class Op>
cudaError_t run_periodic(const Launch &L) {
    int ma, mb;
    PeriodicArgs pa{};
    if (!periodic_fits<Op>(L, &ma, &mb, &pa)) return run_general<Op>(L);
    if constexpr (Op::kPlainB) {
        constexpr int64_t G = 16 / sizeof(typename Op::In);
        const bool blockrow = pa.P <= kBlockRowMaxP && pa.Lb >= (int64_t)kThreads * kBlockRowU * G &&
                              L.numel % pa.Lb == 0;
        if (blockrow && ma == PM_ROWBLOCK && mb == PM_DENSE) return launch_blockrow<Op, true>(L, pa);
        if (blockrow && ma == PM_DENSE && mb == PM_ROWBLOCK) return launch_blockrow<Op, false>(L, pa);
    }
    switch (ma * 3 + mb) {
    case PM_DENSE * 3 + PM_ROWVAL: return launch_periodic<Op, PM_DENSE, PM_ROWVAL>(L, pa);
    case PM_DENSE * 3 + PM_ROWBLOCK: return launch_periodic<Op, PM_DENSE, PM_ROWBLOCK>(L, pa);
    default: break;
    }
    if constexpr (Op::kPlainB) {
        switch (ma * 3 + mb) {
        case PM_ROWVAL * 3 + PM_DENSE: return launch_periodic<Op, PM_ROWVAL, PM_DENSE>(L, pa);
        case PM_ROWBLOCK * 3 + PM_DENSE: return launch_periodic<Op, PM_ROWBLOCK, PM_DENSE>(L, pa);
        case PM_ROWVAL * 3 + PM_ROWBLOCK: return launch_periodic<Op, PM_ROWVAL, PM_ROWBLOCK>(L, pa);
        case PM_ROWBLOCK * 3 + PM_ROWVAL: return launch_periodic<Op, PM_ROWBLOCK, PM_ROWVAL>(L, pa);
        default: break;
        }
    }
    return run_general<Op>(L);
}

// Operators that accept a scalar B given as an attribute (Op::kScalarAttr).
template <class Op, class = void> struct HasScalarAttr : std::false_type {};
template <class Op>
struct HasScalarAttr<Op, std::void_t<decltype(Op::kScalarAttr)>>
    : std::bool_constant<Op::kScalarAttr> {};

// A plan whose B is the attribute value: A is dense, so the right-scalar kernel
// runs it (a single element plans as contiguous), or the general kernel when
// pointers are off the 16-byte alignment.
template <class Op>
cudaError_t launch_with_scalar(const Launch &L) {
    using W = WithScalar<Op>;
    switch (L.family) {
    case FAM_CONTIGUOUS:
    case FAM_RIGHT_SCALAR: return run_scalar<W, false>(L);
    case FAM_GENERAL_STRIDED: return run_general<W>(L);
    default: return cudaErrorInvalidValue;
    }
}

// The buffers allow 16-byte input packs and packs of G outputs (the host
// sends unaligned buffers to the general family, whose row traversal reads
// element by element).
// A rank-2 plan with one input dense (strides (N, 1)) and the other a
// transposed view (strides (1, ld), ld not 0 or 1): 1 when B is the
// transposed one, 0 when A is, -1 otherwise.
inline int transposed_input(const Geom &g) {
    if (g.rank != 2) return -1;
    const int64_t N = g.n[1];
    const bool a_dense = g.sa[0] == N && g.sa[1] == 1, b_dense = g.sb[0] == N && g.sb[1] == 1;
    const bool a_t = g.sa[1] == 1 ? false : g.sa[0] == 1 && g.sa[1] != 0;
    const bool b_t = g.sb[1] == 1 ? false : g.sb[0] == 1 && g.sb[1] != 0;
    if (a_dense && b_t) return 1;
    if (b_dense && a_t) return 0;
    return -1;
}

template <class Op, bool T_IS_B>
cudaError_t run_transposed(const Launch &L) {
    constexpr int64_t TW = kTransTile;
    TransArgs a{};
    a.M = L.g.n[0];
    a.N = L.g.n[1];
    a.ld = T_IS_B ? L.g.sb[1] : L.g.sa[1];
    const int64_t tm = ceil_div(a.M, TW), tn = ceil_div(a.N, TW);
    if (tm * tn > kMaxGrid) return run_general<Op>(L);
    a.tiles_n = (uint32_t)tn;
    return launch_pdl(k_transposed<Op, T_IS_B>, tm * tn, kThreads, L.stream, kargs<Op>(L), a);
}

template <class Op> bool packs_aligned(const Launch &L) {
    constexpr uintptr_t G = 16 / sizeof(typename Op::In);
    return (uintptr_t)L.A % 16 == 0 && (!L.B || (uintptr_t)L.B % 16 == 0) &&
           (uintptr_t)L.out % (G * sizeof(typename Op::Out)) == 0;
}

// Launch the kernel of L.family for operator functor Op.
template <class Op>
cudaError_t launch_op(const Launch &L) {
    if constexpr (!Op::kLegal) {
        return cudaErrorInvalidValue;
    } else {
        if (L.args.with_scalar) {
            if constexpr (HasScalarAttr<Op>::value) return launch_with_scalar<Op>(L);
            else return cudaErrorInvalidValue;
        }
        switch (L.family) {
        case FAM_CONTIGUOUS: return run_contiguous<Op>(L);
        case FAM_RIGHT_SCALAR: return run_scalar<Op, false>(L);
        case FAM_LEFT_SCALAR:
            if constexpr (Op::kPlainB) return run_scalar<Op, true>(L);
            else return cudaErrorInvalidValue;
        case FAM_REPEATED_BLOCK:
            if (L.g.rank == 2 && L.g.n[1] % (16 / (int64_t)sizeof(typename Op::In)) != 0)
                return run_periodic<Op>(L);
            if (L.g.rank == 2) return run_rows_vector<Op, true>(L);
            return run_rows_vector<Op, false>(L);
        case FAM_INNER_VECTOR_OUTER: return run_rows_vector<Op, false>(L);
        case FAM_GENERAL_STRIDED:
            // a transposed input takes the tiled kernel; short rows and outer
            // products stream flat when the buffers allow 16-byte packs;
            // anything else takes the general row traversal
            if constexpr (Op::kPlainB &&
                          std::is_same_v<typename BInOf<Op>::type, typename Op::In>) {
                const int t = transposed_input(L.g);
                if (t == 1) return run_transposed<Op, true>(L);
                if (t == 0) return run_transposed<Op, false>(L);
            }
            if (packs_aligned<Op>(L)) return run_periodic<Op>(L);
            return run_general<Op>(L);
        default: return cudaErrorInvalidValue;
        }
    }
}

// Three-input operators: the row kernel for inner strides in {0, 1}, else the
// element-by-element form.
template <class Op, int G, int IA, int IB, int IC, int V>
cudaError_t run_rows3_kernel(const Launch &L) {
    const RowArgs r = row_args(L.g, G, V, L.num_sms);
    const int64_t tiles = row_tiles(r);
    if (tiles > kMaxGrid) return cudaErrorInvalidConfiguration;
    return launch_pdl(k_rows3<Op, G, IA, IB, IC, V>, tiles, r.tpr * r.rs, L.stream,
                      kargs<Op>(L), r);
}

template <class Op, int IA, int IB, int IC>
cudaError_t run_flat3(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    const int64_t ng = L.numel / G;
    int64_t grid = ceil_div(ng > 0 ? ng : 1, (int64_t)kThreads * kUnrollFlat);
    grid = std::min<int64_t>(grid, kMaxGrid);
    return launch_pdl(k_flat3<Op, IA, IB, IC, kUnrollFlat>, grid, kThreads, L.stream,
                      kargs<Op>(L));
}

template <class Op>
cudaError_t launch_op3(const Launch &L) {
    if constexpr (!Op::kLegal) {
        return cudaErrorInvalidValue;
    } else {
        constexpr int G = 16 / sizeof(typename Op::In);
        // one column group per thread and row: two or three dense inputs hold
        // enough bytes in flight (MulAdd bf16 x[8,64,256,256] * [1,64,1,1] + y:
        // 32.9 us, against 37.7 with two groups)
        constexpr int V = 1;
        if (L.family == FAM_GENERAL_STRIDED) return run_rows3_kernel<Op, 1, 2, 2, 2, 2>(L);
        if (L.family == FAM_EMPTY) return cudaSuccess;
        const int r = L.g.rank;
        const int code = (int)(L.g.sa[r - 1] * 4 + L.g.sb[r - 1] * 2 + L.g.sc[r - 1]);
        if (r == 1) {   // streaming: one tile per CTA
            switch (code) {
            case 7: return run_flat3<Op, 1, 1, 1>(L);
            case 6: return run_flat3<Op, 1, 1, 0>(L);
            case 5: return run_flat3<Op, 1, 0, 1>(L);
            case 4: return run_flat3<Op, 1, 0, 0>(L);
            case 3: return run_flat3<Op, 0, 1, 1>(L);
            case 2: return run_flat3<Op, 0, 1, 0>(L);
            case 1: return run_flat3<Op, 0, 0, 1>(L);
            default: return cudaErrorInvalidValue;
            }
        }
        // one input one value per row, the other two dense: the per-row flat
        // kernel
        if (code == 5 && rowconst3_fits(L.g, G, 1)) return run_rowconst3<Op, 1>(L);
        if (code == 3 && rowconst3_fits(L.g, G, 0)) return run_rowconst3<Op, 0>(L);
        if (code == 6 && rowconst3_fits(L.g, G, 2)) return run_rowconst3<Op, 2>(L);
        switch (code) {
        case 7: return run_rows3_kernel<Op, G, 1, 1, 1, V>(L);
        case 6: return run_rows3_kernel<Op, G, 1, 1, 0, V>(L);
        case 5: return run_rows3_kernel<Op, G, 1, 0, 1, V>(L);
        case 4: return run_rows3_kernel<Op, G, 1, 0, 0, V>(L);
        case 3: return run_rows3_kernel<Op, G, 0, 1, 1, V>(L);
        case 2: return run_rows3_kernel<Op, G, 0, 1, 0, V>(L);
        case 1: return run_rows3_kernel<Op, G, 0, 0, 1, V>(L);
        default: return cudaErrorInvalidValue;
        }
    }
}

// Element type of each class.
template <int DT> struct DtType;
template <> struct DtType<DT_F32> { using type = float; };
template <> struct DtType<DT_F16> { using type = __half; };
template <> struct DtType<DT_BF16> { using type = __nv_bfloat16; };
template <> struct DtType<DT_I32> { using type = int32_t; };
template <> struct DtType<DT_I64> { using type = int64_t; };
template <> struct DtType<DT_U8> { using type = uint8_t; };
template <> struct DtType<DT_U32> { using type = uint32_t; };
template <> struct DtType<DT_BOOL> { using type = Bool8; };
template <> struct DtType<DT_I8> { using type = int8_t; };
template <> struct DtType<DT_I16> { using type = int16_t; };
template <> struct DtType<DT_U16> { using type = uint16_t; };
template <> struct DtType<DT_U64> { using type = uint64_t; };
template <> struct DtType<DT_F64> { using type = double; };

}  // namespace ebin

// Name of this translation unit's entry for group g: launch_<g>_<EBIN_DT>.
#define EBIN_CAT2(a, b) a##b
#define EBIN_CAT(a, b) EBIN_CAT2(a, b)
#define EBIN_GROUP_FN(g) EBIN_CAT(launch_##g##_, EBIN_DT)
