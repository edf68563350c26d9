// Loop-family kernels of the broadcast binary engine for sm_103a, and the
// per-operator launcher that picks one from the plan's family.
//
// Families ("Binary Kernel Design", section "Operators and traversal",
// loop-family table), each a kernel template instantiated per operator and
// element type:
//   k_contiguous   A, B and out advance together             (Contiguous)
//   k_scalar       one operand is a single value             (Left / right scalar)
//   k_rows<2-D>    rank 2: one value per row, or one row block reused for every
//                  row                                        (Repeated contiguous block)
//   k_rows<N-D>    vectorised inner rows, incremental outer offsets
//                                                             (Inner-vector / outer broadcast)
//   k_rows<G=1>    any coalesced strides, element at a time  (General strided)
//
// Memory access: the dense streams move in 16-byte vectors (ld.global.nc with
// L1::no_allocate for inputs that are read once); a warp's 32 lanes touch 512
// consecutive bytes per access.  Offsets advance incrementally ("division and
// modulo are not performed for every output element"): each lane decomposes
// its first index once and afterwards only adds and carries.
//
// Validation ("Compute, scheduling, and safety"): operators that can meet an
// invalid element (integer division by zero, shift counts) write 0 for it and
// OR a bit into the stream's status word once per thread.  There is no trap,
// no assert and no waiting in any kernel.
#pragma once

#include <cstring>

#include "ebin_ops.cuh"

namespace ebin {

constexpr int kThreads = 256;

template <class T, int G> struct alignas(sizeof(T) * G) Pack {
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

template <class T, int G>
__device__ __forceinline__ void st_pack(T *p, const Pack<T, G> &v) {
    *reinterpret_cast<Pack<T, G> *>(p) = v;
}

template <class Op>
__device__ __forceinline__ void flush_err(uint32_t *status, uint32_t err) {
    if constexpr (Op::kValidates) {
        if (err) atomicOr(status, err);
    }
}

// Everything a kernel needs, passed by value.
struct KArgs {
    const void *A;
    const void *B;
    void *out;
    int64_t numel;
    OpArgs args;
    uint32_t *status;
};

// Row traversal (k_rows): the coalesced dims split into an inner row of
// `inner` elements (= cols groups of G) and up to kMaxRank-1 outer digits,
// stored right-aligned in on/osa/osb (digit kMaxRank-2 is next to the row).
// Unused digits have a huge extent so that no carry ever reaches them.
struct RowArgs {
    int64_t cols;          // groups per row
    int64_t ngroups;       // rows * cols
    int64_t per_warp;      // groups handled by each warp (multiple of 32)
    int64_t ia, ib;        // inner element strides of A and B (general kernel)
    int32_t outer;         // number of live outer digits
    int64_t on[kMaxRank - 1];
    int64_t osa[kMaxRank - 1];
    int64_t osb[kMaxRank - 1];
};

// ---------------------------------------------------------------- Contiguous
template <class Op, int U>
__global__ void __launch_bounds__(kThreads) k_contiguous(KArgs p) {
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BV = typename Op::BV;
    constexpr int G = 16 / sizeof(In);
    const In *A = static_cast<const In *>(p.A);
    const In *B = static_cast<const In *>(p.B);
    Out *O = static_cast<Out *>(p.out);
    const int64_t ng = p.numel / G;
    uint32_t err = 0;
    const int64_t step = (int64_t)gridDim.x * (kThreads * U);
    for (int64_t base = (int64_t)blockIdx.x * (kThreads * U) + threadIdx.x; base < ng;
         base += step) {
        Pack<In, G> a[U];
        BV b[U][G];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) {
                a[u] = ld_stream<In, G>(A + g * G);
                if constexpr (Op::kPlainB) {
                    const Pack<In, G> t = ld_stream<In, G>(B + g * G);
#pragma unroll
                    for (int k = 0; k < G; ++k) b[u][k] = t.v[k];
                } else {
#pragma unroll
                    for (int k = 0; k < G; ++k) b[u][k] = Op::loadB(B, g * G + k, p.args);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t g = base + (int64_t)u * kThreads;
            if (g < ng) {
                Pack<Out, G> o;
#pragma unroll
                for (int k = 0; k < G; ++k) o.v[k] = Op::apply(a[u].v[k], b[u][k], p.args, err);
                st_pack<Out, G>(O + g * G, o);
            }
        }
    }
    // ragged tail (numel % G elements)
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
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BV = typename Op::BV;
    constexpr int G = 16 / sizeof(In);
    const In *A = static_cast<const In *>(p.A);
    const In *B = static_cast<const In *>(p.B);
    Out *O = static_cast<Out *>(p.out);
    const In *D = SCALAR_A ? B : A;
    In sa{};
    BV sb{};
    if constexpr (SCALAR_A) sa = A[0];
    else sb = Op::loadB(B, 0, p.args);
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
#pragma unroll
                for (int k = 0; k < G; ++k) {
                    if constexpr (SCALAR_A) o.v[k] = Op::apply(sa, d[u].v[k], p.args, err);
                    else o.v[k] = Op::apply(d[u].v[k], sb, p.args, err);
                }
                st_pack<Out, G>(O + g * G, o);
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
// Repeated block, inner-vector/outer-broadcast and general strided.  The
// output is split into rows of `cols` groups of G elements; every warp owns a
// contiguous range of `per_warp` groups.  Lane l handles groups
// begin + l, begin + l + 32, ...: each access of the warp covers 32
// consecutive groups.  A lane decomposes its first group once; every further
// step adds 32 to its column and carries whole rows into the outer digits,
// updating the A and B row offsets by the digits' strides.
//
// IA / IB: 1 = the operand advances along the row (vector loads), 0 = it is
// constant along the row (one value per row, read once per step), 2 = any
// inner stride (G must be 1).  TWO_D: exactly one outer digit (rank-2 plans),
// so the carry is a single add.
template <class Op, int G, int IA, int IB, bool TWO_D, int U>
__global__ void __launch_bounds__(kThreads) k_rows(KArgs p, RowArgs r) {
    using In = typename Op::In;
    using Out = typename Op::Out;
    using BV = typename Op::BV;
    constexpr int D = kMaxRank - 1;
    static_assert(G == 1 || (IA != 2 && IB != 2), "runtime inner strides need G == 1");
    const In *A = static_cast<const In *>(p.A);
    const In *B = static_cast<const In *>(p.B);
    Out *O = static_cast<Out *>(p.out);

    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t begin = warp * r.per_warp;
    const int64_t end = min(begin + r.per_warp, r.ngroups);
    if (begin >= end) return;

    // first group of this lane -> (row digits, column)
    int64_t g = begin + lane;
    int64_t row = g / r.cols;
    int64_t col = g - row * r.cols;
    int64_t idx[D];
    int64_t rowA = 0, rowB = 0;
    if constexpr (TWO_D) {
        idx[D - 1] = row;
        rowA = row * r.osa[D - 1];
        rowB = row * r.osb[D - 1];
    } else {
#pragma unroll
        for (int d = D - 1; d >= 0; --d) {
            if (d >= D - r.outer) {
                const int64_t q = row / r.on[d];
                idx[d] = row - q * r.on[d];
                row = q;
                rowA += idx[d] * r.osa[d];
                rowB += idx[d] * r.osb[d];
            } else {
                idx[d] = 0;
            }
        }
    }

    uint32_t err = 0;
    while (g < end) {
        int64_t offA[U], offB[U], gs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            gs[u] = g;
            offA[u] = rowA + (IA == 1 ? col * G : IA == 0 ? 0 : col * r.ia);
            offB[u] = rowB + (IB == 1 ? col * G : IB == 0 ? 0 : col * r.ib);
            // advance this lane by 32 groups
            g += 32;
            col += 32;
            while (col >= r.cols) {
                col -= r.cols;
                if constexpr (TWO_D) {
                    rowA += r.osa[D - 1];
                    rowB += r.osb[D - 1];
                } else {
#pragma unroll
                    for (int d = D - 1; d >= 0; --d) {
                        idx[d] += 1;
                        rowA += r.osa[d];
                        rowB += r.osb[d];
                        if (idx[d] < r.on[d]) break;
                        idx[d] = 0;
                        rowA -= r.on[d] * r.osa[d];
                        rowB -= r.on[d] * r.osb[d];
                    }
                }
            }
        }
        // A: a vector per group, or one value per row (IA == 0)
        // B: a vector per group (IB == 1), or one value per row (IB == 0)
        Pack<In, G> a[U];
        In as[U];
        BV b[U][G];
        BV bs[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (gs[u] < end) {
                if constexpr (IA == 1 && G > 1) a[u] = ld_stream<In, G>(A + offA[u]);
                else as[u] = A[offA[u]];
                if constexpr (IB == 1 && G > 1 && Op::kPlainB) {
                    const Pack<In, G> t = ld_stream<In, G>(B + offB[u]);
#pragma unroll
                    for (int k = 0; k < G; ++k) b[u][k] = t.v[k];
                } else if constexpr (IB == 1 && G > 1) {
#pragma unroll
                    for (int k = 0; k < G; ++k) b[u][k] = Op::loadB(B, offB[u] + k, p.args);
                } else {
                    bs[u] = Op::loadB(B, offB[u], p.args);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (gs[u] < end) {
                Pack<Out, G> o;
#pragma unroll
                for (int k = 0; k < G; ++k) {
                    const In x = (IA == 1 && G > 1) ? a[u].v[k] : as[u];
                    if constexpr (IB == 1 && G > 1) o.v[k] = Op::apply(x, b[u][k], p.args, err);
                    else o.v[k] = Op::apply(x, bs[u], p.args, err);
                }
                if constexpr (G > 1) st_pack<Out, G>(O + gs[u] * G, o);
                else O[gs[u]] = o.v[0];
            }
        }
    }
    flush_err<Op>(p.status, err);
}

// ---------------------------------------------------------------- launch helpers
template <class K>
int blocks_per_sm(K kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess ||
        n < 1)
        n = 1;
    return n;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <class Op>
KArgs kargs(const Launch &L) {
    KArgs k;
    k.A = L.A;
    k.B = L.B;
    k.out = L.out;
    k.numel = L.numel;
    k.args = L.args;
    k.status = L.status;
    return k;
}

constexpr int kUnrollFlat = 4;
constexpr int kUnrollRows = 2;

template <class Op>
cudaError_t run_contiguous(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    auto kernel = k_contiguous<Op, kUnrollFlat>;
    static const int bps = blocks_per_sm(kernel);
    const int64_t ng = L.numel / G;
    int64_t grid = ceil_div(ng > 0 ? ng : 1, (int64_t)kThreads * kUnrollFlat);
    grid = std::min<int64_t>(grid, (int64_t)L.num_sms * bps);
    kernel<<<(unsigned)std::max<int64_t>(grid, 1), kThreads, 0, L.stream>>>(kargs<Op>(L));
    return cudaGetLastError();
}

template <class Op, bool SCALAR_A>
cudaError_t run_scalar(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    auto kernel = k_scalar<Op, SCALAR_A, kUnrollFlat>;
    static const int bps = blocks_per_sm(kernel);
    const int64_t ng = L.numel / G;
    int64_t grid = ceil_div(ng > 0 ? ng : 1, (int64_t)kThreads * kUnrollFlat);
    grid = std::min<int64_t>(grid, (int64_t)L.num_sms * bps);
    kernel<<<(unsigned)std::max<int64_t>(grid, 1), kThreads, 0, L.stream>>>(kargs<Op>(L));
    return cudaGetLastError();
}

// Fill RowArgs from the coalesced geometry with rows of `inner` elements
// split into groups of G.
inline RowArgs row_args(const Geom &g, int G) {
    RowArgs r;
    const int rank = g.rank;
    const int64_t inner = g.n[rank - 1];
    r.cols = inner / G;
    r.ngroups = 0;
    r.per_warp = 0;
    r.ia = g.sa[rank - 1];
    r.ib = g.sb[rank - 1];
    r.outer = rank - 1;
    constexpr int D = kMaxRank - 1;
    int64_t rows = 1;
    for (int d = 0; d < D; ++d) {
        r.on[d] = (int64_t)1 << 62;
        r.osa[d] = 0;
        r.osb[d] = 0;
    }
    for (int i = 0; i < rank - 1; ++i) {
        const int d = D - (rank - 1) + i;
        r.on[d] = g.n[i];
        r.osa[d] = g.sa[i];
        r.osb[d] = g.sb[i];
        rows *= g.n[i];
    }
    r.ngroups = rows * r.cols;
    return r;
}

template <class Op, int G, int IA, int IB, bool TWO_D>
cudaError_t run_rows_kernel(const Launch &L, RowArgs r) {
    auto kernel = k_rows<Op, G, IA, IB, TWO_D, kUnrollRows>;
    static const int bps = blocks_per_sm(kernel);
    const int64_t warps_max = (int64_t)L.num_sms * bps * (kThreads / 32);
    // at least 4 steps of 32 groups per warp before spreading wider
    int64_t warps = std::min<int64_t>(warps_max, std::max<int64_t>(1, ceil_div(r.ngroups, 32 * 4)));
    r.per_warp = ceil_div(ceil_div(r.ngroups, warps), 32) * 32;
    warps = ceil_div(r.ngroups, r.per_warp);
    const int64_t grid = ceil_div(warps, kThreads / 32);
    kernel<<<(unsigned)std::max<int64_t>(grid, 1), kThreads, 0, L.stream>>>(kargs<Op>(L), r);
    return cudaGetLastError();
}

template <class Op, bool TWO_D>
cudaError_t run_rows_vector(const Launch &L) {
    constexpr int G = 16 / sizeof(typename Op::In);
    const RowArgs r = row_args(L.g, G);
    const int64_t ia = r.ia, ib = r.ib;
    if (ia == 1 && ib == 1) return run_rows_kernel<Op, G, 1, 1, TWO_D>(L, r);
    if (ia == 1 && ib == 0) return run_rows_kernel<Op, G, 1, 0, TWO_D>(L, r);
    if (ia == 0 && ib == 1) return run_rows_kernel<Op, G, 0, 1, TWO_D>(L, r);
    return cudaErrorInvalidValue;
}

template <class Op>
cudaError_t run_general(const Launch &L) {
    const RowArgs r = row_args(L.g, 1);
    return run_rows_kernel<Op, 1, 2, 2, false>(L, r);
}

// Launch the kernel of L.family for operator functor Op.
template <class Op>
cudaError_t launch_op(const Launch &L) {
    if constexpr (!Op::kLegal) {
        return cudaErrorInvalidValue;
    } else {
        switch (L.family) {
        case FAM_CONTIGUOUS: return run_contiguous<Op>(L);
        case FAM_RIGHT_SCALAR: return run_scalar<Op, false>(L);
        case FAM_LEFT_SCALAR:
            if constexpr (Op::kPlainB) return run_scalar<Op, true>(L);
            else return cudaErrorInvalidValue;
        case FAM_REPEATED_BLOCK: return run_rows_vector<Op, true>(L);
        case FAM_INNER_VECTOR_OUTER: return run_rows_vector<Op, false>(L);
        case FAM_GENERAL_STRIDED: return run_general<Op>(L);
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

}  // namespace ebin

// Name of this translation unit's entry for group g: launch_<g>_<EBIN_DT>.
#define EBIN_CAT2(a, b) a##b
#define EBIN_CAT(a, b) EBIN_CAT2(a, b)
#define EBIN_GROUP_FN(g) EBIN_CAT(launch_##g##_, EBIN_DT)

namespace ebin {
}  // namespace ebin
