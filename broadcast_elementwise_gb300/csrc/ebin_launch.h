// Internal interface between the host planner (ebin_host.cpp) and the kernel
// translation units (k_*.cu).  Not part of the public C ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace ebin {

constexpr int kMaxRank = 8;

// Internal element-type classes, one kernel set each.
enum Dt : int {
    DT_F32 = 0, DT_F16, DT_BF16, DT_I32, DT_I64, DT_U8, DT_U32, DT_BOOL,
    DT_I8, DT_I16, DT_U16, DT_U64, DT_F64, DT_COUNT
};

// Loop families (same numbering as the public ebin_family).
enum Fam : int {
    FAM_EMPTY = 0,
    FAM_CONTIGUOUS = 1,
    FAM_LEFT_SCALAR = 2,
    FAM_RIGHT_SCALAR = 3,
    FAM_REPEATED_BLOCK = 4,
    FAM_INNER_VECTOR_OUTER = 5,
    FAM_GENERAL_STRIDED = 6
};

// Operator parameters read by the device functors.
struct OpArgs {
    int32_t fmod;        // Mod: 0 floor, 1 truncated
    int32_t direction;   // BitShift: 0 left, 1 right
    float eps;           // BatchNormalization
    int32_t has_min;     // Clip
    int32_t has_max;     // Clip
    int64_t plane;       // BatchNormalization, BiasPRelu(BN): elements between parameter rows
    int32_t with_scalar; // B is scalar_b, not a tensor (ncnn binaryop with_scalar)
    float scalar_b;
    float one;           // exactly 1.0f: a multiplier the device code cannot fold away
};

// Coalesced traversal: rank dims, extents n, element strides of A and B.
// The output is dense row-major over n.
struct Geom {
    int32_t rank;
    int64_t n[kMaxRank];
    int64_t sa[kMaxRank];
    int64_t sb[kMaxRank];
    int64_t sc[kMaxRank];   // third input (three-input operators), else 0
};

struct Launch {
    int op;              // public ebin_op code
    int dt;              // input element class (Dt)
    int dt_b;            // B's element class (differs from dt for mixed-type Pow)
    int family;          // Fam (after the alignment fallback)
    Geom g;
    int64_t numel;
    const void *A;
    const void *B;
    const void *C;       // third input (three-input operators), else nullptr
    void *out;
    OpArgs args;
    uint32_t *status;    // device status word, or nullptr for operators that never flag
    cudaStream_t stream;
    int num_sms;
};

// Enqueue the kernel for L; returns cudaSuccess or the launch error.
cudaError_t launch(const Launch &L);

// One function per operator group and element class; each k_<group>.cu is
// compiled once per class (-DEBIN_DT=<Dt>) so the translation units build in
// parallel.  A class outside a group's manifest returns cudaErrorInvalidValue.
#define EBIN_DECLARE_GROUP(g)                                                          \
    cudaError_t launch_##g##_0(const Launch &);                                       \
    cudaError_t launch_##g##_1(const Launch &);                                       \
    cudaError_t launch_##g##_2(const Launch &);                                       \
    cudaError_t launch_##g##_3(const Launch &);                                       \
    cudaError_t launch_##g##_4(const Launch &);                                       \
    cudaError_t launch_##g##_5(const Launch &);                                       \
    cudaError_t launch_##g##_6(const Launch &);                                       \
    cudaError_t launch_##g##_7(const Launch &);                                       \
    cudaError_t launch_##g##_8(const Launch &);                                       \
    cudaError_t launch_##g##_9(const Launch &);                                       \
    cudaError_t launch_##g##_10(const Launch &);                                      \
    cudaError_t launch_##g##_11(const Launch &);                                      \
    cudaError_t launch_##g##_12(const Launch &);
EBIN_DECLARE_GROUP(arith)   // Add Sub Mul Div
EBIN_DECLARE_GROUP(mod)     // Mod
EBIN_DECLARE_GROUP(pow)     // Pow
EBIN_DECLARE_GROUP(cmp)     // Equal Less Greater LessOrEqual GreaterOrEqual
EBIN_DECLARE_GROUP(logic)   // And Or Xor BitwiseAnd/Or/Xor BitShift
EBIN_DECLARE_GROUP(chan)    // PRelu BatchNormalization Clip BiasPRelu BiasPReluBN
EBIN_DECLARE_GROUP(ext)     // Max Min RSub RDiv
EBIN_DECLARE_GROUP(tern)    // MulAdd (three inputs)
EBIN_DECLARE_GROUP(powmix)  // Pow with an exponent of another type
#undef EBIN_DECLARE_GROUP

}  // namespace ebin
