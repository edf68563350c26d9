// Pow with an exponent of another type, for one base element class (EBIN_DT):
// the typed scalar adapters of "Binary Kernel Design" (Compute, scheduling,
// and safety), run by the general kernel only.
#include "ebin_kernels.cuh"

namespace ebin {

template <class Op>
cudaError_t launch_mixed(const Launch &L) {
    if constexpr (!Op::kLegal) {
        return cudaErrorInvalidValue;
    } else {
        if (L.family == FAM_EMPTY) return cudaSuccess;
        if (L.family != FAM_GENERAL_STRIDED) return cudaErrorInvalidValue;
        return run_general<Op>(L);
    }
}

cudaError_t EBIN_GROUP_FN(powmix)(const Launch &L) {
    using TA = DtType<EBIN_DT>::type;
    switch (L.dt_b) {
    case DT_F32: return launch_mixed<OpPowMixed<TA, float>>(L);
    case DT_F16: return launch_mixed<OpPowMixed<TA, __half>>(L);
    case DT_BF16: return launch_mixed<OpPowMixed<TA, __nv_bfloat16>>(L);
    case DT_I32: return launch_mixed<OpPowMixed<TA, int32_t>>(L);
    case DT_I64: return launch_mixed<OpPowMixed<TA, int64_t>>(L);
    case DT_U8: return launch_mixed<OpPowMixed<TA, uint8_t>>(L);
    case DT_U32: return launch_mixed<OpPowMixed<TA, uint32_t>>(L);
    case DT_I8: return launch_mixed<OpPowMixed<TA, int8_t>>(L);
    case DT_I16: return launch_mixed<OpPowMixed<TA, int16_t>>(L);
    case DT_U16: return launch_mixed<OpPowMixed<TA, uint16_t>>(L);
    case DT_U64: return launch_mixed<OpPowMixed<TA, uint64_t>>(L);
    case DT_F64: return launch_mixed<OpPowMixed<TA, double>>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
