// PRelu, inference BatchNormalization, Clip, BiasPRelu and BiasPReluBN for one element
// class (EBIN_DT): the per-channel and scalar broadcasts of the engine.
#include "ebin_kernels.cuh"

namespace ebin {

// BatchNormalization, BiasPRelu or BiasPReluBN with its parameter block in
// x's own type or, beside a 16-bit or binary64 x, in binary32.
template <template <class, class> class Op, class T>
cudaError_t launch_params(const Launch &L) {
    if constexpr (is_fp_v<T>) {
        if (L.dt_b == DT_F32 && !std::is_same_v<T, float>) return launch_op<Op<T, float>>(L);
    }
    if (L.dt_b != L.dt) return cudaErrorInvalidValue;
    return launch_op<Op<T, T>>(L);
}

cudaError_t EBIN_GROUP_FN(chan)(const Launch &L) {
    using T = DtType<EBIN_DT>::type;
    switch (L.op) {
    case 18: return launch_op<OpPRelu<T>>(L);
    case 19: return launch_params<OpBN, T>(L);
    case 20: return launch_op<OpClip<T>>(L);
    case 25: return launch_params<OpBiasPRelu, T>(L);
    case 27: return launch_params<OpBiasPReluBN, T>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
