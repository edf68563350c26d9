// PRelu, inference BatchNormalization, Clip, BiasPRelu and BiasPReluBN for one element
// class (EBIN_DT): the per-channel and scalar broadcasts of the engine.
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(chan)(const Launch &L) {
    using T = DtType<EBIN_DT>::type;
    switch (L.op) {
    case 18: return launch_op<OpPRelu<T>>(L);
    case 19: return launch_op<OpBN<T>>(L);
    case 20: return launch_op<OpClip<T>>(L);
    case 25: return launch_op<OpBiasPRelu<T>>(L);
    case 27: return launch_op<OpBiasPReluBN<T>>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
