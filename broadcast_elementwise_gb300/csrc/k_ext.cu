// ncnn binaryop extras for one element class (EBIN_DT): Max, Min, RSub, RDiv
// (ncnn operators.md, binaryop, operation types 4, 5, 7, 8).
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(ext)(const Launch &L) {
    using T = DtType<EBIN_DT>::type;
    switch (L.op) {
    case 21: return launch_op<OpMinMax<T, true>>(L);
    case 22: return launch_op<OpMinMax<T, false>>(L);
    case 23: return launch_op<OpArith<T, K_RSUB>>(L);
    case 24: return launch_op<OpArith<T, K_RDIV>>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
