// Add, Sub, Mul, Div for one element class (EBIN_DT).
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(arith)(const Launch &L) {
    using T = DtType<EBIN_DT>::type;
    switch (L.op) {
    case 0: return launch_op<OpArith<T, K_ADD>>(L);
    case 1: return launch_op<OpArith<T, K_SUB>>(L);
    case 2: return launch_op<OpArith<T, K_MUL>>(L);
    case 3: return launch_op<OpArith<T, K_DIV>>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
