// Pow for one element class (EBIN_DT): the floating types and signed integers.
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(pow)(const Launch &L) {
    return launch_op<OpPow<DtType<EBIN_DT>::type>>(L);
}

}  // namespace ebin
