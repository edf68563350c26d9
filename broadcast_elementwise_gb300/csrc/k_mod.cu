// Mod (fmod 0 / 1, opset-28 sign rules) for one element class (EBIN_DT).
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(mod)(const Launch &L) {
    return launch_op<OpMod<DtType<EBIN_DT>::type>>(L);
}

}  // namespace ebin
