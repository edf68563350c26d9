// Three-input operators for one element class (EBIN_DT): MulAdd
// (0verkilll/onnx ops, MulAddOp).
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(tern)(const Launch &L) {
    using T = DtType<EBIN_DT>::type;
    switch (L.op) {
    case 26: return launch_op3<OpMulAdd<T>>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
