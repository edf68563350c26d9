// And, Or, Xor (BOOL), BitwiseAnd/Or/Xor (integers) and BitShift (uint8,
// uint32) for one element class (EBIN_DT).
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(logic)(const Launch &L) {
    using T = DtType<EBIN_DT>::type;
    switch (L.op) {
    case 11: return launch_op<OpLogic<T, K_AND>>(L);
    case 12: return launch_op<OpLogic<T, K_OR>>(L);
    case 13: return launch_op<OpLogic<T, K_XOR>>(L);
    case 14: return launch_op<OpBitwise<T, K_AND>>(L);
    case 15: return launch_op<OpBitwise<T, K_OR>>(L);
    case 16: return launch_op<OpBitwise<T, K_XOR>>(L);
    case 17: return launch_op<OpShift<T>>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
