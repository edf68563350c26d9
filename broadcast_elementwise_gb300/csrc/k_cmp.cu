// Equal, Less, Greater, LessOrEqual, GreaterOrEqual for one element class
// (EBIN_DT); one byte per BOOL result.
#include "ebin_kernels.cuh"

namespace ebin {

cudaError_t EBIN_GROUP_FN(cmp)(const Launch &L) {
    using T = DtType<EBIN_DT>::type;
    switch (L.op) {
    case 6: return launch_op<OpCmp<T, K_EQ>>(L);
    case 7: return launch_op<OpCmp<T, K_LT>>(L);
    case 8: return launch_op<OpCmp<T, K_GT>>(L);
    case 9: return launch_op<OpCmp<T, K_LE>>(L);
    case 10: return launch_op<OpCmp<T, K_GE>>(L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ebin
