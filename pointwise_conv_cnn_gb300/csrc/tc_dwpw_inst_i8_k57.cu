// tc_dwpw_inst_i8_k57.cu -- instantiations of the DW->PW kernels for int8 storage (the INT8
// module) and filter sizes 5 and 7 (one of several translation units, compiled in parallel).
#include "tc_dwpw_kernel.cuh"

namespace fcm {
namespace tc {

#define FCM_INST(T, KS, S, MODE, DWB) \
    template cudaError_t launch_k<T, KS, S, MODE, DWB>(const Args &, int, int, uint32_t, cudaStream_t);

FCM_INST(int8_t, 5, 1, FUSED, 0)
FCM_INST(int8_t, 5, 1, DWONLY, 0)
FCM_INST(int8_t, 5, 2, FUSED, 0)
FCM_INST(int8_t, 5, 2, DWONLY, 0)
FCM_INST(int8_t, 7, 1, FUSED, 0)
FCM_INST(int8_t, 7, 1, DWONLY, 0)
FCM_INST(int8_t, 7, 2, FUSED, 0)
FCM_INST(int8_t, 7, 2, DWONLY, 0)

#undef FCM_INST

}  // namespace tc
}  // namespace fcm
