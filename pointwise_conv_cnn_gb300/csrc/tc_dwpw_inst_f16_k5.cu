// tc_dwpw_inst_f16_k5.cu -- instantiations of the DW->PW kernels for half storage and filter size
// 5 (one of several translation units, compiled in parallel).
#include "tc_dwpw_kernel.cuh"

namespace fcm {
namespace tc {

#define FCM_INST(T, KS, S, MODE, DWB) \
    template cudaError_t launch_k<T, KS, S, MODE, DWB>(const Args &, int, int, uint32_t, cudaStream_t);

FCM_INST(__half, 5, 1, FUSED, 0)
FCM_INST(__half, 5, 1, DWONLY, 0)
FCM_INST(__half, 5, 2, FUSED, 0)
FCM_INST(__half, 5, 2, DWONLY, 0)

#undef FCM_INST

}  // namespace tc
}  // namespace fcm
