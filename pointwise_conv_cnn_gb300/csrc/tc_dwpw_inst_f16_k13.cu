// tc_dwpw_inst_f16_k13.cu -- instantiations of the DW->PW kernels for half storage and filter sizes
// 1 and 3 (one of several translation units, compiled in parallel).
#include "tc_dwpw_kernel.cuh"

namespace fcm {
namespace tc {

#define FCM_INST(T, KS, S, MODE, DWB) \
    template cudaError_t launch_k<T, KS, S, MODE, DWB>(const Args &, int, int, uint32_t, cudaStream_t);

FCM_INST(__half, 1, 1, FUSED, 0)
FCM_INST(__half, 1, 1, FUSED, 1)
FCM_INST(__half, 1, 1, DWONLY, 0)
FCM_INST(__half, 1, 1, DWONLY, 1)
FCM_INST(__half, 1, 2, FUSED, 0)
FCM_INST(__half, 1, 2, FUSED, 1)
FCM_INST(__half, 1, 2, DWONLY, 0)
FCM_INST(__half, 1, 2, DWONLY, 1)
FCM_INST(__half, 3, 1, FUSED, 0)
FCM_INST(__half, 3, 1, FUSED, 1)
FCM_INST(__half, 3, 1, DWONLY, 0)
FCM_INST(__half, 3, 1, DWONLY, 1)
FCM_INST(__half, 3, 2, FUSED, 0)
FCM_INST(__half, 3, 2, FUSED, 1)
FCM_INST(__half, 3, 2, DWONLY, 0)
FCM_INST(__half, 3, 2, DWONLY, 1)
FCM_INST(__half, 1, 1, PWONLY, 0)

FCM_INST(__half, 3, 1, FUSED, 2)
FCM_INST(__half, 3, 1, DWONLY, 2)
FCM_INST(__half, 3, 2, FUSED, 2)
FCM_INST(__half, 3, 2, DWONLY, 2)

#undef FCM_INST

}  // namespace tc
}  // namespace fcm
