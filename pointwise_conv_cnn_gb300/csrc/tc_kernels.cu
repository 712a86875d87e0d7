// tc_kernels.cu -- tensor-core (tcgen05) kernels: placeholder until they land.
#include "fcm_internal.h"

int fcm_tc_supported(const fcm_desc *, int, int, int, const char **why) {
    if (why) *why = "tensor-core kernels not built";
    return 0;
}
fcm_status fcm_tc_plan(const fcm_desc *, int, int, int, int, int, TcPlan *) {
    return FCM_ERR_UNSUPPORTED;
}
fcm_status fcm_tc_prepare(fcm_handle *, const void *, const void *) { return FCM_ERR_UNSUPPORTED; }
cudaError_t launch_tc_dwpw(const fcm_handle *, int, const void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_tc_b2b(const fcm_handle *, int, const void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_tc_pw(const fcm_handle *, const void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
