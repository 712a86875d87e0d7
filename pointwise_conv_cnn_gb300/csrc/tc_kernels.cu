// tc_kernels.cu -- dense conv1 on tensor cores: placeholder until the back-to-back kernel lands.
#include "fcm_internal.h"

cudaError_t launch_tc_b2b(const fcm_handle *, int, const void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
