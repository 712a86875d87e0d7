// tc_dwpw_fused_inst_i8_k13.cu -- instantiations of the worker-warp DW->PW kernel for int8
// storage and filter sizes 1 and 3 (one of several translation units, compiled in parallel).
#define FCM_FUSED_KERNEL_BODY
#include "tc_dwpw_fused.cuh"

namespace fcm {
namespace tc {

template cudaError_t launch_fused<int8_t, 1, 1>(const FArgs &, int, int, uint32_t, cudaStream_t);
template cudaError_t launch_fused<int8_t, 1, 2>(const FArgs &, int, int, uint32_t, cudaStream_t);
template cudaError_t launch_fused<int8_t, 3, 1>(const FArgs &, int, int, uint32_t, cudaStream_t);
template cudaError_t launch_fused<int8_t, 3, 2>(const FArgs &, int, int, uint32_t, cudaStream_t);

}  // namespace tc
}  // namespace fcm
