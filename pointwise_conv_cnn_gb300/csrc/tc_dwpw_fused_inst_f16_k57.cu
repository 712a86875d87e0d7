// tc_dwpw_fused_inst_f16_k57.cu -- instantiations of the worker-warp DW->PW kernel for half
// storage and filter sizes 5 and 7 (one of several translation units, compiled in parallel).
#define FCM_FUSED_KERNEL_BODY
#include "tc_dwpw_fused.cuh"

namespace fcm {
namespace tc {

template cudaError_t launch_fused<__half, 5, 1>(const FArgs &, int, int, uint32_t, cudaStream_t);
template cudaError_t launch_fused<__half, 5, 2>(const FArgs &, int, int, uint32_t, cudaStream_t);
template cudaError_t launch_fused<__half, 7, 1>(const FArgs &, int, int, uint32_t, cudaStream_t);
template cudaError_t launch_fused<__half, 7, 2>(const FArgs &, int, int, uint32_t, cudaStream_t);

}  // namespace tc
}  // namespace fcm
