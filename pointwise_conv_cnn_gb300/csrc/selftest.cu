// selftest.cu -- a self-test of the kernels' failure detection: one bounded mbarrier wait that
// cannot complete, through the same wait routine every tensor-core kernel uses.
#include <cuda_runtime.h>

#include "fcm_internal.h"
#include "tc_common.cuh"

namespace {

// One CTA of one warp: initialise an mbarrier expecting one arrival, then wait for its first
// phase, which nothing completes.  mbar_wait gives up after `limit_ns`, sets the error word and
// raises the abort flag; `out` records whether the wait returned success (it must not).
__global__ void wait_timeout_kernel(unsigned *err, unsigned long long limit_ns, int *out) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        fcm::tc::mbar_init(fcm::tc::smem_u32(&bar), 1);
        abort_flag = 0;
        fcm::tc::fence_barrier_init();
    }
    __syncthreads();
    const bool ok = fcm::tc::mbar_wait(fcm::tc::smem_u32(&bar), 0u, &abort_flag, err, limit_ns);
    if (threadIdx.x == 0) *out = ok ? 1 : 0;
}

}  // namespace

extern "C" FCM_API fcm_status fcm_selftest_wait_timeout(unsigned long long limit_ns) {
    if (limit_ns == 0 || limit_ns > 10000000000ull)
        return fcm_fail(FCM_ERR_INVALID_ARG, "limit_ns must be in (0, 10 s]");
    unsigned *err = nullptr;
    int *out = nullptr;
    cudaError_t e = cudaMalloc(&err, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMalloc(&out, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(err, 0, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(out, 0xff, sizeof(int));
    if (e == cudaSuccess) {
        wait_timeout_kernel<<<1, 32>>>(err, limit_ns, out);
        e = cudaGetLastError();
    }
    unsigned word = 0;
    int ok = -1;
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&ok, out, sizeof(ok), cudaMemcpyDeviceToHost);
    if (err) cudaFree(err);
    if (out) cudaFree(out);
    if (e != cudaSuccess)
        return fcm_fail(FCM_ERR_CUDA, "wait self-test: %s", cudaGetErrorString(e));
    if (ok == 0 && (word & FCM_DEVERR_TIMEOUT))
        return fcm_fail(FCM_ERR_TIMEOUT, "the bounded wait ran out and reported it (as designed)");
    return fcm_fail(FCM_ERR_DEVICE_FAULT,
                    "wait self-test: the wait returned %d with error word 0x%x", ok, word);
}
