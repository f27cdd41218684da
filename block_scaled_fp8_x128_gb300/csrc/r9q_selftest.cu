// Failure-detection self-test: a kernel whose bounded waits run out.
//
// Every wait in the GEMM kernels gives up after a bound, records a timeout in
// the device error word and lets the kernel return (no trap, no endless
// loop).  This kernel exercises exactly those wait helpers on an mbarrier or
// a counter that nothing ever completes, so a test can check that the bound
// holds, that the host reads R9Q_ERR_TIMEOUT and that the context stays
// usable afterwards.
#include <cuda_runtime.h>

#include "r9q.h"
#include "r9q_device.cuh"
#include "r9q_stream.cuh"

namespace r9q {
namespace {

__device__ int g_never;   // stays 0: nothing ever increments it

__global__ void wait_timeout_kernel(int* err, int which) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // one arrival expected; none ever comes
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    bool gave_up = false;
    if (which & 1) gave_up |= !mbar_wait(&bar, 0);                 // GEMM pipelines' spinning wait
    if (which & 2) gave_up |= !mbar_wait_sleep(&bar, 0, 1000, 1u << 12);   // sleeping wait (short bound)
    if (which & 4) gave_up |= !mbar_wait_cluster(&bar, 0);         // split-K reduction's cluster wait
    if (which & 8) gave_up |= !wait_count(&g_never, 1);             // quantised-row counter wait
    if (gave_up) record_error(err, kErrTimeout);
}

}  // namespace
}  // namespace r9q

extern "C" int r9q_selftest_wait_timeout(int which, void* stream) {
    if (which < 0 || which > 15) return R9Q_ERR_ARG;
    int* err = nullptr;
    const int rc = r9q::device_error_word(&err);
    if (rc) return rc;
    r9q::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, which);
    return cudaGetLastError() == cudaSuccess ? R9Q_OK : R9Q_ERR_LAUNCH;
}
