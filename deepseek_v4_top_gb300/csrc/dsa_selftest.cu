// Self-test of the bounded waits every kernel of this library uses: one
// warp waits on an mbarrier that nothing arrives on.  The wait gives up
// after its limit (kWaitLimitNs), raises DSA_DEVERR_TIMEOUT and returns, so
// the context stays usable; a test reads the bit and then runs real work.
#include <stdint.h>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace {

__global__ void dsa_wait_selftest_kernel(uint32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);      // one arrival expected, none made
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0, &abort_flag, err);
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t s) {
    dsa_wait_selftest_kernel<<<1, 32, 0, s>>>(err);
    return cudaGetLastError();
}

}  // namespace dsa
