// A test hook for the kernels' bounded waits.  One CTA waits on an mbarrier
// that no thread ever arrives on, with the kernels' own wait (mbar_wait,
// kWaitLimitNs): the wait gives up after its limit, records kStatusTimeout in
// the status word that qmm_kernel_status reads, and the kernel returns.  No
// trap, fault or endless loop is involved, so the context stays usable.
#include <cuda_runtime.h>

#include <cstdint>

#include "qmm_internal.h"
#include "qmm_sm100.cuh"

namespace qmm {

namespace {

__global__ void wait_probe_kernel(int* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status);  // nothing arrives
    __syncthreads();
}

}  // namespace

int launch_wait_probe(void* stream) {
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    return cudaGetLastError();
}

}  // namespace qmm
