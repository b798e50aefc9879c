// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing ever completes, with
// the same bounded wait every pipeline role of the library uses. The wait gives up after its
// cycle limit, records DSA_FAULT_TIMEOUT in the error word and the kernel returns normally, so
// the host reads DSA_ERR_TIMEOUT and the context stays usable. No fault, trap or endless loop.
#include "internal.h"

namespace dsa {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);  // expects one arrival that never comes
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const bool done = mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
        if (done) atomicOr(err, DSA_FAULT_INDEX);  // cannot happen: the phase never completes
    }
}

bool launch_wait_timeout(int* err, cudaStream_t s, int* launches) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(err);
    ++*launches;
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace dsa
