// selftest.cu -- exercises the kernels' failure path on the GPU without a
// fault: one thread waits, through the same bounded mbarrier wait every
// kernel of the library uses, on a barrier that nothing ever completes.  The
// wait gives up at its time limit, ORs the timeout bit into the device status
// word and returns; the kernel then exits normally, so the CUDA context stays
// usable and diffattn_get_device_error reports DIFFATTN_ERR_TIMEOUT.
#include "kernels.h"
#include "ptx.cuh"

namespace diffattn {
namespace {

__global__ void selftest_wait_timeout_kernel(uint32_t* status) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);        // expects one arrival; none is ever made
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const AbortState ab{&abort_flag, status};
        (void)mbar_wait(&bar, 0, ab);   // runs out after the library's wait limit
    }
}

}  // namespace

int launch_selftest_timeout(uint32_t* status, cudaStream_t stream) {
    selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace diffattn
