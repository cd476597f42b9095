// selftest.cu - a bounded wait that is never satisfied.
//
// One thread waits, with the same bounded mbarrier wait every kernel of the
// library uses, on a barrier that nothing arrives on.  The wait gives up
// after the given limit, the kernel records ATTN_DEV_WAIT_TIMEOUT in the
// caller's status word and returns: the path a pipeline takes when a stage
// never fills, exercised without any fault, trap or hang.
#include "common.cuh"
#include "ptx.cuh"

namespace gb300 {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0, nullptr, limit_ns)) flag_status(status, ATTN_DEV_WAIT_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace gb300
