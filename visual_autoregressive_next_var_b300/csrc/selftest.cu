// Diagnostics: a bounded wait that is made to give up.  One thread waits on
// an mbarrier that nothing arrives on; the wait returns after its time limit
// and the kernel records VAR_ERR_TIMEOUT in the call's status word, as a
// pipeline wait of the attention kernels would, then exits.  No fault, no
// hang: the device stays usable.
#include "internal.h"
#include "ptx.cuh"

namespace varattn {

namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int32_t* status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait(b, 0, nullptr, limit_ns)) atomicCAS(status, 0, VAR_ERR_TIMEOUT);
}

}  // namespace

int launch_wait_timeout(int limit_us, cudaStream_t st, int32_t* status)
{
    return cuda_status(launch_kernel(wait_timeout_kernel, dim3(1), dim3(32), 0, st, false,
                                     static_cast<uint64_t>(limit_us) * 1000ull, status));
}

}  // namespace varattn
