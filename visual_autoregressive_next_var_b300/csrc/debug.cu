// Input checks of the debug build (compiled with -DVAR_DEBUG): before a call
// that reads an index list, a small kernel checks every entry on the device
// -- inside [0, N), and strictly ascending where the call requires it -- and
// records VAR_ERR_INVALID_ARG in the call's status word for a bad list.  The
// release build compiles this file to nothing; its kernels clamp bad indices
// (pruned attention) or skip them (restore) without reporting.
#include "internal.h"

namespace varattn {

#ifdef VAR_DEBUG
namespace {

__global__ void __launch_bounds__(256)
    check_indices_kernel(const int32_t* __restrict__ idx, int B, int K, int N, int ascending, int32_t* status)
{
    const long long t = blockIdx.x * 256ll + threadIdx.x;
    if (t >= static_cast<long long>(B) * K) return;
    const int b = static_cast<int>(t / K), j = static_cast<int>(t - static_cast<long long>(b) * K);
    const int v = idx[t];
    bool ok = v >= 0 && v < N;
    if (ascending && j > 0) ok = ok && idx[t - 1] < v;
    (void)b;
    if (!ok) atomicCAS(status, 0, VAR_ERR_INVALID_ARG);
}

}  // namespace

int debug_check_indices(const int32_t* idx, int B, int K, int N, bool ascending, int32_t* status, cudaStream_t st)
{
    if (K <= 0 || !idx) return VAR_OK;
    const long long n = static_cast<long long>(B) * K;
    return cuda_status(launch_kernel(check_indices_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                                     st, false, idx, B, K, N, ascending ? 1 : 0, status));
}
#endif

}  // namespace varattn
