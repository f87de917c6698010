// The library's only door to the CUDA runtime and driver.
//
// Every CUDA call the host code makes goes through the function table below,
// and every kernel is launched by launch_kernel() (cudaLaunchKernelExC), so a
// test can swap the table for a mock that fakes a device and makes a chosen
// call fail (var_test_mock_cuda in include/varattn_test.h).  That reaches each
// VAR_ERR_CUDA branch of the C ABI on a machine without a GPU.  The mock runs
// no kernel; it is for the host logic only.
#pragma once
#include <cstddef>
#include <cstdint>
#include <tuple>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace varattn {

struct CudaOps {
    cudaError_t (*get_device)(int*);
    cudaError_t (*device_attribute)(int*, cudaDeviceAttr, int);
    cudaError_t (*get_symbol_address)(void**, const void*);
    cudaError_t (*func_set_attribute)(const void*, cudaFuncAttribute, int);
    cudaError_t (*launch)(const cudaLaunchConfig_t*, const void*, void**);
    cudaError_t (*memcpy_async)(void*, const void*, size_t, cudaMemcpyKind, cudaStream_t);
    cudaError_t (*memset_async)(void*, int, size_t, cudaStream_t);
    cudaError_t (*stream_sync)(cudaStream_t);
    cudaError_t (*device_sync)();
    // cuTensorMapEncodeTiled, resolved through the runtime's driver entry point
    CUresult (*encode_tiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
};

// The table in use: the real runtime, or the mock while a test has it enabled.
const CudaOps& rt();
// True while the mock is enabled.  Per-device caches are neither read nor
// filled then, so nothing a mock call returned outlives the mock.
bool rt_mocked();

// The current device (VAR_ERR_CUDA-style failure as a non-zero return).
cudaError_t current_device(int* dev);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per device and
// function; max_carveout also asks for the largest shared-memory carveout (for
// a kernel whose resident CTAs per SM fill it).
cudaError_t ensure_smem_attr_raw(const void* func, int bytes, bool max_carveout = false);

// Launch `kern` on `st` with `args` converted to the kernel's parameter types.
// pdl: allow the launch to start as a programmatic dependent of the preceding
// work on the stream (the kernel waits for it with griddepcontrol.wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          Args&&... args)
{
    static_assert(sizeof...(KArgs) == sizeof...(Args), "argument count differs from the kernel's");
    std::tuple<std::remove_cv_t<std::remove_reference_t<KArgs>>...> vals(std::forward<Args>(args)...);
    void* ptrs[sizeof...(KArgs) > 0 ? sizeof...(KArgs) : 1];
    std::apply([&](auto&... v) {
        int i = 0;
        ((ptrs[i++] = static_cast<void*>(&v)), ...);
    }, vals);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = pdl ? at : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return rt().launch(&cfg, reinterpret_cast<const void*>(kern), ptrs);
}

// Set the dynamic shared memory limit of `kern` once per device.
template <typename... KArgs>
cudaError_t ensure_smem_attr(void (*kern)(KArgs...), int bytes, bool max_carveout = false)
{
    return ensure_smem_attr_raw(reinterpret_cast<const void*>(kern), bytes, max_carveout);
}

}  // namespace varattn
