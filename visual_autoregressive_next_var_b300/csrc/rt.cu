// The CUDA function table of rt.h: the real runtime, and the test-only mock
// behind var_test_mock_cuda (include/varattn_test.h).
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "internal.h"
#include "../../include/varattn_test.h"

namespace varattn {

namespace {

// ---------------------------------------------------------------- real runtime

cudaError_t real_get_symbol_address(void** p, const void* sym) { return cudaGetSymbolAddress(p, sym); }
cudaError_t real_func_set_attribute(const void* f, cudaFuncAttribute a, int v) { return cudaFuncSetAttribute(f, a, v); }
cudaError_t real_launch(const cudaLaunchConfig_t* c, const void* f, void** args) { return cudaLaunchKernelExC(c, f, args); }
cudaError_t real_memcpy_async(void* d, const void* s, size_t n, cudaMemcpyKind k, cudaStream_t st)
{
    return cudaMemcpyAsync(d, s, n, k, st);
}
cudaError_t real_memset_async(void* d, int v, size_t n, cudaStream_t st) { return cudaMemsetAsync(d, v, n, st); }
cudaError_t real_device_sync() { return cudaDeviceSynchronize(); }

CUresult real_encode_tiled(CUtensorMap* m, CUtensorMapDataType t, cuuint32_t rank, void* base, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box, const cuuint32_t* es,
                           CUtensorMapInterleave il, CUtensorMapSwizzle sw, CUtensorMapL2promotion l2,
                           CUtensorMapFloatOOBfill oob)
{
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!fn) {
            void* p = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !p)
                return CUDA_ERROR_NOT_FOUND;
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        }
    }
    return fn(m, t, rank, base, dims, strides, box, es, il, sw, l2, oob);
}

const CudaOps kReal = {cudaGetDevice,          cudaDeviceGetAttribute, real_get_symbol_address,
                       real_func_set_attribute, real_launch,            real_memcpy_async,
                       real_memset_async,       cudaStreamSynchronize,  real_device_sync,
                       real_encode_tiled};

// ---------------------------------------------------------------- mock
// A fake device 0 with 148 SMs and 126 MB of L2.  Each call counts; the call whose count equals
// the requested one fails.  Symbol addresses point at a host buffer that only
// the mock's own memcpy touches; launches run nothing.

std::atomic<bool> g_mock{false};
std::atomic<long long> g_calls{0};
std::atomic<long long> g_fail_at{0};
alignas(256) unsigned char g_fake_symbol[256];

bool mock_fail()
{
    const long long n = ++g_calls;
    return n == g_fail_at.load();
}

cudaError_t mock_get_device(int* d)
{
    if (mock_fail()) return cudaErrorNoDevice;
    *d = 0;
    return cudaSuccess;
}
cudaError_t mock_device_attribute(int* v, cudaDeviceAttr a, int)
{
    if (mock_fail()) return cudaErrorInvalidValue;
    *v = a == cudaDevAttrL2CacheSize ? 126 * 1024 * 1024 : 148;
    return cudaSuccess;
}
cudaError_t mock_get_symbol_address(void** p, const void*)
{
    if (mock_fail()) return cudaErrorInvalidSymbol;
    *p = g_fake_symbol;
    return cudaSuccess;
}
cudaError_t mock_func_set_attribute(const void*, cudaFuncAttribute, int)
{
    return mock_fail() ? cudaErrorInvalidValue : cudaSuccess;
}
cudaError_t mock_launch(const cudaLaunchConfig_t*, const void*, void**)
{
    return mock_fail() ? cudaErrorLaunchFailure : cudaSuccess;
}
cudaError_t mock_memcpy_async(void* d, const void*, size_t n, cudaMemcpyKind k, cudaStream_t)
{
    if (mock_fail()) return cudaErrorInvalidValue;
    if (k == cudaMemcpyDeviceToHost) std::memset(d, 0, n);   // the fake device holds zeros
    return cudaSuccess;
}
cudaError_t mock_memset_async(void*, int, size_t, cudaStream_t)
{
    return mock_fail() ? cudaErrorInvalidValue : cudaSuccess;
}
cudaError_t mock_stream_sync(cudaStream_t) { return mock_fail() ? cudaErrorLaunchFailure : cudaSuccess; }
cudaError_t mock_device_sync() { return mock_fail() ? cudaErrorLaunchFailure : cudaSuccess; }
CUresult mock_encode_tiled(CUtensorMap* m, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                           const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                           CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill)
{
    if (mock_fail()) return CUDA_ERROR_INVALID_VALUE;
    std::memset(m, 0, sizeof *m);
    return CUDA_SUCCESS;
}

const CudaOps kMock = {mock_get_device,         mock_device_attribute, mock_get_symbol_address,
                       mock_func_set_attribute, mock_launch,           mock_memcpy_async,
                       mock_memset_async,       mock_stream_sync,      mock_device_sync,
                       mock_encode_tiled};

}  // namespace

const CudaOps& rt() { return g_mock.load() ? kMock : kReal; }

bool rt_mocked() { return g_mock.load(); }

cudaError_t current_device(int* dev)
{
    const cudaError_t e = rt().get_device(dev);
    if (e != cudaSuccess) return e;
    return (*dev < 0 || *dev >= 64) ? cudaErrorInvalidDevice : cudaSuccess;
}

cudaError_t ensure_smem_attr_raw(const void* func, int bytes, bool max_carveout)
{
    int dev = 0;
    if (cudaError_t e = current_device(&dev)) return e;
    if (rt_mocked()) {
        if (cudaError_t e = rt().func_set_attribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) return e;
        return max_carveout ? rt().func_set_attribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, 100)
                            : cudaSuccess;
    }
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, std::pair<int, bool>> done;   // bytes set, carveout set
    std::lock_guard<std::mutex> lk(mu);
    auto& d = done[{dev, func}];
    if (d.first < bytes) {
        if (cudaError_t e = rt().func_set_attribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) return e;
        d.first = bytes;
    }
    if (max_carveout && !d.second) {
        if (cudaError_t e = rt().func_set_attribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, 100))
            return e;
        d.second = true;
    }
    return cudaSuccess;
}

}  // namespace varattn

extern "C" {

int var_test_mock_cuda(int32_t enable, int64_t fail_at)
{
    varattn::g_calls = 0;
    varattn::g_fail_at = enable ? fail_at : 0;
    varattn::g_mock = enable != 0;
    return VAR_OK;
}

int64_t var_test_mock_calls(void) { return varattn::g_calls.load(); }

}  // extern "C"
