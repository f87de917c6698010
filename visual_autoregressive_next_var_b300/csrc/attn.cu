// Dense and pruned (gathered-query) cross-scale attention: host launchers of
// the shared kernel in attn_kernel.cuh.
#include "attn_kernel.cuh"

namespace varattn {

// ---------------------------------------------------------------------------- host

template <int D, int MODE>
static int launch_attn(const StepGeom& g, const void* q, const void* k, const void* v,
                       const int32_t* idx, int n_rows, void* o, cudaStream_t st)
{
    using Lay = AttnLayout<D>;
    static bool attr_done = false;   // per process; the attribute is per function
    auto kern = attn_kernel<D, MODE, DenseMaps>;
    if (!attr_done) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM_BYTES) !=
            cudaSuccess)
            return VAR_ERR_CUDA;
        attr_done = true;
    }
    int32_t* status = device_status_ptr();
    if (!status) return VAR_ERR_CUDA;
    if (n_rows == 0) return VAR_OK;

    DenseMaps maps;
    CUtensorMap& tq = maps.q;
    CUtensorMap& tk = maps.k;
    CUtensorMap& tv = maps.v;
    const uint32_t box[3] = {64, 128, 1};
    const uint64_t BH = static_cast<uint64_t>(g.B) * g.H;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(g.N), BH};
        const uint64_t strides[2] = {D * 2ull, static_cast<uint64_t>(g.N) * D * 2ull};
        if (int rc = encode_tmap_bf16(&tq, q, 3, dims, strides, box)) return rc;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(g.L), BH};
        const uint64_t strides[2] = {D * 2ull, static_cast<uint64_t>(g.cap) * D * 2ull};
        if (int rc = encode_tmap_bf16(&tk, k, 3, dims, strides, box)) return rc;
        if (int rc = encode_tmap_bf16(&tv, v, 3, dims, strides, box)) return rc;
    }
    AttnArgs a = {};
    a.n_rows = n_rows;
    a.n_q = g.N;
    a.L = g.L;
    a.heads = g.H;
    a.pairs_per_bh = (n_rows + 255) / 256;
    a.n_kv = (g.L + 127) / 128;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.idx = idx;
    a.o = static_cast<__nv_bfloat16*>(o);
    a.status = status;
    const dim3 grid(static_cast<unsigned>(BH * a.pairs_per_bh));
    kern<<<grid, 384, Lay::SMEM_BYTES, st>>>(maps, a);
    return cuda_status(cudaGetLastError());
}

int launch_attn_dense(const StepGeom& g, const void* q, const void* k, const void* v, void* o,
                      cudaStream_t st)
{
    if (g.D == 128) return launch_attn<128, MODE_DENSE>(g, q, k, v, nullptr, g.N, o, st);
    if (g.D == 64) return launch_attn<64, MODE_DENSE>(g, q, k, v, nullptr, g.N, o, st);
    return VAR_ERR_UNSUPPORTED;
}

int launch_attn_pruned(const StepGeom& g, const void* q, const void* k, const void* v,
                       const int32_t* idx, int keep_k, void* o, cudaStream_t st)
{
    if (g.D == 128) return launch_attn<128, MODE_GATHER>(g, q, k, v, idx, keep_k, o, st);
    if (g.D == 64) return launch_attn<64, MODE_GATHER>(g, q, k, v, idx, keep_k, o, st);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
