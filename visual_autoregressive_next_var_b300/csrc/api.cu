// The C ABI of include/varattn.h: argument checks, geometry, dispatch.
#include <cmath>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"

namespace varattn {

// One status word per device that loads this library, for calls whose problem
// names no status word of its own.  Kernels record the first fault they detect
// (CAS from 0); var_device_status() reads and clears it.
static __device__ int32_t g_status_word;

static std::mutex g_mu;

int32_t* device_status_ptr()
{
    static int32_t* cache[64] = {};
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return nullptr;
    if (rt_mocked()) {
        void* p = nullptr;
        return rt().get_symbol_address(&p, reinterpret_cast<const void*>(&g_status_word)) == cudaSuccess
                   ? static_cast<int32_t*>(p)
                   : nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (rt().get_symbol_address(&p, reinterpret_cast<const void*>(&g_status_word)) != cudaSuccess || !p)
            return nullptr;
        cache[dev] = static_cast<int32_t*>(p);
    }
    return cache[dev];
}

int32_t* status_word(const var_problem* p)
{
    if (p && p->status) return p->status;
    return device_status_ptr();
}

int sm_count()
{
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return 0;
    int n = 0;
    if (rt_mocked())
        return rt().device_attribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0 ? n : 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        if (rt().device_attribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

long long l2_bytes()
{
    static std::mutex mu;
    static long long cache[64] = {};
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return 0;
    int n = 0;
    if (rt_mocked())
        return rt().device_attribute(&n, cudaDevAttrL2CacheSize, dev) == cudaSuccess && n > 0 ? n : 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        if (rt().device_attribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

int encode_tmap_bf16(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box)
{
    cuuint64_t d[5];
    cuuint64_t s[4];
    cuuint32_t b[5];
    cuuint32_t e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUresult r = rt().encode_tiled(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                                         const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? VAR_OK : VAR_ERR_CUDA;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int resolve(const var_problem* p, int32_t step, StepGeom* g)
{
    if (!p) return VAR_ERR_INVALID_ARG;
    if (p->batch <= 0 || p->heads <= 0 || p->n_scales <= 0 || p->n_scales > VAR_MAX_SCALES)
        return VAR_ERR_INVALID_ARG;
    if (step < 0 || step >= p->n_scales) return VAR_ERR_INVALID_ARG;
    if (p->head_dim != 64 && p->head_dim != 128) return VAR_ERR_UNSUPPORTED;
    long long L = 0;
    for (int i = 0; i <= step; ++i) {
        if (p->side[i] <= 0 || p->side[i] > 4096) return VAR_ERR_INVALID_ARG;
        L += static_cast<long long>(p->side[i]) * p->side[i];
    }
    if (L > (1ll << 30)) return VAR_ERR_UNSUPPORTED;
    const long long cap = p->kv_capacity == 0 ? L : p->kv_capacity;
    if (cap < L) return VAR_ERR_INVALID_ARG;
    if (static_cast<long long>(p->batch) * p->heads > 65535ll * 64) return VAR_ERR_UNSUPPORTED;
    if (!(p->softmax_scale >= 0.f) || !std::isfinite(p->softmax_scale)) return VAR_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p->status) & 3u) return VAR_ERR_INVALID_ARG;
    g->B = p->batch;
    g->H = p->heads;
    g->D = p->head_dim;
    g->side = p->side[step];
    g->N = g->side * g->side;
    g->L = static_cast<int>(L);
    g->cap = static_cast<int>(cap);
    g->scale = p->softmax_scale == 0.f ? 1.0f / std::sqrt(static_cast<float>(p->head_dim))
                                       : p->softmax_scale;
    return VAR_OK;
}

int check_pivot_args(const var_problem* p, int32_t step, const void* x, int32_t channels, int32_t keep_k,
                     const int32_t* idx, StepGeom* g)
{
    if (int rc = resolve(p, step, g)) return rc;
    if (!x || channels <= 0 || channels % 32 != 0 || channels > 16384) return VAR_ERR_INVALID_ARG;
    if (keep_k < 0 || keep_k > g->N) return VAR_ERR_INVALID_ARG;
    if (keep_k > 0 && !idx) return VAR_ERR_INVALID_ARG;
    if (g->N > 16384) return VAR_ERR_UNSUPPORTED;
    if (!aligned16(x)) return VAR_ERR_UNSUPPORTED;
    return VAR_OK;
}

}  // namespace varattn

using namespace varattn;

extern "C" {

int var_attn_dense(const var_problem* p, int32_t step, const void* q, const void* k, const void* v,
                   void* o, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (!q || !k || !v || !o) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return launch_attn_dense(g, q, k, v, o, static_cast<cudaStream_t>(stream), status);
}

size_t var_pivot_workspace_bytes(const var_problem* p, int32_t step, int32_t channels)
{
    StepGeom g;
    if (resolve(p, step, &g) != VAR_OK || channels <= 0 || channels % 32 != 0) return 0;
    return pivot_workspace_bytes(g.B, g.N, channels);
}

int var_pivot_select(const var_problem* p, int32_t step, const void* x, int32_t channels,
                     int32_t keep_k, int32_t* idx, float* scores, void* workspace,
                     size_t workspace_bytes, void* stream)
{
    StepGeom g;
    if (int rc = check_pivot_args(p, step, x, channels, keep_k, idx, &g)) return rc;
    const size_t need = pivot_workspace_bytes(g.B, g.N, channels);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return VAR_ERR_WORKSPACE;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return launch_pivot_select(g.B, g.N, channels, x, keep_k, idx, scores, workspace,
                               workspace_bytes, static_cast<cudaStream_t>(stream), status);
}

int var_attn_pruned(const var_problem* p, int32_t step, const void* q, const void* k, const void* v,
                    const int32_t* idx, int32_t keep_k, void* o_compact, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (keep_k < 0 || keep_k > g.N) return VAR_ERR_INVALID_ARG;
    if (keep_k == 0) return VAR_OK;
    if (!q || !k || !v || !idx || !o_compact) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_compact))
        return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    VAR_DEBUG_CHECK_INDICES(idx, g.B, keep_k, g.N, false, status, static_cast<cudaStream_t>(stream));
    return launch_attn_pruned(g, q, k, v, idx, keep_k, o_compact, static_cast<cudaStream_t>(stream), status,
                              false);
}

int var_attn_pruned_scatter(const var_problem* p, int32_t step, const void* q, const void* k, const void* v,
                            const int32_t* idx, int32_t keep_k, void* out, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (keep_k < 0 || keep_k > g.N) return VAR_ERR_INVALID_ARG;
    if (keep_k == 0) return VAR_OK;
    if (!q || !k || !v || !idx || !out) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    VAR_DEBUG_CHECK_INDICES(idx, g.B, keep_k, g.N, true, status, static_cast<cudaStream_t>(stream));
    return launch_attn_pruned(g, q, k, v, idx, keep_k, out, static_cast<cudaStream_t>(stream), status, true);
}

int var_restore_fill(const var_problem* p, int32_t step, const void* prev, const int32_t* idx, int32_t keep_k,
                     void* out, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (step < 1) return VAR_ERR_INVALID_ARG;
    if (keep_k < 0 || keep_k > g.N) return VAR_ERR_INVALID_ARG;
    if (!prev || !out || (keep_k > 0 && !idx)) return VAR_ERR_INVALID_ARG;
    if (!aligned16(prev) || !aligned16(out)) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    VAR_DEBUG_CHECK_INDICES(idx, g.B, keep_k, g.N, true, status, static_cast<cudaStream_t>(stream));
    return launch_restore_scatter(g.B, g.H, g.D, p->side[step - 1], g.side, prev, nullptr, idx, keep_k, out,
                                  static_cast<cudaStream_t>(stream), status, true);
}

int var_pruned_in_place(const var_problem* p, int32_t step, const void* q, const void* k, const void* v,
                        const void* prev, const int32_t* idx, int32_t keep_k, void* out, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (step < 1) return VAR_ERR_INVALID_ARG;
    if (keep_k < 0 || keep_k > g.N) return VAR_ERR_INVALID_ARG;
    if (!prev || !out || (keep_k > 0 && (!q || !k || !v || !idx))) return VAR_ERR_INVALID_ARG;
    if (!aligned16(prev) || !aligned16(out)) return VAR_ERR_UNSUPPORTED;
    if (keep_k > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v))) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    const auto st = static_cast<cudaStream_t>(stream);
    VAR_DEBUG_CHECK_INDICES(idx, g.B, keep_k, g.N, true, status, st);
    if (keep_k > 0)
        if (int rc = launch_attn_pruned(g, q, k, v, idx, keep_k, out, st, status, true)) return rc;
    // the fill's predecessor on the stream is the attention just launched
    return launch_restore_scatter(g.B, g.H, g.D, p->side[step - 1], g.side, prev, nullptr, idx, keep_k, out, st,
                                  status, true, keep_k > 0);
}

int var_pruned_step(const var_problem* p, int32_t step, const void* x, int32_t channels, int32_t keep_k,
                    const void* q, const void* k, const void* v, const void* prev, int32_t* idx, void* out,
                    void* workspace, size_t workspace_bytes, void* stream)
{
    StepGeom g;
    if (int rc = check_pivot_args(p, step, x, channels, keep_k, idx, &g)) return rc;
    if (step < 1) return VAR_ERR_INVALID_ARG;
    if (!prev || !out || (keep_k > 0 && (!q || !k || !v))) return VAR_ERR_INVALID_ARG;
    if (!aligned16(prev) || !aligned16(out)) return VAR_ERR_UNSUPPORTED;
    if (keep_k > 0 && (!aligned16(q) || !aligned16(k) || !aligned16(v))) return VAR_ERR_UNSUPPORTED;
    const size_t need = pivot_workspace_bytes(g.B, g.N, channels);
    if (keep_k > 0 && (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return VAR_ERR_WORKSPACE;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    const auto st = static_cast<cudaStream_t>(stream);
    const int sp = p->side[step - 1];
    if (keep_k == 0)   // nothing kept: the upsampled grid alone
        return launch_restore_scatter(g.B, g.H, g.D, sp, g.side, prev, nullptr, nullptr, 0, out, st, status, true);
    // pivots, then the pruned attention as a programmatic dependent of the
    // selection (it sets up beside it and reads the indices once they are
    // written), then the fill as a dependent of the attention
    if (int rc = launch_pivot_select(g.B, g.N, channels, x, keep_k, idx, nullptr, workspace, workspace_bytes, st,
                                     status))
        return rc;
    if (int rc = launch_attn_pruned(g, q, k, v, idx, keep_k, out, st, status, true, true)) return rc;
    return launch_restore_scatter(g.B, g.H, g.D, sp, g.side, prev, nullptr, idx, keep_k, out, st, status, true, true);
}

int var_attn_dense_lse(const var_problem* p, int32_t step, const void* q, const void* k, const void* v, void* o,
                       float* lse, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (!q || !k || !v || !o || !lse) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return launch_attn_dense(g, q, k, v, o, static_cast<cudaStream_t>(stream), status, lse);
}

int var_attn_saliency(const var_problem* p, int32_t src_step, const void* q_src, const void* k, const float* lse,
                      float* sal, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, src_step, &g)) return rc;
    if (!q_src || !k || !lse || !sal) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q_src) || !aligned16(k)) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return launch_saliency(g, g.N, g.L, q_src, k, lse, sal, static_cast<cudaStream_t>(stream), status);
}

size_t var_guided_pivot_workspace_bytes(const var_problem* p, int32_t step)
{
    StepGeom g;
    if (resolve(p, step, &g) != VAR_OK) return 0;
    return guided_workspace_bytes(g.B, g.N);
}

int var_guided_pivot_select(const var_problem* p, int32_t step, int32_t src_step, const float* sal,
                            int32_t keep_k, int32_t* idx, float* scores, void* workspace, size_t workspace_bytes,
                            void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (src_step < 0 || src_step >= step) return VAR_ERR_INVALID_ARG;
    if (!sal || keep_k < 0 || keep_k > g.N || (keep_k > 0 && !idx)) return VAR_ERR_INVALID_ARG;
    if (g.N > 16384) return VAR_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < guided_workspace_bytes(g.B, g.N) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return VAR_ERR_WORKSPACE;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return launch_guided_pivot(g.B, g.H, p->side[src_step], g.side, sal, keep_k, idx, scores, workspace,
                               workspace_bytes, static_cast<cudaStream_t>(stream), status);
}

size_t var_guided_pivot_exact_workspace_bytes(const var_problem* p, int32_t step, int32_t src_step)
{
    StepGeom g, gs;
    if (resolve(p, step, &g) != VAR_OK || src_step < 0 || src_step >= step || resolve(p, src_step, &gs) != VAR_OK)
        return 0;
    return guided_exact_workspace_bytes(g.B * g.H, gs.N);
}

int var_guided_pivot_select_exact(const var_problem* p, int32_t step, int32_t src_step, const void* q_src,
                                  const void* k, int32_t keep_k, int32_t* idx, double* values, void* workspace,
                                  size_t workspace_bytes, void* stream)
{
    StepGeom g, gs;
    if (int rc = resolve(p, step, &g)) return rc;
    if (src_step < 0 || src_step >= step) return VAR_ERR_INVALID_ARG;
    if (int rc = resolve(p, src_step, &gs)) return rc;
    if (!q_src || !k || keep_k < 0 || keep_k > g.N || (keep_k > 0 && !idx)) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q_src) || !aligned16(k) || (reinterpret_cast<uintptr_t>(values) & 7)) return VAR_ERR_UNSUPPORTED;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
        workspace_bytes < guided_exact_workspace_bytes(g.B * g.H, gs.N))
        return VAR_ERR_WORKSPACE;
    const double scale64 = p->softmax_scale == 0.f ? 1.0 / std::sqrt(static_cast<double>(p->head_dim))
                                                   : static_cast<double>(p->softmax_scale);
    return launch_guided_exact(gs, g.B, g.H, g.side, q_src, k, scale64, keep_k, idx, values, workspace,
                               workspace_bytes, static_cast<cudaStream_t>(stream));
}

int var_attn_dense_halved(const var_problem* p, int32_t step, const void* q, const void* k, const void* v,
                          void* o, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (g.B % 2 != 0) return VAR_ERR_INVALID_ARG;
    if (!q || !k || !v || !o) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return launch_attn_dense_halved(g, q, k, v, o, static_cast<cudaStream_t>(stream), status);
}

int var_restore_scatter(const var_problem* p, int32_t step, const void* prev, const void* o_compact,
                        const int32_t* idx, int32_t keep_k, void* out, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (step < 1) return VAR_ERR_INVALID_ARG;
    if (keep_k < 0 || keep_k > g.N) return VAR_ERR_INVALID_ARG;
    if (!prev || !out || (keep_k > 0 && (!o_compact || !idx))) return VAR_ERR_INVALID_ARG;
    if (!aligned16(prev) || !aligned16(out) || (keep_k > 0 && !aligned16(o_compact)))
        return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    VAR_DEBUG_CHECK_INDICES(idx, g.B, keep_k, g.N, true, status, static_cast<cudaStream_t>(stream));
    return launch_restore_scatter(g.B, g.H, g.D, p->side[step - 1], g.side, prev, o_compact, idx,
                                  keep_k, out, static_cast<cudaStream_t>(stream), status, false);
}

int var_block_mask_build(const var_problem* p, int32_t step, int32_t qblock_side, int32_t radius,
                         int32_t sink_max_side, int32_t* row_ptr, int32_t* entries,
                         int32_t entries_cap, int32_t* nnz_out, int32_t* n_qblocks_out,
                         int32_t* sink_len_out)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (qblock_side <= 0 || qblock_side > 64 || radius < 0 || sink_max_side < 0)
        return VAR_ERR_INVALID_ARG;
    const int sq = g.side;
    if (sq % qblock_side != 0) return VAR_ERR_UNSUPPORTED;
    // The sink scales must lead the schedule so that they form one flat prefix.
    int sink_len = 0;
    bool in_prefix = true;
    for (int sc = 0; sc <= step; ++sc) {
        const int s = p->side[sc];
        if (s <= sink_max_side) {
            if (!in_prefix) return VAR_ERR_UNSUPPORTED;
            sink_len += s * s;
        } else {
            in_prefix = false;
            if ((s + qblock_side - 1) / qblock_side > 4095) return VAR_ERR_UNSUPPORTED;
        }
    }
    const int nb = sq / qblock_side;
    const int n_qb = nb * nb;
    // Per axis and per key scale: the range of kept key blocks [u0, u1) for query
    // block coordinate qb.  The window of +-radius query blocks is clipped to the
    // grid, mapped into the key scale (low end rounded down, high end up), and
    // widened to that scale's blocks.
    auto block_range = [&](int qb, int s, int* u0, int* u1) {
        const long long lo = std::max(0ll, static_cast<long long>(qblock_side) * (qb - radius));
        const long long hi = std::min(static_cast<long long>(sq),
                                      static_cast<long long>(qblock_side) * (qb + radius + 1));
        const long long lo_s = lo * s / sq;
        const long long hi_s = (hi * s + sq - 1) / sq;
        *u0 = static_cast<int>(lo_s / qblock_side);
        *u1 = static_cast<int>((hi_s + qblock_side - 1) / qblock_side);
    };
    long long nnz = 0;
    for (int qb = 0; qb < n_qb; ++qb) {
        const int by = qb / nb, bx = qb % nb;
        if (row_ptr) row_ptr[qb] = static_cast<int32_t>(nnz);
        for (int sc = 0; sc <= step; ++sc) {
            const int s = p->side[sc];
            if (s <= sink_max_side) continue;
            int uy0, uy1, ux0, ux1;
            block_range(by, s, &uy0, &uy1);
            block_range(bx, s, &ux0, &ux1);
            for (int u = uy0; u < uy1; ++u)
                for (int w = ux0; w < ux1; ++w) {
                    if (entries) {
                        if (nnz >= entries_cap) return VAR_ERR_INVALID_ARG;
                        entries[nnz] = (sc << 24) | (u << 12) | w;
                    }
                    ++nnz;
                }
        }
    }
    if (nnz > 0x7fffffffll) return VAR_ERR_UNSUPPORTED;
    if (row_ptr) row_ptr[n_qb] = static_cast<int32_t>(nnz);
    if (nnz_out) *nnz_out = static_cast<int32_t>(nnz);
    if (n_qblocks_out) *n_qblocks_out = n_qb;
    if (sink_len_out) *sink_len_out = sink_len;
    return VAR_OK;
}

int var_block_mask_plan(const var_problem* p, int32_t step, int32_t qblock_side, const int32_t* row_ptr,
                        const int32_t* entries, int32_t sink_len, int32_t* sq_ptr, int32_t* sq_units,
                        int32_t units_cap, int32_t* sq_order, int32_t* n_squares_out, int32_t* n_units_out)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (qblock_side != 8) return VAR_ERR_UNSUPPORTED;
    if (!row_ptr || !entries || sink_len < 0 || sink_len > g.L) return VAR_ERR_INVALID_ARG;
    if (g.side % 8 != 0) return VAR_ERR_UNSUPPORTED;
    const int nb = g.side / 8, nsq = (nb + 1) / 2, n_sq = nsq * nsq;
    const int n_sink = (sink_len + 63) / 64;
    std::vector<int32_t> counts(n_sq);
    long long total = 0;
    for (int pass = 0; pass < 2; ++pass) {
        total = 0;
        for (int sq = 0; sq < n_sq; ++sq) {
            const int by0 = 2 * (sq / nsq), bx0 = 2 * (sq % nsq);
            // the union of the (up to) four blocks' sorted lists with membership bits
            std::vector<std::pair<int32_t, uint32_t>> uni;
            for (int t = 0; t < 4; ++t) {
                const int by = by0 + (t >> 1), bx = bx0 + (t & 1);
                if (by >= nb || bx >= nb) continue;
                const int qb = by * nb + bx;
                if (row_ptr[qb] < 0 || row_ptr[qb + 1] < row_ptr[qb]) return VAR_ERR_INVALID_ARG;
                for (int i = row_ptr[qb]; i < row_ptr[qb + 1]; ++i) {
                    const int32_t e = entries[i];
                    const int sc = e >> 24, u = (e >> 12) & 0xFFF, v = e & 0xFFF;
                    if (e < 0 || sc > step || u >= (p->side[sc] + 7) / 8 || v >= (p->side[sc] + 7) / 8)
                        return VAR_ERR_INVALID_ARG;
                    uni.emplace_back(e, 1u << t);
                }
            }
            std::sort(uni.begin(), uni.end());
            std::vector<std::pair<int32_t, uint32_t>> merged;
            for (const auto& x : uni) {
                if (!merged.empty() && merged.back().first == x.first) merged.back().second |= x.second;
                else merged.push_back(x);
            }
            const int cnt = n_sink + static_cast<int>(merged.size());
            if (cnt > SPARSE_MAX_UNITS) return VAR_ERR_UNSUPPORTED;
            if (pass == 1) {
                if (sq_ptr) sq_ptr[sq] = static_cast<int32_t>(total);
                int32_t* out = sq_units + 2 * total;
                for (int c = 0; c < n_sink; ++c) {
                    const uint32_t n = static_cast<uint32_t>(std::min(64, sink_len - 64 * c));
                    out[2 * c] = -1 - c;
                    out[2 * c + 1] = static_cast<int32_t>(0xFu | META_SINK | (n == 64 ? META_FULL : 0u) | (n << 16));
                }
                for (size_t m = 0; m < merged.size(); ++m) {
                    const int32_t e = merged[m].first;
                    const int s = p->side[e >> 24], u = (e >> 12) & 0xFFF, v = e & 0xFFF;
                    const uint32_t rows = static_cast<uint32_t>(std::min(8, s - 8 * u));
                    const uint32_t cols = static_cast<uint32_t>(std::min(8, s - 8 * v));
                    out[2 * (n_sink + m)] = e;
                    out[2 * (n_sink + m) + 1] = static_cast<int32_t>(merged[m].second | (rows << 8) | (cols << 12) |
                                                                     ((rows == 8 && cols == 8) ? META_FULL : 0u));
                }
            }
            counts[sq] = cnt;
            total += cnt;
        }
        if (pass == 0) {
            if (n_squares_out) *n_squares_out = n_sq;
            if (n_units_out) *n_units_out = static_cast<int32_t>(total);
            if (!sq_units) return VAR_OK;
            if (total > units_cap || !sq_ptr || !sq_order) return VAR_ERR_INVALID_ARG;
        }
    }
    sq_ptr[n_sq] = static_cast<int32_t>(total);
    // squares with more units first (ties: lower index), so the longest CTAs start earliest
    std::vector<int32_t> order(n_sq);
    for (int i = 0; i < n_sq; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return counts[a] > counts[b]; });
    for (int i = 0; i < n_sq; ++i) sq_order[i] = order[i];
    return VAR_OK;
}

// ---------------------------------------------------------------- dynamic sparse pattern

namespace {

// The decision step's units (see UnitMap).  The decision scale must be a
// non-sink scale whose side is a multiple of 8, and the sink scales a prefix.
int build_unit_map(const var_problem* p, int32_t d, int32_t sink_max_side, varattn::UnitMap* m)
{
    using namespace varattn;
    StepGeom g;
    if (int rc = resolve(p, d, &g)) return rc;
    if (sink_max_side < 0) return VAR_ERR_INVALID_ARG;
    if (g.side % 8 != 0 || g.side <= sink_max_side) return VAR_ERR_UNSUPPORTED;
    *m = UnitMap{};
    m->L = g.L;
    int sc = 0, off = 0;
    while (sc <= d && p->side[sc] <= sink_max_side) {
        off += p->side[sc] * p->side[sc];
        ++sc;
    }
    m->sink_len = off;
    m->n_sink = (off + 63) / 64;
    int u = m->n_sink;
    for (; sc <= d; ++sc) {
        const int s = p->side[sc];
        if (s <= sink_max_side) return VAR_ERR_UNSUPPORTED;   // a sink scale after a non-sink one
        const int nbs = (s + 7) / 8;
        if (nbs > 4095) return VAR_ERR_UNSUPPORTED;
        m->sc[m->n_sc] = sc;
        m->off[m->n_sc] = off;
        m->side[m->n_sc] = s;
        m->ubase[m->n_sc] = u;
        ++m->n_sc;
        u += nbs * nbs;
        off += s * s;
    }
    m->U = u;
    return VAR_OK;
}

}  // namespace

size_t var_workspace_bytes(const var_problem* p, int32_t step, int32_t channels, int32_t keep_k)
{
    StepGeom g;
    if (resolve(p, step, &g) || keep_k < 0 || keep_k > g.N) return 0;
    return var_pivot_workspace_bytes(p, step, channels);
}

int var_selftest_wait_timeout(int32_t limit_us, int32_t* status, void* stream)
{
    if (limit_us <= 0 || limit_us > 10000000) return VAR_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(status) & 3u) return VAR_ERR_INVALID_ARG;
    int32_t* word = status ? status : varattn::device_status_ptr();
    if (!word) return VAR_ERR_CUDA;
    return varattn::launch_wait_timeout(limit_us, static_cast<cudaStream_t>(stream), word);
}

int var_sparvar_units(const var_problem* p, int32_t decision_step, int32_t sink_max_side, int32_t* n_units_out,
                      int32_t* n_sink_units_out)
{
    varattn::UnitMap m;
    if (int rc = build_unit_map(p, decision_step, sink_max_side, &m)) return rc;
    if (n_units_out) *n_units_out = m.U;
    if (n_sink_units_out) *n_sink_units_out = m.n_sink;
    return VAR_OK;
}

size_t var_sparvar_workspace_bytes(const var_problem* p, int32_t decision_step, int32_t sink_max_side)
{
    StepGeom g;
    if (resolve(p, decision_step, &g)) return 0;
    varattn::UnitMap m;
    if (build_unit_map(p, decision_step, sink_max_side, &m)) return 0;
    return varattn::sparvar_workspace_bytes(g, m.U);
}

int var_sparvar_scores_fast(const var_problem* p, int32_t decision_step, int32_t sink_max_side, const void* q,
                            const void* k, const float* lse, void* workspace, size_t workspace_bytes, double* scores,
                            void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, decision_step, &g)) return rc;
    varattn::UnitMap m;
    if (int rc = build_unit_map(p, decision_step, sink_max_side, &m)) return rc;
    if (!q || !k || !lse || !workspace || !scores) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(lse) & 3) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) || (reinterpret_cast<uintptr_t>(scores) & 7))
        return VAR_ERR_UNSUPPORTED;
    if (workspace_bytes < varattn::sparvar_workspace_bytes(g, m.U)) return VAR_ERR_WORKSPACE;
    if ((g.side / 8) * (g.side / 8) > 64) return VAR_ERR_UNSUPPORTED;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return varattn::launch_sparvar_scores_fast(g, m, q, k, lse, workspace, workspace_bytes, scores,
                                               static_cast<cudaStream_t>(stream), status);
}

int var_sparvar_scores(const var_problem* p, int32_t decision_step, int32_t sink_max_side, double tau, int32_t flags,
                       const void* q, const void* k, void* workspace, size_t workspace_bytes, double* scores,
                       int32_t* rescored, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, decision_step, &g)) return rc;
    varattn::UnitMap m;
    if (int rc = build_unit_map(p, decision_step, sink_max_side, &m)) return rc;
    if (!q || !k || !workspace || !scores) return VAR_ERR_INVALID_ARG;
    if (!(tau >= 0.0 && tau <= 1.0) || (flags & ~VAR_SPARVAR_RESCORE_ALL)) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
        (reinterpret_cast<uintptr_t>(scores) & 7) || (reinterpret_cast<uintptr_t>(rescored) & 3))
        return VAR_ERR_UNSUPPORTED;
    if (workspace_bytes < varattn::sparvar_workspace_bytes(g, m.U)) return VAR_ERR_WORKSPACE;
    // the fp64 softmax scale of the definition: 1/sqrt(head_dim) rounded once, or the caller's value
    const double scale64 = p->softmax_scale == 0.f ? 1.0 / std::sqrt(static_cast<double>(p->head_dim))
                                                   : static_cast<double>(p->softmax_scale);
    return varattn::launch_sparvar_scores(g, m, q, k, tau, (flags & VAR_SPARVAR_RESCORE_ALL) ? 1 : 0, scale64,
                                          workspace, workspace_bytes, scores, rescored,
                                          static_cast<cudaStream_t>(stream));
}

int var_sparvar_mask_build(const var_problem* p, int32_t decision_step, int32_t step, int32_t sink_max_side,
                           const double* scores, double tau, int32_t* row_ptr, int32_t* entries,
                           int32_t entries_cap, int32_t* nnz_out, int32_t* n_qblocks_out, int32_t* sink_len_out)
{
    varattn::UnitMap m;
    if (int rc = build_unit_map(p, decision_step, sink_max_side, &m)) return rc;
    StepGeom gk;
    if (int rc = resolve(p, step, &gk)) return rc;
    if (step < decision_step || !scores || !(tau >= 0.0 && tau <= 1.0)) return VAR_ERR_INVALID_ARG;
    if (gk.side % 8 != 0) return VAR_ERR_UNSUPPORTED;
    for (int sc = decision_step + 1; sc <= step; ++sc)
        if ((p->side[sc] + 7) / 8 > 4095) return VAR_ERR_UNSUPPORTED;
    const int s_d = p->side[decision_step];
    const int nb_d = s_d / 8, nb_k = gk.side / 8;
    const int n_qb_d = nb_d * nb_d;
    // Selection per decision block: the sinks, then the other units by decreasing
    // score (equal scores: lower unit first) until the kept mass, added in fp64 in
    // that order, reaches tau of the row's total (added in unit order).
    std::vector<std::vector<int32_t>> blocks(n_qb_d);     // the kept blocks' entries per decision block
    std::vector<int> order(m.U - m.n_sink);
    for (int qb = 0; qb < n_qb_d; ++qb) {
        const double* row = scores + static_cast<size_t>(qb) * m.U;
        double total = 0.0, have = 0.0;
        for (int u = 0; u < m.U; ++u) total += row[u];
        for (int u = 0; u < m.n_sink; ++u) have += row[u];
        for (int i = 0; i < m.U - m.n_sink; ++i) order[i] = m.n_sink + i;
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return row[a] > row[b]; });
        std::vector<int32_t>& out = blocks[qb];
        for (int u : order) {
            if (have >= tau * total) break;
            have += row[u];
            // unit u -> (scale, block row, block column)
            int t = 0;
            while (t + 1 < m.n_sc && u >= m.ubase[t + 1]) ++t;
            const int s = m.side[t], nbs = (s + 7) / 8;
            const int bu = (u - m.ubase[t]) / nbs, bv = (u - m.ubase[t]) % nbs;
            const int sc = m.sc[t];
            if (sc < decision_step) {
                out.push_back((sc << 24) | (bu << 12) | bv);
                continue;
            }
            // a block of the decision scale: itself, and by index mapping the blocks of
            // every later scale up to `step` that meet it rescaled (rounded outward)
            const long long r0 = 8ll * bu, r1 = std::min(8ll * bu + 8, static_cast<long long>(s_d));
            const long long c0 = 8ll * bv, c1 = std::min(8ll * bv + 8, static_cast<long long>(s_d));
            for (int sc2 = decision_step; sc2 <= step; ++sc2) {
                const long long s2 = p->side[sc2];
                const long long lo_r = r0 * s2 / s_d, hi_r = (r1 * s2 + s_d - 1) / s_d;
                const long long lo_c = c0 * s2 / s_d, hi_c = (c1 * s2 + s_d - 1) / s_d;
                for (long long uu = lo_r / 8; uu < (hi_r + 7) / 8; ++uu)
                    for (long long vv = lo_c / 8; vv < (hi_c + 7) / 8; ++vv)
                        out.push_back(static_cast<int32_t>((sc2 << 24) | (uu << 12) | vv));
            }
        }
        std::sort(out.begin(), out.end());
        out.erase(std::unique(out.begin(), out.end()), out.end());
    }
    // Index mapping of the query blocks: target block (by, bx) takes the decision
    // block under its centre.
    long long nnz = 0;
    for (int qb = 0; qb < nb_k * nb_k; ++qb) {
        const int by = qb / nb_k, bx = qb % nb_k;
        const int dy = static_cast<int>((2ll * by + 1) * nb_d / (2ll * nb_k));
        const int dx = static_cast<int>((2ll * bx + 1) * nb_d / (2ll * nb_k));
        const std::vector<int32_t>& src = blocks[dy * nb_d + dx];
        if (row_ptr) row_ptr[qb] = static_cast<int32_t>(nnz);
        if (entries) {
            if (nnz + static_cast<long long>(src.size()) > entries_cap) return VAR_ERR_INVALID_ARG;
            std::copy(src.begin(), src.end(), entries + nnz);
        }
        nnz += static_cast<long long>(src.size());
        if (nnz > 0x7fffffffll) return VAR_ERR_UNSUPPORTED;
    }
    if (row_ptr) row_ptr[nb_k * nb_k] = static_cast<int32_t>(nnz);
    if (nnz_out) *nnz_out = static_cast<int32_t>(nnz);
    if (n_qblocks_out) *n_qblocks_out = nb_k * nb_k;
    if (sink_len_out) *sink_len_out = m.sink_len;
    return VAR_OK;
}

int var_attn_blocksparse(const var_problem* p, int32_t step, const void* q, const void* k,
                         const void* v, const var_block_mask* mask, void* o, void* stream)
{
    StepGeom g;
    if (int rc = resolve(p, step, &g)) return rc;
    if (!q || !k || !v || !o || !mask || !mask->row_ptr || !mask->entries) return VAR_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return VAR_ERR_UNSUPPORTED;
    if (mask->qblock_side <= 0 || g.side % mask->qblock_side != 0) return VAR_ERR_INVALID_ARG;
    const int nb = g.side / mask->qblock_side;
    if (mask->n_qblocks != nb * nb || mask->sink_len < 0 || mask->sink_len > g.L || mask->nnz < 0)
        return VAR_ERR_INVALID_ARG;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    return launch_attn_blocksparse(g, p->side, p->n_scales, step, q, k, v, mask, o,
                                   static_cast<cudaStream_t>(stream), status);
}

int32_t var_keep_count(int32_t n, int32_t num, int32_t den)
{
    if (n < 0 || num < 0 || den <= 0 || num > den) return -1;
    return static_cast<int32_t>(static_cast<int64_t>(n) * num / den);
}

const char* var_status_string(int status)
{
    switch (status) {
    case VAR_OK: return "ok";
    case VAR_ERR_INVALID_ARG: return "invalid argument";
    case VAR_ERR_UNSUPPORTED: return "unsupported configuration";
    case VAR_ERR_CUDA: return "CUDA runtime error";
    case VAR_ERR_TIMEOUT: return "device pipeline wait timed out";
    case VAR_ERR_NUMERIC: return "input outside the exactly handled numeric range";
    case VAR_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

int var_device_status(int32_t* status_out, int32_t clear)
{
    if (!status_out) return VAR_ERR_INVALID_ARG;
    int32_t* p = device_status_ptr();
    if (!p) return VAR_ERR_CUDA;
    if (rt().device_sync() != cudaSuccess) return VAR_ERR_CUDA;
    int32_t v = 0;
    if (rt().memcpy_async(&v, p, sizeof v, cudaMemcpyDeviceToHost, nullptr) != cudaSuccess ||
        rt().stream_sync(nullptr) != cudaSuccess)
        return VAR_ERR_CUDA;
    *status_out = v;
    if (clear && v != 0) {
        if (rt().memset_async(p, 0, sizeof v, nullptr) != cudaSuccess || rt().stream_sync(nullptr) != cudaSuccess)
            return VAR_ERR_CUDA;
    }
    return VAR_OK;
}

int var_check_status(const int32_t* status, int32_t* status_out, int32_t clear, void* stream)
{
    if (!status_out || (reinterpret_cast<uintptr_t>(status) & 3u)) return VAR_ERR_INVALID_ARG;
    int32_t* p = status ? const_cast<int32_t*>(status) : device_status_ptr();
    if (!p) return VAR_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (rt().memcpy_async(&v, p, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        rt().stream_sync(st) != cudaSuccess)
        return VAR_ERR_CUDA;
    *status_out = v;
    if (clear && v != 0) {
        if (rt().memset_async(p, 0, sizeof v, st) != cudaSuccess || rt().stream_sync(st) != cudaSuccess)
            return VAR_ERR_CUDA;
    }
    return VAR_OK;
}

}  // extern "C"
