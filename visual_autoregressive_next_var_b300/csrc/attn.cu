// Dense and pruned (gathered-query) cross-scale attention: host launchers of
// the shared kernel in attn_kernel.cuh.
#include <cstring>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "attn_kernel.cuh"

namespace varattn {

// ---------------------------------------------------------------------------- CTA plan

// A pair CTA runs two 128-row query tiles against every key tile; a split CTA
// runs one tile with its key tiles shared out between the two softmax groups
// (about half the pair's time).  Plan A: all pair slots as pair CTAs (plus the
// odd last tiles as split CTAs).  Plan B: pair CTAs for whole waves only, the
// rest as split CTAs, which shortens a partial last wave of pairs.  The plan
// with the smaller greedy-dispatch makespan is used; plans are cached per shape.
struct TilePlan {
    int n_pair_ctas, n_conv_slots, grid;
};

static double dispatch_makespan(int pairs, int singles, int n_sms)
{
    constexpr double kSplitCost = 0.6;   // split CTA time relative to a pair CTA
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < n_sms; ++i) free_at.push(0.0);
    double end = 0.0;
    for (int i = 0; i < pairs + singles; ++i) {
        const double t = free_at.top() + (i < pairs ? 1.0 : kSplitCost);
        free_at.pop();
        free_at.push(t);
        end = t > end ? t : end;
    }
    return end;
}

static TilePlan plan_tiles(int bh, int tiles_per_bh, int n_sms)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, TilePlan> cache;
    const auto key = std::make_tuple(bh, tiles_per_bh, n_sms);
    if (!rt_mocked()) {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int slots = bh * (tiles_per_bh / 2);
    const int odd = (tiles_per_bh & 1) ? bh : 0;
    TilePlan a{slots, 0, slots + odd};
    const int keep = n_sms * (slots / n_sms);
    TilePlan b{keep, slots - keep, keep + 2 * (slots - keep) + odd};
    TilePlan best = a;
    if (b.n_conv_slots > 0 && slots + odd <= 1 << 16 &&
        dispatch_makespan(b.n_pair_ctas, b.grid - b.n_pair_ctas, n_sms) <
            dispatch_makespan(a.n_pair_ctas, a.grid - a.n_pair_ctas, n_sms) - 1e-9)
        best = b;
    if (rt_mocked()) return best;
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = best;
    return best;
}

// ---------------------------------------------------------------------------- host

template <int D, int MODE>
static int launch_attn(const StepGeom& g, const void* q, const void* k, const void* v,
                       const int32_t* idx, int n_rows, void* o, cudaStream_t st, int32_t* status,
                       bool halved = false, bool scatter = false, float* lse = nullptr, bool pdl = false)
// pdl: a programmatic dependent launch (only the gathered mode takes one; the
// kernel waits for its predecessor after its set-up, before reading inputs)
{
    using Lay = AttnLayout<D>;
    auto kern = attn_kernel<D, MODE, DenseMaps>;
    if (n_rows == 0) return VAR_OK;
    if (ensure_smem_attr(kern, Lay::SMEM_BYTES) != cudaSuccess) return VAR_ERR_CUDA;

    DenseMaps maps;
    CUtensorMap& tq = maps.q;
    CUtensorMap& tk = maps.k;
    CUtensorMap& tv = maps.v;
    const uint32_t box[3] = {64, 128, 1};
    const uint64_t BH = static_cast<uint64_t>(g.B) * g.H;
    // branch halving: CTAs cover the first B/2 batch elements (the conditional branch)
    const uint64_t BH_run = halved ? BH / 2 : BH;
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
    std::memset(&maps.o, 0, sizeof maps.o);
    if (MODE == MODE_DENSE) {
        // the output rows, for the epilogue's tile stores (all B*H, so a repeated
        // half lands inside the map)
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(n_rows), BH};
        const uint64_t strides[2] = {D * 2ull, static_cast<uint64_t>(n_rows) * D * 2ull};
        if (int rc = encode_tmap_bf16(&maps.o, o, 3, dims, strides, box)) return rc;
    }
    AttnArgs a = {};
    a.n_rows = n_rows;
    a.n_q = g.N;
    a.L = g.L;
    a.heads = g.H;
    a.tiles_per_bh = (n_rows + 127) / 128;
    a.slots_per_bh = a.tiles_per_bh / 2;
    const int n_sms = sm_count();
    if (n_sms <= 0) return VAR_ERR_CUDA;
    const TilePlan plan = plan_tiles(static_cast<int>(BH_run), a.tiles_per_bh, n_sms);
    a.n_pair_ctas = plan.n_pair_ctas;
    a.n_conv_slots = plan.n_conv_slots;
    a.n_kv = (g.L + 127) / 128;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.idx = idx;
    a.o = static_cast<__nv_bfloat16*>(o);
    a.o_repeat = halved ? static_cast<int64_t>(BH_run) * n_rows * D : 0;
    a.scatter = scatter ? 1 : 0;
    a.lse = lse;
    a.status = status;
    return cuda_status(launch_kernel(kern, dim3(static_cast<unsigned>(plan.grid)), dim3(384), Lay::SMEM_BYTES, st,
                                     pdl, maps, a));
}

int launch_attn_dense(const StepGeom& g, const void* q, const void* k, const void* v, void* o,
                      cudaStream_t st, int32_t* status, float* lse)
{
    if (g.D == 128) return launch_attn<128, MODE_DENSE>(g, q, k, v, nullptr, g.N, o, st, status, false, false, lse);
    if (g.D == 64) return launch_attn<64, MODE_DENSE>(g, q, k, v, nullptr, g.N, o, st, status, false, false, lse);
    return VAR_ERR_UNSUPPORTED;
}

int launch_attn_pruned(const StepGeom& g, const void* q, const void* k, const void* v,
                       const int32_t* idx, int keep_k, void* o, cudaStream_t st, int32_t* status, bool scatter,
                       bool after_select)
{
    if (g.D == 128)
        return launch_attn<128, MODE_GATHER>(g, q, k, v, idx, keep_k, o, st, status, false, scatter, nullptr,
                                             after_select);
    if (g.D == 64)
        return launch_attn<64, MODE_GATHER>(g, q, k, v, idx, keep_k, o, st, status, false, scatter, nullptr,
                                            after_select);
    return VAR_ERR_UNSUPPORTED;
}

int launch_attn_dense_halved(const StepGeom& g, const void* q, const void* k, const void* v, void* o,
                             cudaStream_t st, int32_t* status)
{
    if (g.D == 128) return launch_attn<128, MODE_DENSE>(g, q, k, v, nullptr, g.N, o, st, status, true);
    if (g.D == 64) return launch_attn<64, MODE_DENSE>(g, q, k, v, nullptr, g.N, o, st, status, true);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
