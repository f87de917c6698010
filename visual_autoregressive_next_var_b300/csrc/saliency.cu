// Attention-guided pivot selection for sm_103a ("ARVAR" Key Design 2:
// attention retrospect).  The importance of the current step's positions is
// read from the attention of an earlier, smaller step T-M of the same layer:
// that step's self-attention block (its queries against its own scale's keys)
// is aggregated into a spatial saliency per source position, the map is
// interpolated to the current grid, and the Top-K positions are the pivots.
//
// Aggregation (the pages leave the axis open, and note that averaging each
// row of a row-normalised matrix is constant): the probability a source key
// receives, averaged over the source step's queries and over the heads,
//   sal[b, j] = 1/(H N') sum_h sum_i softmax_h(i, L' - N' + j),
// with the softmax over all L' keys the source step attends.
//
//   saliency_kernel      per (b, h) and 128 keys of the self block: S^T =
//                        K_self Q^T on the tensor cores (tcgen05, TMEM),
//                        p = 2^(s scale log2e - lse_i) with the row
//                        log2-sum-exp the source step's dense attention wrote,
//                        summed over the queries by the thread owning the key
//                        row (no cross-thread reduction); written per head.
//   guided_upsample      head mean, bilinear upsampling to the current grid
//                        (half-pixel centres, edge clamp, as the restore), one
//                        thread per target token.
//   selection            the pivot selection kernel on exact keys (equal
//                        values: the lower flat index first).
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace varattn {

namespace {

template <int D>
struct SalLayout {
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = 128 * 128;      // 128 rows x 64 bf16, 128-byte swizzle
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int NSQ = 2;                      // query tile ring
    static constexpr int OFF_K = 0;                    // the CTA's 128 keys (A operand)
    static constexpr int OFF_Q = OFF_K + TILE_BYTES;   // query tiles (B operand)
    static constexpr int OFF_LSE = OFF_Q + NSQ * TILE_BYTES;   // [4 warps][128] float, warp-private
    static constexpr int OFF_BAR = OFF_LSE + 4 * 128 * 4;
    static constexpr int B_KF = 0;                     // key tile resident
    static constexpr int B_QF = 1;                     // [NSQ] query slot full
    static constexpr int B_QE = B_QF + NSQ;            // [NSQ] query slot free
    static constexpr int B_SF = B_QE + NSQ;            // [2] S^T buffer computed
    static constexpr int B_SE = B_SF + 2;              // [2] S^T buffer consumed
    static constexpr int B_DR = B_SE + 2;              // drain before teardown
    static constexpr int NBAR = B_DR + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 256;         // two 128-column S^T buffers
};

struct SalMaps {
    CUtensorMap q;    // 3-D (D, N', B*H), box (64, 128, 1)
    CUtensorMap k;    // 3-D (D, L', B*H), box (64, 128, 1)
};

struct SalArgs {
    int32_t n_src;          // N' = source grid tokens (the self block)
    int32_t self0;          // L' - N': first key row of the self block
    int32_t n_qt;           // ceil(N' / 128)
    int32_t key_tiles;      // ceil(N' / 128) key tiles per (b, h)
    float scale_log2;       // softmax scale * log2(e)
    const float* lse;       // [B*H][N'] row log2-sum-exp
    float* sal;             // [B*H][N'] per-head sums over the queries
    int32_t* status;
};

__device__ __forceinline__ void record_fault(volatile int* abort_flag, int32_t* status, int code)
{
    *abort_flag = 1;
    atomicCAS(status, 0, code);
}

template <int D>
__global__ void __launch_bounds__(256, 2) saliency_kernel(const __grid_constant__ SalMaps maps, const SalArgs a)
{
    using Lay = SalLayout<D>;
    constexpr int NSQ = Lay::NSQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + Lay::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::OFF_MISC + 4);

    const int bh = blockIdx.x / a.key_tiles;
    const int kt = blockIdx.x - bh * a.key_tiles;
    const int n_qt = a.n_qt;

    if (threadIdx.x == 0) {
        mbar_init(bar(Lay::B_KF), 1);
        for (int s = 0; s < NSQ; ++s) {
            mbar_init(bar(Lay::B_QF + s), 1);
            mbar_init(bar(Lay::B_QE + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(Lay::B_SF + t), 1);
            mbar_init(bar(Lay::B_SE + t), 128);
        }
        mbar_init(bar(Lay::B_DR), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(Lay::B_KF), Lay::TILE_BYTES);
            for (int hh = 0; hh < Lay::HALVES; ++hh)
                tma_load_3d(sbase + Lay::OFF_K + hh * Lay::HALF_BYTES, &maps.k, hh * 64, a.self0 + kt * 128, bh,
                            bar(Lay::B_KF));
            int issued = 0;
            for (int t = 0; t < n_qt; ++t) {
                const int s = t % NSQ;
                if (!mbar_wait(bar(Lay::B_QE + s), ((t / NSQ) & 1) ^ 1, abort_flag)) {
                    record_fault(abort_flag, a.status, VAR_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(bar(Lay::B_QF + s), Lay::TILE_BYTES);
                for (int hh = 0; hh < Lay::HALVES; ++hh)
                    tma_load_3d(sbase + Lay::OFF_Q + s * Lay::TILE_BYTES + hh * Lay::HALF_BYTES, &maps.q, hh * 64,
                                t * 128, bh, bar(Lay::B_QF + s));
                ++issued;
            }
            // every copy this thread started lands before the CTA may exit
            mbar_wait(bar(Lay::B_KF), 0, nullptr);
            for (int t = (issued > NSQ ? issued - NSQ : 0); t < issued; ++t)
                mbar_wait(bar(Lay::B_QF + t % NSQ), (t / NSQ) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer: S^T = K Q^T
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16(128, 128, false, false);
            bool ok = mbar_wait(bar(Lay::B_KF), 0, abort_flag);
            for (int t = 0; ok && t < n_qt; ++t) {
                const int s = t % NSQ, buf = t & 1;
                ok = mbar_wait(bar(Lay::B_QF + s), (t / NSQ) & 1, abort_flag) &&
                     mbar_wait(bar(Lay::B_SE + buf), ((t >> 1) & 1) ^ 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint32_t ka = sbase + Lay::OFF_K;
                const uint32_t qb = sbase + Lay::OFF_Q + s * Lay::TILE_BYTES;
                const uint32_t dst = tmem + static_cast<uint32_t>(buf * 128);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * Lay::HALF_BYTES + (kk % 4) * 32;
                    umma_ss(dst, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qb + off, 16, 1024), IDESC,
                            kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(Lay::B_SF + buf));
                umma_commit(bar(Lay::B_QE + s));
            }
            if (!ok) record_fault(abort_flag, a.status, VAR_ERR_TIMEOUT);
            umma_commit(bar(Lay::B_DR));
            mbar_wait(bar(Lay::B_DR), 0, nullptr);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ consumers: one key row each
        // Each warp stages a tile's 128 query statistics in its own slice of shared
        // memory (4 per lane) and reads them back as broadcast 16-byte loads.
        const int r = (warp & 3) * 32 + lane;
        float* lw = reinterpret_cast<float*>(smem + Lay::OFF_LSE) + (warp & 3) * 128;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float sl2 = a.scale_log2;
        const float* lse_bh = a.lse + static_cast<size_t>(bh) * a.n_src;
        uint64_t acc2 = f2_pack(0.f, 0.f);
        bool ok = true;
        for (int t = 0; t < n_qt; ++t) {
            const int buf = t & 1;
            const int q0 = t * 128;
            if (!mbar_wait(bar(Lay::B_SF + buf), (t >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            __syncwarp();                              // the previous tile's reads are done
#pragma unroll
            for (int e = 0; e < 4; ++e) {              // columns past N': probability 0
                const int qi = q0 + lane * 4 + e;
                lw[lane * 4 + e] = qi < a.n_src ? __ldg(lse_bh + qi) : INFINITY;
            }
            __syncwarp();
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t sv[32];
                tmem_ld32(tmem + lane_base + static_cast<uint32_t>(buf * 128 + c0), sv);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(lw + c0 + c);
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sv[c]), sl2, -l4.x));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(sv[c + 1]), sl2, -l4.y));
                    const float p2 = ex2_approx(fmaf(__uint_as_float(sv[c + 2]), sl2, -l4.z));
                    const float p3 = ex2_approx(fmaf(__uint_as_float(sv[c + 3]), sl2, -l4.w));
                    acc2 = f2_add(acc2, f2_pack(p0, p1));
                    acc2 = f2_add(acc2, f2_pack(p2, p3));
                }
            }
            tc_fence_before();
            mbar_arrive(bar(Lay::B_SE + buf));
        }
        if (!ok) {
            record_fault(abort_flag, a.status, VAR_ERR_TIMEOUT);
        } else {
            float s0, s1;
            f2_unpack(acc2, s0, s1);
            const int j = kt * 128 + r;
            if (j < a.n_src) a.sal[static_cast<size_t>(bh) * a.n_src + j] = s0 + s1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::TMEM_COLS);
    }
}

// head mean of the per-head sums, bilinear upsampling from the sp x sp source
// grid to the s x s grid; keys for the selection (lo = hi = the value)
__global__ void __launch_bounds__(256)
    guided_upsample_kernel(const float* __restrict__ sal, int H, int sp, int s, float ratio, float inv_hn,
                           float* __restrict__ lo, float* __restrict__ hi, float* __restrict__ scores)
{
    // the top-K kernel that follows (a programmatic dependent) may set up now;
    // it reads lo / hi only after this grid has completed
    pdl_launch_dependents();
    const int b = blockIdx.y;
    const int N = s * s, Np = sp * sp;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N) return;
    const int y = t / s, x = t - y * s;
    const float sy = fmaxf((static_cast<float>(y) + 0.5f) * ratio - 0.5f, 0.f);
    const float sx = fmaxf((static_cast<float>(x) + 0.5f) * ratio - 0.5f, 0.f);
    const int y0 = min(static_cast<int>(sy), sp - 1), x0 = min(static_cast<int>(sx), sp - 1);
    const int y1 = min(y0 + 1, sp - 1), x1 = min(x0 + 1, sp - 1);
    const float ly = sy - static_cast<float>(y0), lx = sx - static_cast<float>(x0);
    const int src[4] = {y0 * sp + x0, y0 * sp + x1, y1 * sp + x0, y1 * sp + x1};
    float m[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float acc = 0.f;
        for (int h = 0; h < H; ++h) acc += __ldg(sal + (static_cast<size_t>(b) * H + h) * Np + src[q]);
        m[q] = acc * inv_hn;
    }
    const float v = (1.f - ly) * ((1.f - lx) * m[0] + lx * m[1]) + ly * ((1.f - lx) * m[2] + lx * m[3]);
    const size_t o = static_cast<size_t>(b) * N + t;
    lo[o] = v;
    hi[o] = v;
    if (scores) scores[o] = v;
}

struct GuidedWs {
    size_t lo, hi, band_idx, band_score, total;
};

inline GuidedWs guided_ws_layout(int B, int N)
{
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    GuidedWs w{};
    size_t o = 0;
    w.lo = o;         o = al(o + sizeof(float) * B * N);
    w.hi = o;         o = al(o + sizeof(float) * B * N);
    w.band_idx = o;   o = al(o + sizeof(int) * B * N);
    w.band_score = o; o = al(o + sizeof(double) * B * N);
    w.total = o;
    return w;
}

template <int D>
int launch_saliency_d(const StepGeom& g, int n_src, int L_src, const void* q, const void* k, const float* lse,
                      float* sal, cudaStream_t st, int32_t* status)
{
    using Lay = SalLayout<D>;
    if (ensure_smem_attr(saliency_kernel<D>, Lay::SMEM_BYTES) != cudaSuccess) return VAR_ERR_CUDA;
    SalMaps maps;
    const uint64_t BH = static_cast<uint64_t>(g.B) * g.H;
    const uint32_t box[3] = {64, 128, 1};
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(n_src), BH};
        const uint64_t strides[2] = {D * 2ull, static_cast<uint64_t>(n_src) * D * 2ull};
        if (int rc = encode_tmap_bf16(&maps.q, q, 3, dims, strides, box)) return rc;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(L_src), BH};
        const uint64_t strides[2] = {D * 2ull, static_cast<uint64_t>(g.cap) * D * 2ull};
        if (int rc = encode_tmap_bf16(&maps.k, k, 3, dims, strides, box)) return rc;
    }
    SalArgs a{};
    a.n_src = n_src;
    a.self0 = L_src - n_src;
    a.n_qt = (n_src + 127) / 128;
    a.key_tiles = (n_src + 127) / 128;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.lse = lse;
    a.sal = sal;
    a.status = status;
    const uint64_t grid = BH * static_cast<uint64_t>(a.key_tiles);
    if (grid > 0x7fffffffull) return VAR_ERR_UNSUPPORTED;
    return cuda_status(launch_kernel(saliency_kernel<D>, dim3(static_cast<unsigned>(grid)), dim3(256), Lay::SMEM_BYTES,
                                     st, false, maps, a));
}

}  // namespace

int launch_saliency(const StepGeom& g, int n_src, int L_src, const void* q, const void* k, const float* lse,
                    float* sal, cudaStream_t st, int32_t* status)
{
    if (g.D == 128) return launch_saliency_d<128>(g, n_src, L_src, q, k, lse, sal, st, status);
    if (g.D == 64) return launch_saliency_d<64>(g, n_src, L_src, q, k, lse, sal, st, status);
    return VAR_ERR_UNSUPPORTED;
}

size_t guided_workspace_bytes(int B, int N) { return guided_ws_layout(B, N).total; }

int launch_guided_pivot(int B, int H, int sp, int s, const float* sal, int keep_k, int32_t* idx, float* scores,
                        void* ws, size_t ws_bytes, cudaStream_t st, int32_t* status)
{
    const int N = s * s;
    const GuidedWs w = guided_ws_layout(B, N);
    if (ws_bytes < w.total) return VAR_ERR_WORKSPACE;
    auto* base = static_cast<uint8_t*>(ws);
    auto* lo = reinterpret_cast<float*>(base + w.lo);
    auto* hi = reinterpret_cast<float*>(base + w.hi);
    const dim3 grid((N + 255) / 256, B);
    if (launch_kernel(guided_upsample_kernel, grid, dim3(256), 0, st, false, sal, H, sp, s,
                      static_cast<float>(sp) / static_cast<float>(s),
                      1.0f / (static_cast<float>(H) * static_cast<float>(sp * sp)), lo, hi, scores) != cudaSuccess)
        return VAR_ERR_CUDA;
    if (keep_k == 0) return VAR_OK;
    return launch_select_exact(B, N, keep_k, lo, hi, reinterpret_cast<int*>(base + w.band_idx),
                               reinterpret_cast<double*>(base + w.band_score), idx, st, status);
}

}  // namespace varattn
