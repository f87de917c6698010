// Dense and pruned (gathered-query) cross-scale attention for sm_103a.
//
// Computes, per (b, h) and query row i, softmax(q_i K^T * scale) V over the L
// tokens of scales 0..step ("SparVAR" abstract: every step attends to all
// tokens of the historical scales).  The pruned variant takes its query rows
// from an index list ("FastVAR" abstract, cached token pruning; "ARVAR" Key
// Design 2: Top-K indices gather the tokens that are recomputed).
//
// One CTA = one (b, h) and two 128-row query tiles (ping-pong), 12 warps:
//   warp 0      TMA producer: Q tiles once, then K_j / V_j into two rings
//   warp 1      UMMA issuer (one thread): S_t = Q_t K_j^T, O_t += P_t V_j
//   warp 2      tensor-memory allocator
//   warps 4-7   softmax group 0 (query tile 0, one thread per row)
//   warps 8-11  softmax group 1 (query tile 1)
// Tensor memory (512 columns): S0 | S1 | O0 | O1.  P_t (bf16) overwrites the
// first columns of S_t and feeds the PV product straight from tensor memory.
// The softmax is the online one in fp32 with exp2; the running maximum is
// only moved (and O rescaled) when a new maximum exceeds it by 2^8.
#include <cfloat>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace varattn {

template <int D>
struct AttnLayout {
    static constexpr int BM = 128;              // rows per query tile
    static constexpr int BN = 128;              // keys per KV tile
    static constexpr int HALVES = D / 64;       // 128-byte column slabs of a tile
    static constexpr int HALF_BYTES = 128 * 128;
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int NS = (D == 128) ? 2 : 4;   // ring depth (K and V each)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
    static constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_V + NS * TILE_BYTES;
    // barrier slots
    static constexpr int B_QF = 0;               // [2]  query tile t resident
    static constexpr int B_KF = 2;               // [NS] K slot full
    static constexpr int B_KE = B_KF + NS;       // [NS] K slot free
    static constexpr int B_VF = B_KE + NS;       // [NS] V slot full
    static constexpr int B_VE = B_VF + NS;       // [NS] V slot free
    static constexpr int B_SF = B_VE + NS;       // [2]  S_t computed
    static constexpr int B_PF = B_SF + 2;        // [2]  P_t written (and O_t rescaled)
    static constexpr int B_OF = B_PF + 2;        // [1]  all products done
    static constexpr int B_DR = B_OF + 1;        // [1]  drain before teardown
    static constexpr int NBAR = B_DR + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
};

struct AttnArgs {
    int32_t n_rows;         // output rows per (b,h): N (dense) or keep_k (pruned)
    int32_t n_q;            // rows of the Q tensor per (b,h)
    int32_t L;              // visible cached keys
    int32_t heads;
    int32_t pairs_per_bh;   // ceil(n_rows / 256)
    int32_t n_kv;           // ceil(L / 128)
    float scale_log2;       // softmax scale * log2(e)
    const __nv_bfloat16* q; // gather source (pruned)
    const int32_t* idx;     // [B][n_rows] (pruned)
    __nv_bfloat16* o;       // [B][H][n_rows][D]
    int32_t* status;
};

__device__ __forceinline__ void record_fault(volatile int* abort_flag, int32_t* status, int code)
{
    *abort_flag = 1;
    atomicCAS(status, 0, code);
}

template <int D, bool GATHER>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs args)
{
    using Lay = AttnLayout<D>;
    constexpr int NS = Lay::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + Lay::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::OFF_MISC + 4);

    const int bh = blockIdx.x / args.pairs_per_bh;
    const int row0 = (blockIdx.x % args.pairs_per_bh) * 256;
    const int n_kv = args.n_kv;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) mbar_init(bar(Lay::B_QF + t), GATHER ? 128 : 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(Lay::B_KF + s), 1);
            mbar_init(bar(Lay::B_KE + s), 1);
            mbar_init(bar(Lay::B_VF + s), 1);
            mbar_init(bar(Lay::B_VE + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(Lay::B_SF + t), 1);
            mbar_init(bar(Lay::B_PF + t), 128);
        }
        mbar_init(bar(Lay::B_OF), 1);
        mbar_init(bar(Lay::B_DR), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (!GATHER) tma_prefetch_desc(&tm_q);
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
            if (!GATHER) {
                for (int t = 0; t < 2; ++t) {
                    mbar_arrive_expect_tx(bar(Lay::B_QF + t), Lay::TILE_BYTES);
                    for (int hh = 0; hh < Lay::HALVES; ++hh)
                        tma_load_3d(sbase + Lay::OFF_Q + t * Lay::TILE_BYTES + hh * Lay::HALF_BYTES,
                                    &tm_q, hh * 64, row0 + t * 128, bh, bar(Lay::B_QF + t));
                }
            }
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % NS;
                const uint32_t ph = (j / NS) & 1;
                if (!mbar_wait(bar(Lay::B_KE + s), ph ^ 1, abort_flag)) {
                    record_fault(abort_flag, args.status, VAR_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(bar(Lay::B_KF + s), Lay::TILE_BYTES);
                for (int hh = 0; hh < Lay::HALVES; ++hh)
                    tma_load_3d(sbase + Lay::OFF_K + s * Lay::TILE_BYTES + hh * Lay::HALF_BYTES,
                                &tm_k, hh * 64, j * 128, bh, bar(Lay::B_KF + s));
                ++k_issued;
                if (!mbar_wait(bar(Lay::B_VE + s), ph ^ 1, abort_flag)) {
                    record_fault(abort_flag, args.status, VAR_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(bar(Lay::B_VF + s), Lay::TILE_BYTES);
                for (int hh = 0; hh < Lay::HALVES; ++hh)
                    tma_load_3d(sbase + Lay::OFF_V + s * Lay::TILE_BYTES + hh * Lay::HALF_BYTES,
                                &tm_v, hh * 64, j * 128, bh, bar(Lay::B_VF + s));
                ++v_issued;
            }
            // Every copy this thread started must land before the CTA may exit.
            for (int j = (k_issued > NS ? k_issued - NS : 0); j < k_issued; ++j)
                mbar_wait(bar(Lay::B_KF + j % NS), (j / NS) & 1, nullptr);
            for (int j = (v_issued > NS ? v_issued - NS : 0); j < v_issued; ++j)
                mbar_wait(bar(Lay::B_VF + j % NS), (j / NS) & 1, nullptr);
            if (!GATHER)
                for (int t = 0; t < 2; ++t) mbar_wait(bar(Lay::B_QF + t), 0, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
            auto qk = [&](int t, int s) {
                const uint32_t qa = sbase + Lay::OFF_Q + t * Lay::TILE_BYTES;
                const uint32_t kb = sbase + Lay::OFF_K + s * Lay::TILE_BYTES;
                const uint32_t dst = tmem + (t ? Lay::COL_S1 : Lay::COL_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * Lay::HALF_BYTES + (kk % 4) * 32;
                    umma_ss(dst, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                            IDESC_QK, kk > 0 ? 1u : 0u);
                }
            };
            auto pv = [&](int t, int s, bool acc) {
                const uint32_t vb = sbase + Lay::OFF_V + s * Lay::TILE_BYTES;
                const uint32_t dst = tmem + (t ? Lay::COL_O1 : Lay::COL_O0);
                const uint32_t pa = tmem + (t ? Lay::COL_S1 : Lay::COL_S0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts(dst, pa + kk * 8, sdesc_sw128(vb + kk * 2048, Lay::HALF_BYTES, 1024),
                            IDESC_PV, (acc || kk > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(bar(Lay::B_QF + 0), 0, abort_flag) &&
                      mbar_wait(bar(Lay::B_QF + 1), 0, abort_flag) &&
                      mbar_wait(bar(Lay::B_KF + 0), 0, abort_flag);
            if (ok && n_kv > 0) {
                tc_fence_after();
                qk(0, 0);
                umma_commit(bar(Lay::B_SF + 0));
                qk(1, 0);
                umma_commit(bar(Lay::B_SF + 1));
                umma_commit(bar(Lay::B_KE + 0));
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int s = j % NS;
                const uint32_t ph = (j / NS) & 1;
                const bool more = j + 1 < n_kv;
                const int s1 = (j + 1) % NS;
                const uint32_t ph1 = ((j + 1) / NS) & 1;
                ok = mbar_wait(bar(Lay::B_VF + s), ph, abort_flag) &&
                     mbar_wait(bar(Lay::B_PF + 0), j & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                pv(0, s, j > 0);
                if (more) {
                    if (!(ok = mbar_wait(bar(Lay::B_KF + s1), ph1, abort_flag))) break;
                    tc_fence_after();
                    qk(0, s1);
                    umma_commit(bar(Lay::B_SF + 0));
                }
                if (!(ok = mbar_wait(bar(Lay::B_PF + 1), j & 1, abort_flag))) break;
                tc_fence_after();
                pv(1, s, j > 0);
                umma_commit(bar(Lay::B_VE + s));
                if (more) {
                    qk(1, s1);
                    umma_commit(bar(Lay::B_SF + 1));
                    umma_commit(bar(Lay::B_KE + s1));
                }
            }
            if (!ok) record_fault(abort_flag, args.status, VAR_ERR_TIMEOUT);
            else umma_commit(bar(Lay::B_OF));
            // No UMMA may still be running when tensor memory is released.
            umma_commit(bar(Lay::B_DR));
            mbar_wait(bar(Lay::B_DR), 0, nullptr);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax groups
        const int g = (warp - 4) >> 2;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + (g ? Lay::COL_S1 : Lay::COL_S0);
        const uint32_t tO = tmem + lane_base + (g ? Lay::COL_O1 : Lay::COL_O0);
        const int qrow = row0 + g * 128 + r;
        const int b = bh / args.heads;

        if (GATHER) {
            // This thread's query row, gathered by index, into the swizzled tile.
            uint8_t* qs = smem + Lay::OFF_Q + g * Lay::TILE_BYTES;
            uint4 chunk[D / 8];
            if (qrow < args.n_rows) {
                int tok = __ldg(args.idx + static_cast<size_t>(b) * args.n_rows + qrow);
                tok = min(max(tok, 0), args.n_q - 1);
                const uint4* src = reinterpret_cast<const uint4*>(
                    args.q + (static_cast<size_t>(bh) * args.n_q + tok) * D);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) chunk[c] = __ldg(src + c);
            } else {
#pragma unroll
                for (int c = 0; c < D / 8; ++c) chunk[c] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const int hh = c >> 3, cc = c & 7;
                *reinterpret_cast<uint4*>(qs + hh * Lay::HALF_BYTES + r * 128 + ((cc ^ (r & 7)) << 4)) =
                    chunk[c];
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(Lay::B_QF + g));
        }

        const float sl2 = args.scale_log2;
        float m_run = -INFINITY;
        float l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            if (!mbar_wait(bar(Lay::B_SF + g), j & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
            tmem_wait_ld();
            const int valid = args.L - j * 128;
            if (valid < 128) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= valid) s[c >> 5][c & 31] = __float_as_uint(-INFINITY);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c >> 5][c & 31]));
            const float m_tile = mx * sl2;
            const bool need = m_tile > m_run + 8.0f;
            const float m_new = need ? m_tile : m_run;
            const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
            l_run *= alpha;
            m_run = m_new;
            // P = exp2(S * scale*log2e - m), packed to bf16 pairs, 16 columns at a time
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(s[cc][2 * c]), sl2, neg_m));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(s[cc][2 * c + 1]), sl2, neg_m));
                    sum0 += p0;
                    sum1 += p1;
                    pk[c] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tS + cc * 16, pk);
            }
            l_run += sum0 + sum1;
            // O_t *= alpha where the running maximum moved (the previous PV has
            // completed: its commit preceded this tile's S commit)
            if (__any_sync(0xffffffffu, need && j > 0)) {
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tmem_st32(tO + c0, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(Lay::B_PF + g));
        }
        if (ok) ok = mbar_wait(bar(Lay::B_OF), 0, abort_flag);
        if (!ok) {
            record_fault(abort_flag, args.status, VAR_ERR_TIMEOUT);
        } else {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
            __nv_bfloat16* dst = args.o + (static_cast<size_t>(bh) * args.n_rows + qrow) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
                tmem_wait_ld();
                if (qrow < args.n_rows) {
                    uint32_t w[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                    for (int c = 0; c < 4; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------- host

template <int D, bool GATHER>
static int launch_attn(const StepGeom& g, const void* q, const void* k, const void* v,
                       const int32_t* idx, int n_rows, void* o, cudaStream_t st)
{
    using Lay = AttnLayout<D>;
    static bool attr_done = false;   // per process; the attribute is per function
    auto kern = attn_fwd_kernel<D, GATHER>;
    if (!attr_done) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM_BYTES) !=
            cudaSuccess)
            return VAR_ERR_CUDA;
        attr_done = true;
    }
    int32_t* status = device_status_ptr();
    if (!status) return VAR_ERR_CUDA;
    if (n_rows == 0) return VAR_OK;

    CUtensorMap tq, tk, tv;
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
    AttnArgs a;
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
    kern<<<grid, 384, Lay::SMEM_BYTES, st>>>(tq, tk, tv, a);
    return cuda_status(cudaGetLastError());
}

int launch_attn_dense(const StepGeom& g, const void* q, const void* k, const void* v, void* o,
                      cudaStream_t st)
{
    if (g.D == 128) return launch_attn<128, false>(g, q, k, v, nullptr, g.N, o, st);
    if (g.D == 64) return launch_attn<64, false>(g, q, k, v, nullptr, g.N, o, st);
    return VAR_ERR_UNSUPPORTED;
}

int launch_attn_pruned(const StepGeom& g, const void* q, const void* k, const void* v,
                       const int32_t* idx, int keep_k, void* o, cudaStream_t st)
{
    if (g.D == 128) return launch_attn<128, true>(g, q, k, v, idx, keep_k, o, st);
    if (g.D == 64) return launch_attn<64, true>(g, q, k, v, idx, keep_k, o, st);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
