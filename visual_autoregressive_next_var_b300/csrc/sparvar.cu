// Dynamic sparse attention pattern ("SparVAR" abstract: the sparse attention
// pattern of later high-resolution scales is predicted from a sparse decision
// scale and carried to them by index mapping).
//
// Block scores of the decision step, A[qb][u]: the attention mass unit u (64
// keys) receives from each query of the 8x8 query block qb, averaged over the
// block's 64 queries, the heads and the batch.  The selection that follows (the
// units by decreasing score until a fraction tau of the mass is kept) is an
// integer result decided by floating point, so the scores are made exact
// enough to decide it as the fp64 definition does:
//
//   1. unit_mass_kernel    fp32 on the CUDA cores, one CTA per (qb, b, h), with
//                          a rigorous bound on every block score (below).
//   2. unit_certify_kernel per qb: the scores summed over (b, h), intervals
//                          [A - E, A + E], and a check that every unit's keep /
//                          drop decision at tau is the same for every value in
//                          the intervals; a block whose decision is not settled
//                          is flagged.
//   3. unit_rescore_rows_kernel, unit_rescore_reduce_kernel
//                          the flagged blocks are re-scored in fp64 in the
//                          definition's own evaluation order (dot products
//                          sequential over channels, the softmax denominator
//                          sequential over keys, the masses added key by key,
//                          the block sum in the order (b, h, y, x)), a few
//                          blocks per round.
// The selection and the index mapping run on the host (api.cu) on these
// scores: on a certified block the host's decision on the fp32-based values
// equals the fp64 one, on a re-scored block it uses the fp64 values.
//
// Bound of kernel 1, per query row (reference m = the row's largest computed
// score, so the largest term is exactly 1 and the row total l >= 1):
//   s_j = q . k_j: exact bf16 products, fp32 fused multiply-adds in chunks of
//       16 channels, each chunk added to a running total, so every product
//       meets at most 22 rounded additions: |s^ - s| <= g ||q|| ||k_j|| with
//       g = 26u/(1 - 26u), u = 2^-24 (margin included); ||q|| and the unit's
//       largest ||k_j|| are rounded up.
//   x_j = fl(fl(s^_j - m) c), c = fl(scale log2 e): relative error of x below
//       2^-20 (two roundings and c's own).
//   p_j = exp2f(x_j): at most 2 ulp (CUDA's documented bound).
//   A term's relative error is then at most 2^b - 1 <= 0.694 b (b < 2^-8) with
//   b = g ||q|| ||k_j|| c + 2^-20 |x_j|, plus 2^-22 for exp2f.  Over a unit the
//   p-weighted mean of |x_j| is at most log2(n_u / S_u) (Jensen: p log(1/p) is
//   concave), n_u <= 64 keys, S_u the unit's sum, which adds at most 6
//   roundings: r_u = 0.694 (g ||q|| max||k|| c + 2^-20 (log2(64/S_u) + 1))
//   + 2^-20 + 8u.  mass_u = S_u / l, l = sum_u S_u in fp64: relative error at
//   most r_u + r_l, r_l the S-weighted mean of the r_u plus U 2^-52.
//   Subnormal exp2f results add at most 2^-140 absolute per unit.
// The block score's absolute error bound E is the sum over its rows of
// mass_u (r_u + r_l + 2^-50) + 2^-140, divided like the score, plus
// (L + 4096) 2^-51 of the score for the fp64 roundings of the sums and of the
// definition itself.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace varattn {

namespace {

constexpr int kSvRows = 64;          // queries of an 8x8 block
constexpr int kSvThreads = 128;      // a thread: 8 rows x 4 keys of a 64 x 64 tile
constexpr int kSvMaxU = 512;         // units the mass kernel keeps in shared memory
constexpr int kRescoreBlocks = 4;    // flagged blocks re-scored per round
constexpr int kRescoreWarps = 4;

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct SvWs {
    size_t part, perr, flags, rows, total;
};

__host__ __device__ inline SvWs sv_ws_layout(int BH, int n_qb, int U)
{
    SvWs w{};
    size_t o = 0;
    w.part = o;  o = align256(o + sizeof(double) * BH * n_qb * U);
    w.perr = o;  o = align256(o + sizeof(double) * BH * n_qb * U);
    w.flags = o; o = align256(o + sizeof(int) * n_qb);
    w.rows = o;  o = align256(o + sizeof(double) * kRescoreBlocks * BH * 64 * U);
    w.total = o;
    return w;
}

// Shared memory of the mass kernel: Qt [D][64] fp32, Kt [D][64] bf16 bits,
// Su [64][U] fp32, kmax [U], nq [64], keys [64] int, then (8-byte aligned)
// lrow [64] and rlrow [64] fp64.
__host__ __device__ inline size_t sv_off_rows(int D, int U)
{
    const size_t o = static_cast<size_t>(D) * 64 * 6 + 4 * (static_cast<size_t>(kSvRows) * U + U + 2 * kSvRows);
    return (o + 7) & ~static_cast<size_t>(7);
}

// Key of slot t in [0, 64) of unit u (flat cache index), or -1 (no key there).
__device__ __forceinline__ int unit_key(const UnitMap& m, int u, int t)
{
    if (u < m.n_sink) {
        const int j = 64 * u + t;
        return j < m.sink_len ? j : -1;
    }
    int sc = 0;
    while (sc + 1 < m.n_sc && u >= m.ubase[sc + 1]) ++sc;
    const int s = m.side[sc], nbs = (s + 7) >> 3;
    const int loc = u - m.ubase[sc];
    const int r = 8 * (loc / nbs) + (t >> 3), c = 8 * (loc % nbs) + (t & 7);
    return (r < s && c < s) ? m.off[sc] + r * s + c : -1;
}

__device__ __forceinline__ int unit_of(const UnitMap& m, int j)
{
    if (j < m.sink_len) return j >> 6;
    int t = 0;
    while (t + 1 < m.n_sc && j >= m.off[t + 1]) ++t;
    const int s = m.side[t];
    const int local = j - m.off[t];
    const int r = local / s, c = local - r * s;
    return m.ubase[t] + (r >> 3) * ((s + 7) >> 3) + (c >> 3);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The relative bound r_u of a unit sum S (see the file header).
__device__ __forceinline__ float unit_bound(float gq_c, float kmax_u, float s)
{
    if (!(s > 0.f)) return 0.f;
    const float b = __fadd_ru(__fmul_ru(gq_c, kmax_u), __fmul_ru(0x1p-20f, __log2f(64.f / s) + 1.f));
    return b < 0x1p-8f ? __fadd_ru(__fmul_ru(0.694f, b), 0x1p-20f + 8.f * 0x1p-24f) : 1e30f;
}

// ------------------------------------------------------------------ 1. masses

template <int D>
__global__ void __launch_bounds__(kSvThreads)
    unit_mass_kernel(const UnitMap m, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                     int side, int cap, float c_log2, double* __restrict__ part, double* __restrict__ perr)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int U = m.U;
    float* Qt = reinterpret_cast<float*>(smem);                           // [D][64]
    uint16_t* Kt = reinterpret_cast<uint16_t*>(smem + D * 64 * 4);        // [D][64] bf16 bits
    float* Su = reinterpret_cast<float*>(smem + D * 64 * 6);              // [64][U]
    float* kmax = Su + kSvRows * U;                                       // [U]
    float* nq = kmax + U;                                                 // [64]
    int* keys = reinterpret_cast<int*>(nq + kSvRows);                     // [64]
    double* lrow = reinterpret_cast<double*>(smem + sv_off_rows(D, U));   // [64]
    double* rlrow = lrow + kSvRows;                                       // [64]

    const int nb = side >> 3;
    const int qb = blockIdx.x, bh = blockIdx.y;
    const int by = qb / nb, bx = qb - by * nb;
    const int tid = threadIdx.x, lane = tid & 31;
    const int kg = tid & 15, rg = tid >> 4;          // keys 4kg..4kg+3; rows 8rg..8rg+7 (query block row rg)
    const int N = side * side;
    const __nv_bfloat16* kb = k + static_cast<size_t>(bh) * cap * D;

    // the block's 64 queries (row 8y + x), transposed to fp32, and their norms (rounded up)
    for (int e = tid; e < kSvRows * D / 8; e += kSvThreads) {
        const int row = e / (D / 8), c0 = (e % (D / 8)) * 8;
        const int i = (by * 8 + (row >> 3)) * side + bx * 8 + (row & 7);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(q + (static_cast<size_t>(bh) * N + i) * D + c0));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            Qt[(c0 + 2 * h) * kSvRows + row] = bf_lo(w[h]);
            Qt[(c0 + 2 * h + 1) * kSvRows + row] = bf_hi(w[h]);
        }
    }
    __syncthreads();
    if (tid < kSvRows) {
        float ss = 0.f;
        for (int c = 0; c < D; ++c) ss = __fmaf_ru(Qt[c * kSvRows + tid], Qt[c * kSvRows + tid], ss);
        nq[tid] = __fsqrt_ru(ss);
    }

    float mrow[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) mrow[r] = -INFINITY;

    for (int pass = 0; pass < 2; ++pass) {
        for (int u = 0; u < U; ++u) {
            __syncthreads();                                   // the previous unit's tile is consumed
            if (tid < 64) keys[tid] = unit_key(m, u, tid);
            __syncthreads();
            // the unit's keys, transposed (bf16 bits; a missing key reads as zeros)
            for (int e = tid; e < 64 * D / 8; e += kSvThreads) {
                const int t = e / (D / 8), c0 = (e % (D / 8)) * 8;
                const int j = keys[t];
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (j >= 0) v = __ldg(reinterpret_cast<const uint4*>(kb + static_cast<size_t>(j) * D + c0));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    Kt[(c0 + 2 * h) * 64 + t] = static_cast<uint16_t>(w[h] & 0xFFFFu);
                    Kt[(c0 + 2 * h + 1) * 64 + t] = static_cast<uint16_t>(w[h] >> 16);
                }
            }
            __syncthreads();
            if (pass == 0 && tid < 32) {
                // largest key norm of the unit (rounded up): lane t takes slots t and t + 32
                float mx = 0.f;
                for (int t = lane; t < 64; t += 32) {
                    float ss = 0.f;
                    for (int c = 0; c < D; ++c) {
                        const float kv = __uint_as_float(static_cast<uint32_t>(Kt[c * 64 + t]) << 16);
                        ss = __fmaf_ru(kv, kv, ss);
                    }
                    mx = fmaxf(mx, __fsqrt_ru(ss));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                if (lane == 0) kmax[u] = mx;
            }
            // scores of rows 8rg..8rg+7 x keys (4kg, 4kg+1), (4kg+2, 4kg+3): chunks of
            // 16 channels, each added to the running total
            uint64_t tot[8][2];
#pragma unroll
            for (int r = 0; r < 8; ++r) tot[r][0] = tot[r][1] = 0ull;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 16) {
                uint64_t ch[8][2];
#pragma unroll
                for (int r = 0; r < 8; ++r) ch[r][0] = ch[r][1] = 0ull;
#pragma unroll 4
                for (int c = c0; c < c0 + 16; ++c) {
                    const float4 qa = *reinterpret_cast<const float4*>(Qt + c * kSvRows + 8 * rg);
                    const float4 qc = *reinterpret_cast<const float4*>(Qt + c * kSvRows + 8 * rg + 4);
                    const uint2 kw = *reinterpret_cast<const uint2*>(Kt + c * 64 + 4 * kg);
                    const uint64_t k01 = f2_pack(bf_lo(kw.x), bf_hi(kw.x));
                    const uint64_t k23 = f2_pack(bf_lo(kw.y), bf_hi(kw.y));
                    const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qc.x, qc.y, qc.z, qc.w};
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const uint64_t qq = f2_pack(qv[r], qv[r]);
                        ch[r][0] = f2_fma(qq, k01, ch[r][0]);
                        ch[r][1] = f2_fma(qq, k23, ch[r][1]);
                    }
                }
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    tot[r][0] = f2_add(tot[r][0], ch[r][0]);
                    tot[r][1] = f2_add(tot[r][1], ch[r][1]);
                }
            }
            const bool v0 = keys[4 * kg] >= 0, v1 = keys[4 * kg + 1] >= 0;
            const bool v2 = keys[4 * kg + 2] >= 0, v3 = keys[4 * kg + 3] >= 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float s0, s1, s2, s3;
                f2_unpack(tot[r][0], s0, s1);
                f2_unpack(tot[r][1], s2, s3);
                if (!v0) s0 = -INFINITY;
                if (!v1) s1 = -INFINITY;
                if (!v2) s2 = -INFINITY;
                if (!v3) s3 = -INFINITY;
                if (pass == 0) {
                    float mx = fmaxf(fmaxf(s0, s1), fmaxf(s2, s3));
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    mrow[r] = fmaxf(mrow[r], mx);
                } else {
                    const float mr = mrow[r];
                    const float p0 = exp2f(__fmul_rn(__fsub_rn(s0, mr), c_log2));
                    const float p1 = exp2f(__fmul_rn(__fsub_rn(s1, mr), c_log2));
                    const float p2 = exp2f(__fmul_rn(__fsub_rn(s2, mr), c_log2));
                    const float p3 = exp2f(__fmul_rn(__fsub_rn(s3, mr), c_log2));
                    float sm = __fadd_rn(__fadd_rn(p0, p1), __fadd_rn(p2, p3));
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) sm = __fadd_rn(sm, __shfl_xor_sync(0xffffffffu, sm, off));
                    if (kg == 0) Su[(8 * rg + r) * U + u] = sm;
                }
            }
        }
    }
    __syncthreads();
    // per row: the total l (fp64) and the S-weighted mean of the unit bounds
    constexpr float kG = 26.f * 0x1p-24f / (1.f - 26.f * 0x1p-24f);
    const float c_up = __fmul_ru(c_log2, 1.0f + 0x1p-20f);
    if (tid < kSvRows) {
        double l = 0.0, wr = 0.0;
        for (int u = 0; u < U; ++u) l += static_cast<double>(Su[tid * U + u]);
        const float gq = __fmul_ru(__fmul_ru(kG, nq[tid]), c_up);
        for (int u = 0; u < U; ++u) {
            const float s = Su[tid * U + u];
            wr += static_cast<double>(s) * static_cast<double>(unit_bound(gq, kmax[u], s));
        }
        lrow[tid] = l;
        rlrow[tid] = wr / l + static_cast<double>(U) * 0x1p-52;
    }
    __syncthreads();
    // per unit: the block's sum over its 64 rows in (y, x) order, and the bound
    for (int u = tid; u < U; u += kSvThreads) {
        double acc = 0.0, err = 0.0;
        for (int row = 0; row < kSvRows; ++row) {
            const float s = Su[row * U + u];
            const double ms = static_cast<double>(s) / lrow[row];
            const float gq = __fmul_ru(__fmul_ru(kG, nq[row]), c_up);
            acc += ms;
            err += ms * (static_cast<double>(unit_bound(gq, kmax[u], s)) + rlrow[row] + 0x1p-50) + 0x1p-140;
        }
        const size_t o = (static_cast<size_t>(bh) * gridDim.x + qb) * U + u;
        part[o] = acc;
        perr[o] = err * (1.0 + 0x1p-40);
    }
}

// ------------------------------------------------------------------ 2. certify

// Per block: scores (sum over (b, h) / (B H 64)), intervals, and whether the
// selection at tau is settled for every value in them.  force: flag every block.
__global__ void __launch_bounds__(256)
    unit_certify_kernel(const double* __restrict__ part, const double* __restrict__ perr, int BH, int U, int n_sink,
                        int L, double tau, int force, double* __restrict__ scores, int* __restrict__ flags,
                        int32_t* __restrict__ rescored)
{
    extern __shared__ double sh[];            // lo[U], hi[U]
    __shared__ double red[2][8];
    __shared__ int bad;
    double* lo = sh;
    double* hi = sh + U;
    const int qb = blockIdx.x, n_qb = gridDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const double inv = 1.0 / (static_cast<double>(BH) * 64.0);
    const double slack = (static_cast<double>(L) + 4096.0) * 0x1p-51;   // fp64 roundings, both sides
    if (tid == 0) bad = force;
    double slo = 0.0, shi = 0.0;
    for (int u = tid; u < U; u += blockDim.x) {
        double a = 0.0, e = 0.0;
        for (int b = 0; b < BH; ++b) {
            const size_t o = (static_cast<size_t>(b) * n_qb + qb) * U + u;
            a += part[o];
            e += perr[o];
        }
        const double A = a * inv;
        const double E = e * inv * (1.0 + 0x1p-40) + A * slack + 1e-300;
        scores[static_cast<size_t>(qb) * U + u] = A;
        lo[u] = fmax(A - E, 0.0);
        hi[u] = A + E;
        slo += lo[u];
        shi += hi[u];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        slo += __shfl_xor_sync(0xffffffffu, slo, off);
        shi += __shfl_xor_sync(0xffffffffu, shi, off);
    }
    if (lane == 0) {
        red[0][warp] = slo;
        red[1][warp] = shi;
    }
    __syncthreads();
    double tot_lo = 0.0, tot_hi = 0.0, sink_lo = 0.0, sink_hi = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        tot_lo += red[0][w];
        tot_hi += red[1][w];
    }
    for (int u = 0; u < n_sink; ++u) {
        sink_lo += lo[u];
        sink_hi += hi[u];
    }
    const double t_lo = tau * tot_lo * (1.0 - slack), t_hi = tau * tot_hi * (1.0 + slack);
    for (int u = n_sink + tid; u < U; u += blockDim.x) {
        // the mass the definition has added before it considers u: the sinks and
        // the units ranked before u (larger score, or equal score and lower index)
        double h_lo = sink_lo, h_hi = sink_hi;
        for (int v = n_sink; v < U; ++v) {
            if (v == u) continue;
            if (lo[v] > hi[u] || (v < u && lo[v] >= hi[u])) h_lo += lo[v];   // surely before u
            if (hi[v] > lo[u] || (v < u && hi[v] >= lo[u])) h_hi += hi[v];   // possibly before u
        }
        h_lo *= 1.0 - slack;
        h_hi *= 1.0 + slack;
        const bool keep = h_hi < t_lo, drop = h_lo >= t_hi;
        if (!keep && !drop) bad = 1;
    }
    __syncthreads();
    if (tid == 0) {
        flags[qb] = bad;
        if (rescored) rescored[qb] = 0;
    }
}

// ------------------------------------------------------------------ 3. fp64 re-score

// The rank-th flagged block, or -1.
__device__ __forceinline__ int flagged_block(const int* flags, int n_qb, int rank)
{
    int seen = 0;
    for (int qb = 0; qb < n_qb; ++qb) {
        if (flags[qb]) {
            if (seen == rank) return qb;
            ++seen;
        }
    }
    return -1;
}

// One warp per query row of a flagged block, in the definition's order: s_j =
// (sum_c q_c k_jc sequential) * scale, mx = max_j s_j, l = sum_j exp(s_j - mx)
// sequential over j, mass[unit(j)] += exp(s_j - mx) / l sequential over j.
template <int D>
__global__ void __launch_bounds__(kRescoreWarps * 32)
    unit_rescore_rows_kernel(const UnitMap m, const __nv_bfloat16* __restrict__ q,
                             const __nv_bfloat16* __restrict__ k, const int* __restrict__ flags, int n_qb, int round,
                             int side, int cap, int BH, double scale, double* __restrict__ rows)
{
    extern __shared__ double shr[];                   // per warp: q[D], mass[U]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_block = BH * 64;
    const int gr = blockIdx.x * kRescoreWarps + warp;  // row of the round
    const int slot = gr / per_block;
    if (slot >= kRescoreBlocks) return;
    const int qb = flagged_block(flags, n_qb, round * kRescoreBlocks + slot);
    if (qb < 0) return;
    const int idx = gr - slot * per_block;             // (b, h, y, x), x fastest
    const int bhh = idx >> 6, y = (idx >> 3) & 7, x = idx & 7;
    const int nb = side >> 3, by = qb / nb, bx = qb - by * nb;
    const int i = (by * 8 + y) * side + bx * 8 + x;
    const int N = side * side;
    double* qd = shr + warp * (D + m.U);
    double* mass = qd + D;
    const __nv_bfloat16* qrow = q + (static_cast<size_t>(bhh) * N + i) * D;
    for (int c = lane; c < D; c += 32) qd[c] = static_cast<double>(__bfloat162float(qrow[c]));
    for (int u = lane; u < m.U; u += 32) mass[u] = 0.0;
    __syncwarp();
    const __nv_bfloat16* kb = k + static_cast<size_t>(bhh) * cap * D;
    // bf16 x bf16 products are exact in fp64, so a fused multiply-add rounds
    // exactly as the separate multiply and add of the definition
    auto score = [&](int j) -> double {
        const uint4* kr = reinterpret_cast<const uint4*>(kb + static_cast<size_t>(j) * D);
        double dot = 0.0;
        for (int c0 = 0; c0 < D / 8; ++c0) {
            const uint4 v = __ldg(kr + c0);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                dot = __fma_rn(qd[8 * c0 + 2 * h], static_cast<double>(bf_lo(w[h])), dot);
                dot = __fma_rn(qd[8 * c0 + 2 * h + 1], static_cast<double>(bf_hi(w[h])), dot);
            }
        }
        return __dmul_rn(dot, scale);
    };
    double mx = -INFINITY;
    for (int j = lane; j < m.L; j += 32) mx = fmax(mx, score(j));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    double l = 0.0;
    for (int j0 = 0; j0 < m.L; j0 += 32) {
        const int j = j0 + lane;
        const double e = j < m.L ? exp(__dsub_rn(score(j), mx)) : 0.0;
        const int n = min(32, m.L - j0);
        for (int t = 0; t < n; ++t) l = __dadd_rn(l, __shfl_sync(0xffffffffu, e, t));
    }
    for (int j0 = 0; j0 < m.L; j0 += 32) {
        const int j = j0 + lane;
        double term = 0.0;
        int uj = 0;
        if (j < m.L) {
            term = __ddiv_rn(exp(__dsub_rn(score(j), mx)), l);
            uj = unit_of(m, j);
        }
        const int n = min(32, m.L - j0);
        for (int t = 0; t < n; ++t) {
            const double tv = __shfl_sync(0xffffffffu, term, t);
            const int ut = __shfl_sync(0xffffffffu, uj, t);
            if (lane == 0) mass[ut] = __dadd_rn(mass[ut], tv);
        }
    }
    __syncwarp();
    double* out = rows + (static_cast<size_t>(slot) * per_block + idx) * m.U;
    for (int u = lane; u < m.U; u += 32) out[u] = mass[u];
}

// The re-scored blocks' scores: the rows' masses added in (b, h, y, x) order.
__global__ void __launch_bounds__(128)
    unit_rescore_reduce_kernel(const double* __restrict__ rows, const int* __restrict__ flags, int n_qb, int round,
                               int BH, int U, double* __restrict__ scores, int32_t* __restrict__ rescored)
{
    const int slot = blockIdx.y;
    const int qb = flagged_block(flags, n_qb, round * kRescoreBlocks + slot);
    if (qb < 0) return;
    const int per_block = BH * 64;
    for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < U; u += gridDim.x * blockDim.x) {
        double acc = 0.0;
        for (int r = 0; r < per_block; ++r)
            acc = __dadd_rn(acc, rows[(static_cast<size_t>(slot) * per_block + r) * U + u]);
        scores[static_cast<size_t>(qb) * U + u] = __ddiv_rn(acc, static_cast<double>(per_block));
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && rescored) rescored[qb] = 1;
}

template <int D>
int launch_sparvar_d(const StepGeom& g, const UnitMap& m, const void* q, const void* k, double tau, int force,
                     double scale64, void* ws, double* scores, int32_t* rescored, cudaStream_t st)
{
    const int BH = g.B * g.H;
    const int nb = g.side / 8, n_qb = nb * nb;
    const SvWs w = sv_ws_layout(BH, n_qb, m.U);
    auto* base = static_cast<uint8_t*>(ws);
    auto* part = reinterpret_cast<double*>(base + w.part);
    auto* perr = reinterpret_cast<double*>(base + w.perr);
    auto* flags = reinterpret_cast<int*>(base + w.flags);
    auto* rows = reinterpret_cast<double*>(base + w.rows);
    const auto* qp = static_cast<const __nv_bfloat16*>(q);
    const auto* kp = static_cast<const __nv_bfloat16*>(k);
    const size_t smem = sv_off_rows(D, m.U) + 2 * sizeof(double) * kSvRows;
    if (ensure_smem_attr(unit_mass_kernel<D>, static_cast<int>(smem)) != cudaSuccess) return VAR_ERR_CUDA;
    const float c_log2 = g.scale * 1.4426950408889634f;
    if (launch_kernel(unit_mass_kernel<D>, dim3(n_qb, BH), dim3(kSvThreads), smem, st, false, m, qp, kp, g.side,
                      g.cap, c_log2, part, perr) != cudaSuccess)
        return VAR_ERR_CUDA;
    const size_t csm = 2 * sizeof(double) * m.U;
    if (ensure_smem_attr(unit_certify_kernel, static_cast<int>(csm)) != cudaSuccess) return VAR_ERR_CUDA;
    if (launch_kernel(unit_certify_kernel, dim3(n_qb), dim3(256), csm, st, false, static_cast<const double*>(part),
                      static_cast<const double*>(perr), BH, m.U, m.n_sink, m.L, tau, force, scores, flags,
                      rescored) != cudaSuccess)
        return VAR_ERR_CUDA;
    const size_t rsm = sizeof(double) * kRescoreWarps * (D + m.U);
    if (ensure_smem_attr(unit_rescore_rows_kernel<D>, static_cast<int>(rsm)) != cudaSuccess) return VAR_ERR_CUDA;
    const int rows_per_round = kRescoreBlocks * BH * 64;
    for (int round = 0; round * kRescoreBlocks < n_qb; ++round) {
        if (launch_kernel(unit_rescore_rows_kernel<D>, dim3((rows_per_round + kRescoreWarps - 1) / kRescoreWarps),
                          dim3(kRescoreWarps * 32), rsm, st, false, m, qp, kp, static_cast<const int*>(flags), n_qb,
                          round, g.side, g.cap, BH, scale64, rows) != cudaSuccess)
            return VAR_ERR_CUDA;
        if (launch_kernel(unit_rescore_reduce_kernel, dim3((m.U + 127) / 128, kRescoreBlocks), dim3(128), 0, st,
                          false, static_cast<const double*>(rows), static_cast<const int*>(flags), n_qb, round, BH,
                          m.U, scores, rescored) != cudaSuccess)
            return VAR_ERR_CUDA;
    }
    return VAR_OK;
}


// ------------------------------------------------------------------ fast path (tensor cores)

// Block scores in fp32 from the decision step's row log2-sum-exp (written by
// its dense attention): per (b, h) and 128 keys, S^T = K Q^T on the tensor
// cores, p = 2^(s scale log2 e - lse_i), and the thread owning a key row adds
// each group of 8 consecutive queries (one row of one 8x8 query block) into
// that block's column of a shared-memory table.  A second kernel sums, per
// (block, unit), the unit's keys over (b, h) in a fixed order (fp64), so the
// result is deterministic.  No error bound: the selection on these scores can
// differ from the fp64 definition's where two candidates are within the fp32
// rounding of the cut.
constexpr int kFastMaxQb = 64;       // query blocks of the decision step (side <= 64)

template <int D>
struct FastLayout {
    static constexpr int HALVES = D / 64;
    static constexpr int HALF_BYTES = 128 * 128;
    static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
    static constexpr int NSQ = 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_Q = OFF_K + TILE_BYTES;
    static constexpr int OFF_LSE = OFF_Q + NSQ * TILE_BYTES;   // [4 warps][128] float
    static constexpr int OFF_BAR = OFF_LSE + 4 * 128 * 4;
    static constexpr int B_KF = 0;
    static constexpr int B_QF = 1;                             // [NSQ]
    static constexpr int B_QE = B_QF + NSQ;                    // [NSQ]
    static constexpr int B_SF = B_QE + NSQ;                    // [2]
    static constexpr int B_SE = B_SF + 2;                      // [2]
    static constexpr int B_DR = B_SE + 2;
    static constexpr int NBAR = B_DR + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_RED = OFF_MISC + 16;              // [n_qb][128] float
    static constexpr uint32_t TMEM_COLS = 256;
    static size_t smem_bytes(int n_qb) { return OFF_RED + static_cast<size_t>(n_qb) * 128 * 4 + 1024; }
};

struct FastMaps {
    CUtensorMap q;    // 3-D (D, N', B*H), box (64, 128, 1)
    CUtensorMap k;    // 3-D (D, L', B*H), box (64, 128, 1)
};

struct FastArgs {
    int32_t n_q;            // N' (decision step queries)
    int32_t side;           // its grid side (a multiple of 8)
    int32_t n_qb;           // (side / 8)^2
    int32_t n_qt;           // ceil(N' / 128)
    int32_t L;              // keys of the decision step
    int32_t n_kt;           // ceil(L / 128)
    float scale_log2;
    const float* lse;       // [B*H][N']
    float* part;            // [B*H][n_qb][n_kt * 128]
    int32_t* status;
};

template <int D>
__global__ void __launch_bounds__(256, 2) unit_mass_fast_kernel(const __grid_constant__ FastMaps maps, const FastArgs a)
{
    using Lay = FastLayout<D>;
    constexpr int NSQ = Lay::NSQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + Lay::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::OFF_MISC + 4);
    float* red = reinterpret_cast<float*>(smem + Lay::OFF_RED);

    const int bh = blockIdx.x / a.n_kt;
    const int kt = blockIdx.x - bh * a.n_kt;
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
                tma_load_3d(sbase + Lay::OFF_K + hh * Lay::HALF_BYTES, &maps.k, hh * 64, kt * 128, bh, bar(Lay::B_KF));
            int issued = 0;
            for (int t = 0; t < n_qt; ++t) {
                const int s = t % NSQ;
                if (!mbar_wait(bar(Lay::B_QE + s), ((t / NSQ) & 1) ^ 1, abort_flag)) {
                    *abort_flag = 1;
                    atomicCAS(a.status, 0, VAR_ERR_TIMEOUT);
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
                const uint32_t qa = sbase + Lay::OFF_Q + s * Lay::TILE_BYTES;
                const uint32_t dst = tmem + static_cast<uint32_t>(buf * 128);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * Lay::HALF_BYTES + (kk % 4) * 32;
                    umma_ss(dst, sdesc_sw128(ka + off, 16, 1024), sdesc_sw128(qa + off, 16, 1024), IDESC,
                            kk > 0 ? 1u : 0u);
                }
                umma_commit(bar(Lay::B_SF + buf));
                umma_commit(bar(Lay::B_QE + s));
            }
            if (!ok) {
                *abort_flag = 1;
                atomicCAS(a.status, 0, VAR_ERR_TIMEOUT);
            }
            umma_commit(bar(Lay::B_DR));
            mbar_wait(bar(Lay::B_DR), 0, nullptr);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ consumers: one key row each
        const int r = (warp & 3) * 32 + lane;
        float* lw = reinterpret_cast<float*>(smem + Lay::OFF_LSE) + (warp & 3) * 128;
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const float sl2 = a.scale_log2;
        const float* lse_bh = a.lse + static_cast<size_t>(bh) * a.n_q;
        const int nb = a.side >> 3;
        for (int qb = 0; qb < a.n_qb; ++qb) red[qb * 128 + r] = 0.f;
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
                lw[lane * 4 + e] = qi < a.n_q ? __ldg(lse_bh + qi) : INFINITY;
            }
            __syncwarp();
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t sv[32];
                tmem_ld32(tmem + lane_base + static_cast<uint32_t>(buf * 128 + c0), sv);
                tmem_wait_ld();
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    // queries q0 + c0 + 8 g8 .. + 7: one row of one 8x8 query block
                    float sum = 0.f;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int col = 8 * g8 + c;
                        sum += ex2_approx(fmaf(__uint_as_float(sv[col]), sl2, -lw[c0 + col]));
                    }
                    const int i0 = q0 + c0 + 8 * g8;
                    if (i0 < a.n_q) {
                        const int y = i0 / a.side, x = i0 - y * a.side;
                        red[((y >> 3) * nb + (x >> 3)) * 128 + r] += sum;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(Lay::B_SE + buf));
        }
        if (!ok) {
            *abort_flag = 1;
            atomicCAS(a.status, 0, VAR_ERR_TIMEOUT);
        } else {
            const int j = kt * 128 + r;
            const size_t lpad = static_cast<size_t>(a.n_kt) * 128;
            if (j < a.L)
                for (int qb = 0; qb < a.n_qb; ++qb)
                    a.part[(static_cast<size_t>(bh) * a.n_qb + qb) * lpad + j] = red[qb * 128 + r];
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, Lay::TMEM_COLS);
    }
}

// scores[qb][u] = sum over (b, h) in order, then the unit's keys, of the block's
// masses, / (B H 64); one warp per (block, unit), fp64, fixed order
__global__ void __launch_bounds__(32)
    unit_mass_fast_reduce(const UnitMap m, const float* __restrict__ part, int BH, int n_qb, int n_kt,
                          double* __restrict__ scores)
{
    const int u = blockIdx.x, qb = blockIdx.y, lane = threadIdx.x;
    const int j0 = unit_key(m, u, lane), j1 = unit_key(m, u, lane + 32);
    const size_t lpad = static_cast<size_t>(n_kt) * 128;
    double acc = 0.0;
    for (int bh = 0; bh < BH; ++bh) {
        const float* pr = part + (static_cast<size_t>(bh) * n_qb + qb) * lpad;
        const double v0 = j0 >= 0 ? static_cast<double>(__ldg(pr + j0)) : 0.0;
        const double v1 = j1 >= 0 ? static_cast<double>(__ldg(pr + j1)) : 0.0;
        acc = __dadd_rn(acc, __dadd_rn(v0, v1));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc = __dadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    if (lane == 0) scores[static_cast<size_t>(qb) * m.U + u] = acc / (static_cast<double>(BH) * 64.0);
}

template <int D>
int launch_sparvar_fast_d(const StepGeom& g, const UnitMap& m, const void* q, const void* k, const float* lse,
                          void* ws, double* scores, cudaStream_t st, int32_t* status)
{
    using Lay = FastLayout<D>;
    const int BH = g.B * g.H;
    const int nb = g.side / 8, n_qb = nb * nb;
    const int n_kt = (g.L + 127) / 128;
    FastMaps maps;
    const uint32_t box[3] = {64, 128, 1};
    const uint64_t BHu = static_cast<uint64_t>(BH);
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(g.N), BHu};
        const uint64_t strides[2] = {D * 2ull, static_cast<uint64_t>(g.N) * D * 2ull};
        if (int rc = encode_tmap_bf16(&maps.q, q, 3, dims, strides, box)) return rc;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(g.L), BHu};
        const uint64_t strides[2] = {D * 2ull, static_cast<uint64_t>(g.cap) * D * 2ull};
        if (int rc = encode_tmap_bf16(&maps.k, k, 3, dims, strides, box)) return rc;
    }
    FastArgs a = {};
    a.n_q = g.N;
    a.side = g.side;
    a.n_qb = n_qb;
    a.n_qt = (g.N + 127) / 128;
    a.L = g.L;
    a.n_kt = n_kt;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.lse = lse;
    a.part = static_cast<float*>(ws);
    a.status = status;
    const size_t smem = Lay::smem_bytes(n_qb);
    auto kern = unit_mass_fast_kernel<D>;
    if (ensure_smem_attr(kern, static_cast<int>(smem)) != cudaSuccess) return VAR_ERR_CUDA;
    if (launch_kernel(kern, dim3(static_cast<unsigned>(BH * n_kt)), dim3(256), smem, st, false, maps, a) !=
        cudaSuccess)
        return VAR_ERR_CUDA;
    return cuda_status(launch_kernel(unit_mass_fast_reduce, dim3(m.U, n_qb), dim3(32), 0, st, false, m,
                                     static_cast<const float*>(ws), BH, n_qb, n_kt, scores));
}

size_t fast_part_bytes(const StepGeom& g)
{
    const int nb = g.side / 8;
    const size_t n_kt = static_cast<size_t>((g.L + 127) / 128);
    return static_cast<size_t>(g.B) * g.H * nb * nb * n_kt * 128 * sizeof(float);
}

}  // namespace

size_t sparvar_workspace_bytes(const StepGeom& g, int U)
{
    const int nb = g.side / 8;
    const size_t certified = sv_ws_layout(g.B * g.H, nb * nb, U).total;
    const size_t fast = fast_part_bytes(g);
    return certified > fast ? certified : fast;
}

int launch_sparvar_scores_fast(const StepGeom& g, const UnitMap& m, const void* q, const void* k, const float* lse,
                               void* ws, size_t ws_bytes, double* scores, cudaStream_t st, int32_t* status)
{
    if (ws_bytes < sparvar_workspace_bytes(g, m.U)) return VAR_ERR_WORKSPACE;
    const int nb = g.side / 8;
    if (nb * nb > kFastMaxQb) return VAR_ERR_UNSUPPORTED;
    if (g.D == 128) return launch_sparvar_fast_d<128>(g, m, q, k, lse, ws, scores, st, status);
    if (g.D == 64) return launch_sparvar_fast_d<64>(g, m, q, k, lse, ws, scores, st, status);
    return VAR_ERR_UNSUPPORTED;
}

int launch_sparvar_scores(const StepGeom& g, const UnitMap& m, const void* q, const void* k, double tau, int force,
                          double scale64, void* ws, size_t ws_bytes, double* scores, int32_t* rescored,
                          cudaStream_t st)
{
    if (ws_bytes < sparvar_workspace_bytes(g, m.U)) return VAR_ERR_WORKSPACE;
    if (m.U > kSvMaxU) return VAR_ERR_UNSUPPORTED;
    if (g.D == 128) return launch_sparvar_d<128>(g, m, q, k, tau, force, scale64, ws, scores, rescored, st);
    if (g.D == 64) return launch_sparvar_d<64>(g, m, q, k, tau, force, scale64, ws, scores, rescored, st);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
