// Pivot selection for cached token pruning on sm_103a.
//
// "FastVAR: Linear Visual Autoregressive Modeling via Cached Token Pruning"
// (abstract): only pivotal tokens are forwarded; "ARVAR" Key Design 2: Top-K
// indices gather them.  Score of token i of batch element b:
//     score[b,i] = || x[b,i,:] - mean_i x[b,i,:] ||_2^2
// The K largest are kept (equal scores: lower index first), returned ascending.
//
// The ranking is that of the fp64 evaluation (mean = fp64 channel sum / N,
// score = fp64 pairwise-halving tree over channels of rounded squared
// differences), reached with fp32 work on nearly every token.  Two kernels:
//
//   1. colsum (HBM pass over X).  Exact channel sums.  A cluster of 8 CTAs
//      owns a 128-channel chunk of one batch element, each CTA a slab of
//      rows.  Per element: x = hi + lo split exactly by two fp32 "magic"
//      additions (hi a multiple of 2^-13, |x| < 512; lo a multiple of 2^-36),
//      the float bit patterns summed as wrapping 32-bit integers, which is an
//      exact fixed-point sum.  A thread that meets |x| >= 512 redoes its rows
//      with 64-bit fixed point.  The cluster merges its CTAs' partial sums
//      through distributed shared memory; the exact sum is rounded once to
//      fp64, divided by N (the fp64 mean), and rounded to fp32 for the scores.
//      Launches the score kernel early (programmatic dependent launch).
//   2. score + select (L2 pass over X).  One warp per token: fp32 score with
//      a rigorous bound eps_i >= |fp32 score - fp64 score| (below), stored as
//      lo_i = score - eps (rounded down), hi_i = score + eps (rounded up).
//      The last CTA of a batch element to finish selects: T_lo = K-th largest
//      lo, T_hi = (K+1)-th largest hi (radix select); lo_i > T_hi => certainly
//      kept, hi_i < T_lo => certainly dropped; the band in between is either
//      decided by count (all kept or all dropped) or re-scored in fp64 in the
//      exact evaluation order, the remaining slots going to the best band
//      tokens by (score desc, index asc).  Output compaction keeps order.
//
// Error bound of kernel 2.  m' is the fp32 mean, mu the exact mean,
// E >= ||m' - mu||_2 = 2^-24 ||m'|| (1 + 2^-23) + 2^-120.  A lane sums its
// channels' terms fl(x - m')^2 with fused multiply-adds in 8 chains of at
// most h1 = ceil(C / 256) terms, adds the chains as a 3-level tree and the
// lanes as a 5-level butterfly: every term meets at most h = h1 + 8 rounded
// additions, so |s - S'| <= (h + 2) u S' (u = 2^-24, S' = sum (x - m')^2).
// |S' - S| <= 2 E sqrt(S') + 3 E^2 for S = sum (x - mu)^2, and the fp64
// evaluation differs from S by far less than 2^-44 (S + 2||m'|| sqrt(S) +
// ||m'||^2 + 1).  eps is the sum of the three, every operation rounded up.
#include <cfloat>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace varattn {

namespace {

constexpr int kSlabs = 8;                 // CTAs per cluster: row slabs of one chunk
constexpr int kChunk = 128;               // channels per chunk (256 bytes of a row)
constexpr int kSegs = kChunk / 8;         // 16-byte segments of a chunk row
constexpr int kSumThreads = 256;
constexpr int kRowGroups = kSumThreads / kSegs;   // rows in flight per CTA pass
constexpr int kSumUnroll = 8;

constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kTokPerWarp = 2;
constexpr int kScoreTok = kScoreWarps * kTokPerWarp;   // tokens per score CTA

constexpr int kScoreSmemMax = 220 * 1024;    // dynamic shared memory cap of the score kernel

constexpr float kMagA = 1536.0f;          // 1.5 * 2^10: ulp 2^-13 on [1024, 2048)
constexpr float kMagB = 0x1.8p-13f;       // 1.5 * 2^-13: ulp 2^-36 on [2^-13, 2^-12)
constexpr float kFastMax = 512.0f;        // |x| below this takes the two-window path

struct PivotWs {
    size_t mean64, mean32, lok, hik, band_idx, band_score, counters, total;
};

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ constexpr PivotWs pivot_ws_layout(int B, int N, int C)
{
    PivotWs w{};
    size_t o = 0;
    w.mean64 = o;     o = align256(o + sizeof(double) * B * C);
    w.mean32 = o;     o = align256(o + sizeof(float) * B * C);
    w.lok = o;        o = align256(o + sizeof(float) * B * N);
    w.hik = o;        o = align256(o + sizeof(float) * B * N);
    w.band_idx = o;   o = align256(o + sizeof(int) * B * N);
    w.band_score = o; o = align256(o + sizeof(double) * B * N);
    w.counters = o;   o = align256(o + sizeof(int) * B);
    w.total = o;
    return w;
}

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void ld_peer_pair(uint32_t local_addr, uint32_t rank, long long& a, long long& b)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.v2.s64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(ra) : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// ------------------------------------------------------------------ 1. colsum

// 64-bit fixed point: hi (LSB 2^-24) for |x| >= 2^-17, lo (LSB 2^-60) for
// 2^-53 <= |x| < 2^-17; smaller magnitudes contribute nothing.
__device__ __forceinline__ void accum_fixed(uint32_t h, long long& hi, long long& lo, bool& bad)
{
    const uint32_t e = (h >> 7) & 0xFFu;
    const long long m = static_cast<long long>((h & 0x7Fu) | 0x80u);
    if (e >= 110u) {
        if (e >= 147u) bad = true;             // |x| >= 2^20, inf or nan
        const long long v = m << min(e - 110u, 36u);
        hi += (h & 0x8000u) ? -v : v;
    } else if (e >= 74u) {
        const long long v = m << (e - 74u);
        lo += (h & 0x8000u) ? -v : v;
    }
}

// Correctly rounded (to nearest even) conversion of a 128-bit integer to fp64.
__device__ double i128_to_f64_rn(__int128 t)
{
    const bool neg = t < 0;
    unsigned __int128 u = neg ? static_cast<unsigned __int128>(-t) : static_cast<unsigned __int128>(t);
    if (u == 0) return 0.0;
    const uint64_t uh = static_cast<uint64_t>(u >> 64), ul = static_cast<uint64_t>(u);
    const int nbits = uh ? 128 - __clzll(static_cast<long long>(uh)) : 64 - __clzll(static_cast<long long>(ul));
    double r;
    if (nbits <= 53) {
        r = static_cast<double>(ul);
    } else {
        const int sh = nbits - 53;
        unsigned __int128 mant = u >> sh;
        const unsigned __int128 rem = u - (mant << sh);
        const unsigned __int128 half = static_cast<unsigned __int128>(1) << (sh - 1);
        if (rem > half || (rem == half && (mant & 1))) mant += 1;
        const double scale = __longlong_as_double(static_cast<long long>(1023 + sh) << 52);
        r = static_cast<double>(static_cast<uint64_t>(mant)) * scale;   // exact
    }
    return neg ? -r : r;
}

__global__ void __cluster_dims__(kSlabs, 1, 1) __launch_bounds__(kSumThreads)
    pivot_colsum_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, double* __restrict__ mean64,
                        float* __restrict__ mean32, int* __restrict__ counters, int32_t* status)
{
    __shared__ long long red_p[kRowGroups][kChunk];
    __shared__ long long red_q[kRowGroups][kChunk];
    __shared__ __align__(16) long long part[kChunk][2];   // this CTA's (p, q) per channel

    pdl_launch_dependents();
    const int rank = static_cast<int>(cluster_rank());    // == blockIdx.x (cluster spans x)
    const int chunk = blockIdx.y, b = blockIdx.z;
    const int rg = threadIdx.x / kSegs, seg = threadIdx.x % kSegs;
    const int c = chunk * kChunk + seg * 8;
    const int slab = (N + kSlabs - 1) / kSlabs;
    const int r0 = min(N, rank * slab), r1 = min(N, r0 + slab);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) counters[b] = 0;

    // exact sum of this thread's elements = p * 2^-24 + q * 2^-60
    long long p[8], q[8];
    bool bad = false;
    if (c < C) {
        const __nv_bfloat16* base = x + static_cast<size_t>(b) * N * C + c;
        uint32_t acc_a[8], acc_b[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc_a[e] = acc_b[e] = 0u;
        float mx = 0.f;
        const uint64_t mag_a = f2_pack(kMagA, kMagA), mag_b = f2_pack(kMagB, kMagB);
        auto accum = [&](const uint4& v) {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = __uint_as_float(w[e] << 16), x1 = __uint_as_float(w[e] & 0xFFFF0000u);
                const uint64_t x2 = f2_pack(x0, x1);
                const uint64_t s2 = f2_add(x2, mag_a);                 // RN(x + 1.5*2^10)
                const uint64_t l2 = f2_sub(x2, f2_sub(s2, mag_a));     // x - hi, exact
                const uint64_t t2 = f2_add(l2, mag_b);                 // RN(lo + 1.5*2^-13)
                float s0, s1, t0, t1;
                f2_unpack(s2, s0, s1);
                f2_unpack(t2, t0, t1);
                acc_a[2 * e] += __float_as_uint(s0);
                acc_a[2 * e + 1] += __float_as_uint(s1);
                acc_b[2 * e] += __float_as_uint(t0);
                acc_b[2 * e + 1] += __float_as_uint(t1);
                mx = fmax3(mx, fabsf(x0), fabsf(x1));
            }
        };
        int r = r0 + rg;
        for (; r + kRowGroups * (kSumUnroll - 1) < r1; r += kRowGroups * kSumUnroll) {
            uint4 v[kSumUnroll];
#pragma unroll
            for (int u = 0; u < kSumUnroll; ++u) v[u] = ld_stream16(base + static_cast<size_t>(r + kRowGroups * u) * C);
#pragma unroll
            for (int u = 0; u < kSumUnroll; ++u) accum(v[u]);
        }
        for (; r < r1; r += kRowGroups) accum(ld_stream16(base + static_cast<size_t>(r) * C));
        const int nr = r0 + rg < r1 ? (r1 - r0 - rg + kRowGroups - 1) / kRowGroups : 0;
        if (mx < kFastMax) {
            // every element added bits(M) + (its value in ulps of the window)
            const uint32_t bias_a = static_cast<uint32_t>(nr) * __float_as_uint(kMagA);
            const uint32_t bias_b = static_cast<uint32_t>(nr) * __float_as_uint(kMagB);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                p[e] = static_cast<long long>(static_cast<int32_t>(acc_a[e] - bias_a)) * (1ll << 11);
                q[e] = static_cast<long long>(static_cast<int32_t>(acc_b[e] - bias_b)) * (1ll << 24);
            }
        } else {
            // an element at or beyond the fast window: redo these rows in 64-bit fixed point
#pragma unroll
            for (int e = 0; e < 8; ++e) p[e] = q[e] = 0;
            for (int rr = r0 + rg; rr < r1; rr += kRowGroups) {
                const uint4 v = ld_stream16(base + static_cast<size_t>(rr) * C);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    accum_fixed(w[e] & 0xFFFFu, p[2 * e], q[2 * e], bad);
                    accum_fixed(w[e] >> 16, p[2 * e + 1], q[2 * e + 1], bad);
                }
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = q[e] = 0;
    }
    if (bad) atomicCAS(status, 0, VAR_ERR_NUMERIC);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        red_p[rg][seg * 8 + e] = p[e];
        red_q[rg][seg * 8 + e] = q[e];
    }
    __syncthreads();
    if (threadIdx.x < kChunk) {
        long long sp = 0, sq = 0;
#pragma unroll
        for (int g = 0; g < kRowGroups; ++g) {
            sp += red_p[g][threadIdx.x];
            sq += red_q[g][threadIdx.x];
        }
        part[threadIdx.x][0] = sp;
        part[threadIdx.x][1] = sq;
    }
    cluster_sync_all();
    // CTA `rank` finishes channels [rank*16, rank*16 + 16) of the chunk
    constexpr int kPer = kChunk / kSlabs;
    if (threadIdx.x < kPer) {
        const int cl = rank * kPer + threadIdx.x;
        const int cc = chunk * kChunk + cl;
        long long sp = 0, sq = 0;
        const uint32_t la = smem_u32(&part[cl][0]);
#pragma unroll
        for (int k = 0; k < kSlabs; ++k) {
            long long a, bq;
            ld_peer_pair(la, static_cast<uint32_t>(k), a, bq);
            sp += a;
            sq += bq;
        }
        if (cc < C) {
            const __int128 t = static_cast<__int128>(sp) * (static_cast<__int128>(1) << 36) + static_cast<__int128>(sq);
            const double s = i128_to_f64_rn(t) * 0x1p-60;     // exact power-of-two scaling
            const double m = __ddiv_rn(s, static_cast<double>(N));
            mean64[static_cast<size_t>(b) * C + cc] = m;
            mean32[static_cast<size_t>(b) * C + cc] = __double2float_rn(m);
        }
    }
    cluster_sync_all();    // peers may still be reading this CTA's partial sums
}

// ------------------------------------------------------------------ 2. score + select

// Order-preserving map float -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// fp64 score of one token in the exact evaluation order: lane l sums channels
// [l*q, (l+1)*q) as a halving tree, the 32 lane sums are combined pairwise by
// the xor butterfly (the top five levels of the same tree; C = 32 q).
__device__ double tree64(const __nv_bfloat16* x, const double* m, int n)
{
    if (n == 1) {
        const double d = __dsub_rn(static_cast<double>(__bfloat162float(x[0])), m[0]);
        return __dmul_rn(d, d);
    }
    const int h = n / 2;
    const double a = tree64(x, m, h);
    const double bb = tree64(x + h, m + h, n - h);
    return __dadd_rn(a, bb);
}

// The rank-`ra`-largest of ka[0..n) and the rank-`rb`-largest of kb[0..n)
// (1-based), by 8-bit radix select with warp-aggregated shared histograms.
// All threads of the CTA call it.
__device__ void dual_radix_select(const uint32_t* ka, int ra, const uint32_t* kb, int rb, int n,
                                  int (*hist)[256], int* sel, uint32_t& out_a, uint32_t& out_b)
{
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    uint32_t pre_a = 0, pre_b = 0, msk = 0;
    int want_a = ra, want_b = rb;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int j = tid; j < 512; j += nt) hist[j >> 8][j & 255] = 0;
        __syncthreads();
        for (int base = warp * 32; base < n; base += nt) {
            const int i = base + lane;
            uint32_t da = 0xFFFFFFFFu, db = 0xFFFFFFFFu;
            if (i < n) {
                const uint32_t a = ka[i], bb = kb[i];
                if ((a & msk) == pre_a) da = (a >> shift) & 255u;
                if ((bb & msk) == pre_b) db = (bb >> shift) & 255u;
            }
            const uint32_t pa = __match_any_sync(0xffffffffu, da);
            if (da != 0xFFFFFFFFu && lane == __ffs(pa) - 1) atomicAdd(&hist[0][da], __popc(pa));
            const uint32_t pb = __match_any_sync(0xffffffffu, db);
            if (db != 0xFFFFFFFFu && lane == __ffs(pb) - 1) atomicAdd(&hist[1][db], __popc(pb));
        }
        __syncthreads();
        if (warp < 2) {
            // lane l owns digits 255-8l .. 248-8l (descending)
            const int* hh = hist[warp];
            const int want = warp ? want_b : want_a;
            int cnt[8];
            int tot = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                cnt[k] = hh[255 - 8 * lane - k];
                tot += cnt[k];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const int excl = incl - tot;
            if (excl < want && want <= incl) {
                int run = excl;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (run < want && want <= run + cnt[k]) {
                        sel[2 * warp] = 255 - 8 * lane - k;
                        sel[2 * warp + 1] = want - run;
                    }
                    run += cnt[k];
                }
            }
        }
        __syncthreads();
        pre_a |= static_cast<uint32_t>(sel[0]) << shift;
        want_a = sel[1];
        pre_b |= static_cast<uint32_t>(sel[2]) << shift;
        want_b = sel[3];
        msk |= 0xFFu << shift;
    }
    out_a = pre_a;
    out_b = pre_b;
}

// Exclusive prefix over the CTA's warps of per-warp totals v (lane-uniform);
// returns this warp's offset and writes the total.  All threads call it.
__device__ __forceinline__ int warp_offsets(int v, int* scratch, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    int off = 0, tot = 0;
    for (int w = 0; w < nw; ++w) {
        const int s = scratch[w];
        off += w < warp ? s : 0;
        tot += s;
    }
    __syncthreads();
    *total = tot;
    return off;
}

__global__ void __launch_bounds__(kScoreThreads)
    pivot_score_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, int K, const float* __restrict__ mean32,
                       const double* __restrict__ mean64, float* __restrict__ lo_g, float* __restrict__ hi_g,
                       float* __restrict__ scores, int* __restrict__ counters, int* __restrict__ band_idx_g,
                       double* __restrict__ band_score_g, int32_t* __restrict__ idx_out, int32_t* status)
{
    extern __shared__ __align__(16) uint8_t psm[];
    float* m_s = reinterpret_cast<float*>(psm);                                   // [C]
    uint32_t* klo = reinterpret_cast<uint32_t*>(psm + ((static_cast<size_t>(C) * 4 + 15) & ~size_t(15)));  // [N]
    uint32_t* khi = klo + N;                                                      // [N]
    uint8_t* flg = reinterpret_cast<uint8_t*>(khi + N);                           // [N]
    __shared__ int hist[2][256];
    __shared__ int sel[4];
    __shared__ int wsc[kScoreWarps];
    __shared__ float red[kScoreWarps];
    __shared__ int is_last;

    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();   // the channel means of the colsum kernel

    float ss = 0.f;
    for (int c = tid; c < C; c += kScoreThreads) {
        const float m = mean32[static_cast<size_t>(b) * C + c];
        m_s[c] = m;
        ss = __fmaf_ru(m, m, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss = __fadd_ru(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float n2 = 0.f;
#pragma unroll
    for (int w = 0; w < kScoreWarps; ++w) n2 = __fadd_ru(n2, red[w]);
    const float mn = __fsqrt_ru(n2);                                    // >= ||m'||
    const float E = __fadd_ru(__fmul_ru(mn, 0x1.000002p-24f), 0x1p-120f);   // >= ||m' - mu||
    const int nchunk = C / 8;                                           // 16-byte chunks per row
    const int h1 = (nchunk + 31) / 32;
    const float c1 = static_cast<float>(h1 + 8 + 3) * 0x1p-24f;
    const float E3 = __fmul_ru(3.f, __fmul_ru(E, E));
    const float mn2 = __fadd_ru(__fmul_ru(mn, mn), 1.f);
    const uint64_t neg1 = f2_pack(-1.f, -1.f);

    for (int t = 0; t < kTokPerWarp; ++t) {
        const int i = blockIdx.x * kScoreTok + warp * kTokPerWarp + t;
        if (i >= N) break;
        const uint4* row = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(b) * N + i) * C);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        for (int k0 = 0; k0 < h1; k0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int ch = lane + 32 * (k0 + k);
                v[k] = ch < nchunk ? __ldg(row + ch) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int ch = lane + 32 * (k0 + k);
                if (ch < nchunk) {
                    const float4 ma = *reinterpret_cast<const float4*>(m_s + ch * 8);
                    const float4 mb = *reinterpret_cast<const float4*>(m_s + ch * 8 + 4);
                    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                    const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint64_t x2 = f2_pack(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
                        const uint64_t d2 = f2_fma(f2_pack(mm[2 * e], mm[2 * e + 1]), neg1, x2);   // fl(x - m')
                        acc[e] = f2_fma(d2, d2, acc[e]);
                    }
                }
            }
        }
        float a[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_unpack(acc[e], a[2 * e], a[2 * e + 1]);
        float s = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) {
            if (!(s >= 0.f) || isinf(s)) atomicCAS(status, 0, VAR_ERR_NUMERIC);   // nan / inf input
            const float e1 = __fmul_ru(c1, s);
            const float rs = __fsqrt_ru(__fmul_ru(s, __fadd_ru(1.f, __fmul_ru(2.f, c1))));
            const float e2 = __fadd_ru(__fmul_ru(__fmul_ru(2.f, E), rs), E3);
            const float e3 = __fmul_ru(0x1p-44f, __fadd_ru(__fadd_ru(s, __fmul_ru(__fmul_ru(2.f, mn), rs)), mn2));
            const float eps = __fadd_ru(__fadd_ru(e1, e2), e3);
            const size_t o = static_cast<size_t>(b) * N + i;
            lo_g[o] = __fsub_rd(s, eps);
            hi_g[o] = __fadd_ru(s, eps);
            if (scores) scores[o] = s;
        }
    }

    // ---- the last CTA of batch element b selects
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(&counters[b], 1) == static_cast<int>(gridDim.x) - 1;
    __syncthreads();
    if (!is_last || K == 0) return;
    __threadfence();
    int32_t* out = idx_out + static_cast<size_t>(b) * K;
    if (K == N) {
        for (int j = tid; j < N; j += kScoreThreads) out[j] = j;
        return;
    }
    for (int j = tid; j < N; j += kScoreThreads) {
        klo[j] = f32_key(__ldcg(lo_g + static_cast<size_t>(b) * N + j));
        khi[j] = f32_key(__ldcg(hi_g + static_cast<size_t>(b) * N + j));
    }
    __syncthreads();
    uint32_t t_lo, t_hi;
    dual_radix_select(klo, K, khi, K + 1, N, hist, sel, t_lo, t_hi);

    // classify (1 certainly kept, 2 band, 0 certainly dropped); warp w owns a
    // contiguous range of tokens, so ballots keep the output ascending
    const int per_warp = ((N + kScoreWarps - 1) / kScoreWarps + 31) & ~31;
    const int w0 = min(N, warp * per_warp), w1 = min(N, w0 + per_warp);
    int n_in = 0, n_band = 0;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        int f = 0;
        if (i < w1) {
            f = klo[i] > t_hi ? 1 : (khi[i] < t_lo ? 0 : 2);
            flg[i] = static_cast<uint8_t>(f);
        }
        n_in += __popc(__ballot_sync(0xffffffffu, f == 1));
        n_band += __popc(__ballot_sync(0xffffffffu, f == 2));
    }
    int tot_in, tot_band;
    const int off_in = warp_offsets(n_in, wsc, &tot_in);
    const int off_band = warp_offsets(n_band, wsc, &tot_band);
    const int need = K - tot_in;
    if (need < 0 || need > tot_band) {
        if (tid == 0) atomicCAS(status, 0, VAR_ERR_NUMERIC);
        return;
    }
    const uint32_t lt = (1u << lane) - 1u;
    if (need == 0 || need == tot_band) {
        // the band is decided by count alone
        const bool keep_band = need > 0;
        int pos = off_in + (keep_band ? off_band : 0);
        for (int i0 = w0; i0 < w1; i0 += 32) {
            const int i = i0 + lane;
            const int f = i < w1 ? flg[i] : 0;
            const bool kept = f == 1 || (f == 2 && keep_band);
            const uint32_t m = __ballot_sync(0xffffffffu, kept);
            if (kept) out[pos + __popc(m & lt)] = i;
            pos += __popc(m);
        }
        return;
    }
    // fp64 re-score of the band in the exact evaluation order
    int* band_idx = band_idx_g + static_cast<size_t>(b) * N;
    double* band_score = band_score_g + static_cast<size_t>(b) * N;
    {
        int pos = off_band;
        for (int i0 = w0; i0 < w1; i0 += 32) {
            const int i = i0 + lane;
            const bool inb = i < w1 && flg[i] == 2;
            const uint32_t m = __ballot_sync(0xffffffffu, inb);
            if (inb) band_idx[pos + __popc(m & lt)] = i;
            pos += __popc(m);
        }
    }
    __syncthreads();
    const int q = C / 32;
    const double* mb = mean64 + static_cast<size_t>(b) * C;
    for (int j = warp; j < tot_band; j += kScoreWarps) {
        const int i = band_idx[j];
        const __nv_bfloat16* row = x + (static_cast<size_t>(b) * N + i) * C;
        double v = tree64(row + lane * q, mb + lane * q, q);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) v = __dadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) band_score[j] = v;
    }
    __syncthreads();
    for (int j = tid; j < tot_band; j += kScoreThreads) {
        const double sj = band_score[j];
        const int ij = band_idx[j];
        int better = 0;
        for (int t = 0; t < tot_band && better < need; ++t) {
            const double st = band_score[t];
            better += (st > sj) || (st == sj && band_idx[t] < ij);
        }
        flg[ij] = better < need ? 1 : 0;
    }
    __syncthreads();
    int n_sel = 0;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        n_sel += __popc(__ballot_sync(0xffffffffu, i < w1 && flg[i] == 1));
    }
    int tot_sel;
    int pos = warp_offsets(n_sel, wsc, &tot_sel);
    if (tid == 0 && tot_sel != K) atomicCAS(status, 0, VAR_ERR_NUMERIC);
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const bool kept = i < w1 && flg[i] == 1;
        const uint32_t m = __ballot_sync(0xffffffffu, kept);
        if (kept && pos + __popc(m & lt) < K) out[pos + __popc(m & lt)] = i;
        pos += __popc(m);
    }
}

size_t score_smem_bytes(int N, int C)
{
    return ((static_cast<size_t>(C) * 4 + 15) & ~size_t(15)) + static_cast<size_t>(N) * 9;
}

}  // namespace

size_t pivot_workspace_bytes(int B, int N, int C) { return pivot_ws_layout(B, N, C).total; }

int launch_pivot_select(int B, int N, int C, const void* xv, int keep_k, int32_t* idx, float* scores,
                        void* ws, size_t ws_bytes, cudaStream_t st)
{
    const PivotWs w = pivot_ws_layout(B, N, C);
    if (ws_bytes < w.total) return VAR_ERR_WORKSPACE;
    const size_t smem = score_smem_bytes(N, C);
    if (smem > kScoreSmemMax) return VAR_ERR_UNSUPPORTED;
    int32_t* status = device_status_ptr();
    if (!status) return VAR_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return VAR_ERR_CUDA;
    {
        static std::mutex mu;
        static bool attr[64] = {};
        std::lock_guard<std::mutex> lk(mu);
        if (!attr[dev]) {
            if (cudaFuncSetAttribute(pivot_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kScoreSmemMax) != cudaSuccess)
                return VAR_ERR_CUDA;
            attr[dev] = true;
        }
    }
    auto* base = static_cast<uint8_t*>(ws);
    auto* m64 = reinterpret_cast<double*>(base + w.mean64);
    auto* m32 = reinterpret_cast<float*>(base + w.mean32);
    auto* lok = reinterpret_cast<float*>(base + w.lok);
    auto* hik = reinterpret_cast<float*>(base + w.hik);
    auto* bidx = reinterpret_cast<int*>(base + w.band_idx);
    auto* bsc = reinterpret_cast<double*>(base + w.band_score);
    auto* cnt = reinterpret_cast<int*>(base + w.counters);
    const auto* x = static_cast<const __nv_bfloat16*>(xv);

    {
        const dim3 grid(kSlabs, (C + kChunk - 1) / kChunk, B);
        pivot_colsum_kernel<<<grid, kSumThreads, 0, st>>>(x, N, C, m64, m32, cnt, status);
        if (cudaGetLastError() != cudaSuccess) return VAR_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kScoreTok - 1) / kScoreTok, B, 1);
    cfg.blockDim = dim3(kScoreThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, pivot_score_kernel, x, N, C, keep_k,
                                             static_cast<const float*>(m32), static_cast<const double*>(m64),
                                             lok, hik, scores, cnt, bidx, bsc, idx, status);
    return cuda_status(e);
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot allocate device memory at the
// point where they select pivots: an engine that hands out all device memory
// itself and gives a plug-in no workspace, or a latency-critical stream where
// cudaMalloc (which may synchronise the device) is not allowed after start-up.
// For them the workspace lives in this file-scope array instead, sized for
// B <= 4, N <= 16384, C <= 4096 (about 1.5 MB).  Every GPU that loads the
// library holds it until the process exits.

constexpr int kNoAllocMaxB = 4;
constexpr int kNoAllocMaxN = 16384;
constexpr int kNoAllocMaxC = 4096;
constexpr size_t kNoAllocBytes = pivot_ws_layout(kNoAllocMaxB, kNoAllocMaxN, kNoAllocMaxC).total;

static __device__ __align__(256) uint8_t g_pivot_scratch[kNoAllocBytes];

// Device address of g_pivot_scratch on the current device.  Host code may not
// use the symbol itself (it names a host-side shadow); the address is looked
// up once per device, with that device current, and cached.
static uint8_t* pivot_scratch_ptr()
{
    static std::mutex mu;
    static uint8_t* cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pivot_scratch) != cudaSuccess || !p) return nullptr;
        cache[dev] = static_cast<uint8_t*>(p);
    }
    return cache[dev];
}

}  // namespace varattn

extern "C" int var_pivot_select_noalloc(const var_problem* p, int32_t step, const void* x,
                                        int32_t channels, int32_t keep_k, int32_t* idx, float* scores,
                                        void* stream)
{
    using namespace varattn;
    if (!p || step < 0 || step >= p->n_scales || p->n_scales > VAR_MAX_SCALES) return VAR_ERR_INVALID_ARG;
    if (p->batch <= 0 || p->side[step] <= 0 || p->side[step] > 4096) return VAR_ERR_INVALID_ARG;
    if (!x || channels <= 0 || channels % 32 != 0) return VAR_ERR_INVALID_ARG;
    const int B = p->batch;
    const int N = p->side[step] * p->side[step];
    if (keep_k < 0 || keep_k > N) return VAR_ERR_INVALID_ARG;
    if (keep_k > 0 && !idx) return VAR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0) return VAR_ERR_UNSUPPORTED;
    if (B > kNoAllocMaxB || N > kNoAllocMaxN || channels > kNoAllocMaxC) return VAR_ERR_WORKSPACE;
    const size_t need = pivot_workspace_bytes(B, N, channels);
    if (need > kNoAllocBytes) return VAR_ERR_WORKSPACE;
    uint8_t* ws = pivot_scratch_ptr();
    if (!ws) return VAR_ERR_CUDA;
    // Nothing in the scratch needs clearing: every word is written before it
    // is read within a call (the colsum kernel resets the per-batch counters).
    return launch_pivot_select(B, N, channels, x, keep_k, idx, scores, ws, kNoAllocBytes,
                               static_cast<cudaStream_t>(stream));
}
