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
// differences), reached with fp32 work on nearly every token.  Three kernels:
//
//   1. colsum (HBM pass over X).  Exact channel sums.  A cluster of 4 CTAs
//      owns a 128-channel chunk of one batch element, each CTA a slab of
//      rows streamed through a cp.async ring in shared memory.  Per element:
//      x = hi + lo split exactly by two fp32 "magic" additions (hi a multiple
//      of 2^-13, |x| < 512; lo a multiple of 2^-36), the float bit patterns
//      summed as wrapping 32-bit integers, which is an exact fixed-point sum.
//      A thread that meets |x| >= 512 redoes its rows in 64-bit fixed point.
//      The cluster merges its CTAs' partial sums through distributed shared
//      memory; the exact sum is rounded once to fp64, divided by N (the fp64
//      mean), and rounded to fp32 for the scores.
//   2. score (L2 pass over X; the first chunks of each token are read before
//      the wait for the means).  One warp per token: fp32 score with a
//      rigorous bound eps_i >= |fp32 score - fp64 score| (below), stored as
//      lo_i = score - eps (rounded down), hi_i = score + eps (rounded up).
//   3. select, one 1024-thread CTA per batch element, keys in registers:
//      T_lo = K-th largest lo, T_hi = (K+1)-th largest hi (histogram
//      narrowing, then brute force on a small range); lo_i > T_hi =>
//      certainly kept, hi_i < T_lo => certainly dropped; the band in between
//      is decided by count (all kept or all dropped) or re-scored in fp64 in
//      the exact evaluation order, the remaining slots going to the best band
//      tokens by (score desc, index asc).  Compaction keeps ascending order.
//   Kernels 2 and 3 are programmatic dependent launches of their predecessor.
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

constexpr int kSlabs = 4;                 // CTAs per cluster: row slabs of one chunk
constexpr int kChunk = 128;               // channels per chunk (256 bytes of a row)
constexpr int kSegs = kChunk / 8;         // 16-byte segments of a chunk row
constexpr int kSumThreads = 512;
constexpr int kRowGroups = kSumThreads / kSegs;   // rows per CTA pass (a thread takes 2 per stage)
constexpr int kStageRows = 64;            // rows per cp.async stage (16 KB)
constexpr int kStages = 4;                // stages in flight
constexpr int kRingBytes = kStages * kStageRows * kChunk * 2;

constexpr int kScoreThreads = 256;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kTokPerWarp = 2;
constexpr int kScoreTok = kScoreWarps * kTokPerWarp;   // tokens per score CTA

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxKeysPerThread = 16;     // N <= kSelThreads * kMaxKeysPerThread
constexpr int kMaxN = kSelThreads * kMaxKeysPerThread;
constexpr int kSelBins = 2048;            // histogram bins per narrowing level (power of two)
constexpr int kSelCand = 256;             // ranges this small are ranked by brute force

constexpr float kMagA = 1536.0f;          // 1.5 * 2^10: ulp 2^-13 on [1024, 2048)
constexpr float kMagB = 0x1.8p-13f;       // 1.5 * 2^-13: ulp 2^-36 on [2^-13, 2^-12)
constexpr float kFastMax = 512.0f;        // |x| below this takes the two-window path

struct PivotWs {
    size_t mean64, mean32, lok, hik, band_idx, band_score, total;
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
    w.total = o;
    return w;
}

// ------------------------------------------------------------------ PTX helpers

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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int n>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory"); }

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

// Adds rows a and b of 8 channels (one 16-byte word each) to the two-window
// fixed-point sums: acc_a in ulps of 2^-13 (plus bits(kMagA) per row), acc_b
// in ulps of 2^-36 (plus bits(kMagB) per row); mx tracks max |x|.
__device__ __forceinline__ void accum_rows2(const uint4& va, const uint4& vb, uint32_t (&acc_a)[8],
                                            uint32_t (&acc_b)[8], float& mx)
{
    const uint64_t mag_a = f2_pack(kMagA, kMagA), mag_b = f2_pack(kMagB, kMagB);
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float sa[2], ta[2], sb[2], tb[2];
        {
            const float x0 = __uint_as_float(wa[e] << 16), x1 = __uint_as_float(wa[e] & 0xFFFF0000u);
            const uint64_t x2 = f2_pack(x0, x1);
            const uint64_t s2 = f2_add(x2, mag_a);                 // RN(x + 1.5*2^10)
            const uint64_t l2 = f2_sub(x2, f2_sub(s2, mag_a));     // x - hi, exact
            const uint64_t t2 = f2_add(l2, mag_b);                 // RN(lo + 1.5*2^-13), exact
            f2_unpack(s2, sa[0], sa[1]);
            f2_unpack(t2, ta[0], ta[1]);
            mx = fmax3(mx, fabsf(x0), fabsf(x1));
        }
        {
            const float x0 = __uint_as_float(wb[e] << 16), x1 = __uint_as_float(wb[e] & 0xFFFF0000u);
            const uint64_t x2 = f2_pack(x0, x1);
            const uint64_t s2 = f2_add(x2, mag_a);
            const uint64_t l2 = f2_sub(x2, f2_sub(s2, mag_a));
            const uint64_t t2 = f2_add(l2, mag_b);
            f2_unpack(s2, sb[0], sb[1]);
            f2_unpack(t2, tb[0], tb[1]);
            mx = fmax3(mx, fabsf(x0), fabsf(x1));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            acc_a[2 * e + h] += __float_as_uint(sa[h]) + __float_as_uint(sb[h]);
            acc_b[2 * e + h] += __float_as_uint(ta[h]) + __float_as_uint(tb[h]);
        }
    }
}

__global__ void __cluster_dims__(kSlabs, 1, 1) __launch_bounds__(kSumThreads)
    pivot_colsum_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, double* __restrict__ mean64,
                        float* __restrict__ mean32, int32_t* status)
{
    extern __shared__ __align__(128) uint8_t ring[];                // [kStages][kStageRows][kChunk] bf16
    __shared__ __align__(16) long long part[kChunk][2];              // this CTA's (p, q) per channel

    pdl_launch_dependents();
    const int rank = static_cast<int>(cluster_rank());    // == blockIdx.x (the cluster spans x)
    const int chunk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const int rg = tid / kSegs, seg = tid % kSegs;
    const int c = chunk * kChunk + seg * 8;
    const bool cvalid = c < C;
    const int slab = (N + kSlabs - 1) / kSlabs;
    const int r0 = min(N, rank * slab), r1 = min(N, r0 + slab);
    const int nstage = (r1 - r0 + kStageRows - 1) / kStageRows;
    const __nv_bfloat16* base = x + static_cast<size_t>(b) * N * C + c;
    const uint32_t ring_s = smem_u32(ring);

    // stage st: rows r0 + st*64 + [0, 64); this thread copies rows rg and rg + kRowGroups
    auto issue = [&](int st) {
        if (st < nstage && cvalid) {
            const int rbase = r0 + st * kStageRows;
            const uint32_t slot = ring_s + static_cast<uint32_t>((st % kStages) * kStageRows * kChunk * 2);
#pragma unroll
            for (int j = 0; j < kStageRows / kRowGroups; ++j) {
                const int rr = rg + kRowGroups * j;
                if (rbase + rr < r1)
                    cp_async16(slot + static_cast<uint32_t>(rr * kChunk * 2 + seg * 16),
                               base + static_cast<size_t>(rbase + rr) * C);
            }
        }
        cp_async_commit();
    };

    uint32_t acc_a[8], acc_b[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc_a[e] = acc_b[e] = 0u;
    float mx = 0.f;
    static_assert(kStageRows == 2 * kRowGroups, "a thread takes rows rg and rg + kRowGroups of a stage");
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) issue(st);
    for (int st = 0; st < nstage; ++st) {
        issue(st + kStages - 1);
        cp_async_wait<kStages - 1>();
        __syncthreads();
        if (cvalid) {
            const uint8_t* slot = ring + (st % kStages) * kStageRows * kChunk * 2 + seg * 16;
            const int rows = min(kStageRows, r1 - r0 - st * kStageRows);
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            uint4 va, vb;
            if (rows == kStageRows) {
                va = *reinterpret_cast<const uint4*>(slot + rg * kChunk * 2);
                vb = *reinterpret_cast<const uint4*>(slot + (rg + kRowGroups) * kChunk * 2);
            } else {                                   // rows past the slab add x = 0
                va = rg < rows ? *reinterpret_cast<const uint4*>(slot + rg * kChunk * 2) : z;
                vb = rg + kRowGroups < rows ? *reinterpret_cast<const uint4*>(slot + (rg + kRowGroups) * kChunk * 2) : z;
            }
            accum_rows2(va, vb, acc_a, acc_b, mx);
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // exact sum of this thread's elements = p * 2^-24 + q * 2^-60
    long long p[8], q[8];
    bool bad = false;
    if (mx < kFastMax) {
        // every row slot added bits(M) + (its value in ulps of the window)
        const uint32_t nr = static_cast<uint32_t>(nstage * 2);          // row slots per thread
        const uint32_t bias_a = nr * __float_as_uint(kMagA), bias_b = nr * __float_as_uint(kMagB);
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
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + static_cast<size_t>(rr) * C));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                accum_fixed(w[e] & 0xFFFFu, p[2 * e], q[2 * e], bad);
                accum_fixed(w[e] >> 16, p[2 * e + 1], q[2 * e + 1], bad);
            }
        }
    }
    if (bad) atomicCAS(status, 0, VAR_ERR_NUMERIC);
    // the two row groups of a warp share channels (lanes l and l ^ 16)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        p[e] += __shfl_xor_sync(0xffffffffu, p[e], 16);
        q[e] += __shfl_xor_sync(0xffffffffu, q[e], 16);
    }
    // lanes < 16 hold a warp's partial sums: entry (warp, e, segment) of 16 bytes,
    // so a warp's stores of one e are contiguous (no bank conflicts)
    static_assert(kSegs == 16, "two row groups per warp");
    longlong2* red = reinterpret_cast<longlong2*>(ring);    // [warps][8][16], the ring is idle now
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < 16) {
#pragma unroll
        for (int e = 0; e < 8; ++e) red[(warp * 8 + e) * 16 + seg] = make_longlong2(p[e], q[e]);
    }
    __syncthreads();
    if (tid < kChunk) {
        // thread (e, segment) = (tid / 16, tid % 16): channel segment*8 + e, summed over the warps
        const int e = tid >> 4, sg = tid & 15;
        long long sp = 0, sq = 0;
#pragma unroll
        for (int w = 0; w < kSumThreads / 32; ++w) {
            const longlong2 v = red[(w * 8 + e) * 16 + sg];
            sp += v.x;
            sq += v.y;
        }
        part[sg * 8 + e][0] = sp;
        part[sg * 8 + e][1] = sq;
    }
    cluster_sync_all();
    // CTA `rank` finishes channels [rank*kPer, rank*kPer + kPer) of the chunk: thread
    // (channel, peer) = (tid / kSlabs, tid % kSlabs) reads one peer's partial
    // sums, the kSlabs lanes of a channel add them
    constexpr int kPer = kChunk / kSlabs;
    if (tid < kPer * kSlabs) {
        const int cl = rank * kPer + tid / kSlabs;
        const int cc = chunk * kChunk + cl;
        long long sp, sq;
        ld_peer_pair(smem_u32(&part[cl][0]), static_cast<uint32_t>(tid % kSlabs), sp, sq);
#pragma unroll
        for (int off = 1; off < kSlabs; off <<= 1) {
            sp += __shfl_xor_sync(0xffffffffu, sp, off);
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
        }
        if (tid % kSlabs == 0 && cc < C) {
            const __int128 t = static_cast<__int128>(sp) * (static_cast<__int128>(1) << 36) + static_cast<__int128>(sq);
            const double s = i128_to_f64_rn(t) * 0x1p-60;     // exact power-of-two scaling
            const double m = __ddiv_rn(s, static_cast<double>(N));
            mean64[static_cast<size_t>(b) * C + cc] = m;
            mean32[static_cast<size_t>(b) * C + cc] = __double2float_rn(m);
        }
    }
    cluster_sync_all();    // peers may still be reading this CTA's partial sums
}

// ------------------------------------------------------------------ 2. score

__global__ void __launch_bounds__(kScoreThreads, 4)
    pivot_score_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, const float* __restrict__ mean32,
                       float* __restrict__ lo_g, float* __restrict__ hi_g, float* __restrict__ scores,
                       int32_t* status)
{
    extern __shared__ __align__(16) float m_s[];   // [C]
    __shared__ float red[kScoreWarps];
    const int b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();
    const int nchunk = C / 8;                                           // 16-byte chunks per row
    const int h1 = (nchunk + 31) / 32;
    // the warp's tokens are scored together: one read of the means serves both
    const int i0 = blockIdx.x * kScoreTok + warp * kTokPerWarp;
    const uint4* rows[kTokPerWarp];
    bool tv[kTokPerWarp];
#pragma unroll
    for (int t = 0; t < kTokPerWarp; ++t) {
        tv[t] = i0 + t < N;
        rows[t] = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(b) * N + min(i0 + t, N - 1)) * C);
    }
    constexpr int kBatch = 4;                                           // chunks per token in flight
    // X is not written by the colsum kernel: the first batch is read before
    // waiting for the means
    uint4 v[kTokPerWarp][kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
        const int ch = lane + 32 * k;
#pragma unroll
        for (int t = 0; t < kTokPerWarp; ++t)
            v[t][k] = (ch < nchunk && tv[t]) ? __ldg(rows[t] + ch) : make_uint4(0u, 0u, 0u, 0u);
    }
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
    const float c1 = static_cast<float>(h1 + 8 + 3) * 0x1p-24f;
    const float E3 = __fmul_ru(3.f, __fmul_ru(E, E));
    const float mn2 = __fadd_ru(__fmul_ru(mn, mn), 1.f);
    const uint64_t neg1 = f2_pack(-1.f, -1.f);

    uint64_t acc[kTokPerWarp][4];
#pragma unroll
    for (int t = 0; t < kTokPerWarp; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0ull;
    for (int k0 = 0; k0 < h1; k0 += kBatch) {
        if (k0 > 0) {
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int ch = lane + 32 * (k0 + k);
#pragma unroll
                for (int t = 0; t < kTokPerWarp; ++t)
                    v[t][k] = (ch < nchunk && tv[t]) ? __ldg(rows[t] + ch) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int ch = lane + 32 * (k0 + k);
            if (ch < nchunk) {
                const float4 ma = *reinterpret_cast<const float4*>(m_s + ch * 8);
                const float4 mb = *reinterpret_cast<const float4*>(m_s + ch * 8 + 4);
                const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
                for (int t = 0; t < kTokPerWarp; ++t) {
                    const uint32_t w[4] = {v[t][k].x, v[t][k].y, v[t][k].z, v[t][k].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint64_t x2 = f2_pack(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
                        const uint64_t d2 = f2_fma(f2_pack(mm[2 * e], mm[2 * e + 1]), neg1, x2);   // fl(x - m')
                        acc[t][e] = f2_fma(d2, d2, acc[t][e]);
                    }
                }
            }
        }
    }
    float sums[kTokPerWarp];
#pragma unroll
    for (int t = 0; t < kTokPerWarp; ++t) {
        float a[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_unpack(acc[t][e], a[2 * e], a[2 * e + 1]);
        float sm = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
        sums[t] = sm;
    }
    // lane t finishes token t of the warp: bound and outputs
    if (lane < kTokPerWarp) {
        const int i = blockIdx.x * kScoreTok + warp * kTokPerWarp + lane;
        float s = sums[0];
#pragma unroll
        for (int t = 1; t < kTokPerWarp; ++t)
            if (lane == t) s = sums[t];
        if (i < N) {
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
}

// ------------------------------------------------------------------ 3. select

// Order-preserving map float -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// fp64 score of one token in the exact evaluation order: lane l sums channels
// [l*q, (l+1)*q) as a halving tree, the 32 lane sums are combined pairwise by
// the xor butterfly (the top five levels of the same tree; C = 32 q).
// Subtrees of 8 or fewer leaves whose size is a power of two are expanded at
// compile time; above them the tree (split at n/2 rounded down) is walked
// iteratively with a small explicit stack, so no recursion and little stack.
template <int n>
__device__ __forceinline__ double tree64_pow2(const __nv_bfloat16* x, const double* m)
{
    if constexpr (n == 1) {
        const double d = __dsub_rn(static_cast<double>(__bfloat162float(x[0])), m[0]);
        return __dmul_rn(d, d);
    } else {
        const double a = tree64_pow2<n / 2>(x, m);
        const double bb = tree64_pow2<n / 2>(x + n / 2, m + n / 2);
        return __dadd_rn(a, bb);
    }
}

__device__ __forceinline__ bool tree64_leaf_block(const __nv_bfloat16* x, const double* m, int n, double& r)
{
    switch (n) {
    case 1: r = tree64_pow2<1>(x, m); return true;
    case 2: r = tree64_pow2<2>(x, m); return true;
    case 4: r = tree64_pow2<4>(x, m); return true;
    case 8: r = tree64_pow2<8>(x, m); return true;
    default: return false;
    }
}

__device__ __noinline__ double tree64(const __nv_bfloat16* x, const double* m, int n)
{
    constexpr int kDepth = 16;                 // n <= 2^15 leaves
    int fs[kDepth], fn[kDepth], fst[kDepth];   // frame: start, size, state
    double fl[kDepth];                         // frame: left subtree's sum
    int sp = 0;
    fs[0] = 0; fn[0] = n; fst[0] = 0; sp = 1;
    double ret = 0.0;
    while (sp > 0) {
        const int t = sp - 1;
        double leaf;
        if (fst[t] == 0 && tree64_leaf_block(x + fs[t], m + fs[t], fn[t], leaf)) {
            ret = leaf;
            --sp;
        } else if (fst[t] == 0) {              // descend left
            fst[t] = 1;
            fs[sp] = fs[t]; fn[sp] = fn[t] / 2; fst[sp] = 0; ++sp;
        } else if (fst[t] == 1) {              // left done: descend right
            fl[t] = ret;
            fst[t] = 2;
            fs[sp] = fs[t] + fn[t] / 2; fn[sp] = fn[t] - fn[t] / 2; fst[sp] = 0; ++sp;
        } else {                               // both done
            ret = __dadd_rn(fl[t], ret);
            --sp;
        }
    }
    return ret;
}

// Sum over threads with a larger index of v (exclusive suffix sum over the
// CTA in thread order); every thread calls it.  wtmp: kSelWarps ints.
__device__ __forceinline__ int block_suffix_excl(int v, int* wtmp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int s = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, s, off);
        if (lane + off < 32) s += y;
    }
    __syncthreads();
    if (lane == 0) wtmp[warp] = s;
    __syncthreads();
    int t = (lane > warp && lane < kSelWarps) ? wtmp[lane] : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    return t + s - v;
}

// Sum over threads with a smaller index of v (exclusive prefix sum); every
// thread calls it; *total receives the sum over the CTA.
__device__ __forceinline__ int block_prefix_excl(int v, int* wtmp, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int s = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
    }
    __syncthreads();
    if (lane == 31) wtmp[warp] = s;
    __syncthreads();
    int t = (lane < warp) ? wtmp[lane] : 0;
    int all = wtmp[lane];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        t += __shfl_xor_sync(0xffffffffu, t, off);
        all += __shfl_xor_sync(0xffffffffu, all, off);
    }
    *total = all;
    return t + s - v;
}

struct SelShared {
    int hist[2][kSelBins];
    uint32_t cand[2][kSelCand];
    int wtmp[kSelWarps];
    int blk[kMaxKeysPerThread * kSelWarps];   // per (k, warp) block: packed counts, then offsets
    uint32_t red[4][kSelWarps];
    uint32_t lo[2], hi[2];                 // narrowing state per side: inclusive key range,
    int want[2], cnt[2], done[2], ncand[2];   // the answer's rank in it, keys in it
    uint32_t res[2];
    uint8_t keep_band[kMaxN];              // band tokens kept after the fp64 re-score
};

// The r0-th largest of side 0's keys and the r1-th largest of side 1's keys
// (1-based; equal keys count separately).  Token i = tid + kSelThreads*k holds
// k0[k], k1[k] when i < n.  Each side keeps an inclusive key range holding its
// answer; a level histograms the range into power-of-two bins and keeps the bin
// where the descending count reaches the rank; a range of at most kSelCand keys
// is ranked by brute force.
template <int KPT>
__device__ void dual_kth_largest(const uint32_t (&k0)[KPT], const uint32_t (&k1)[KPT],
                                 int n, int r0, int r1, SelShared& S, uint32_t& out0, uint32_t& out1)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t mn0 = 0xFFFFFFFFu, mx0 = 0u, mn1 = 0xFFFFFFFFu, mx1 = 0u;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        if (tid + kSelThreads * k < n) {
            mn0 = min(mn0, k0[k]); mx0 = max(mx0, k0[k]);
            mn1 = min(mn1, k1[k]); mx1 = max(mx1, k1[k]);
        }
    }
    mn0 = __reduce_min_sync(0xffffffffu, mn0);
    mx0 = __reduce_max_sync(0xffffffffu, mx0);
    mn1 = __reduce_min_sync(0xffffffffu, mn1);
    mx1 = __reduce_max_sync(0xffffffffu, mx1);
    if (lane == 0) {
        S.red[0][warp] = mn0; S.red[1][warp] = mx0; S.red[2][warp] = mn1; S.red[3][warp] = mx1;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t a = __reduce_min_sync(0xffffffffu, S.red[0][lane]);
        const uint32_t bq = __reduce_max_sync(0xffffffffu, S.red[1][lane]);
        const uint32_t c = __reduce_min_sync(0xffffffffu, S.red[2][lane]);
        const uint32_t d = __reduce_max_sync(0xffffffffu, S.red[3][lane]);
        if (lane == 0) {
            S.lo[0] = a; S.hi[0] = bq; S.lo[1] = c; S.hi[1] = d;
            S.want[0] = r0; S.want[1] = r1;
            S.cnt[0] = S.cnt[1] = n;
            S.done[0] = S.done[1] = 0;
        }
    }
    __syncthreads();
    for (int level = 0; level < 8; ++level) {
        // this level's state, read by every thread before anyone updates it;
        // mode per side: 0 done, 1 histogram, 2 brute force
        int mode[2], shift[2], want[2];
        uint32_t rlo[2], rhi[2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            rlo[s] = S.lo[s];
            rhi[s] = S.hi[s];
            want[s] = S.want[s];
            mode[s] = S.done[s] ? 0 : (rlo[s] == rhi[s] ? 0 : (S.cnt[s] <= kSelCand ? 2 : 1));
            const uint32_t span_m1 = rhi[s] - rlo[s];            // span - 1
            const int bits = span_m1 ? 32 - __clz(static_cast<int>(span_m1)) : 0;   // span <= 2^bits
            shift[s] = max(0, bits - 11);
        }
        if (S.done[0] && S.done[1]) break;
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                if (!S.done[s] && rlo[s] == rhi[s]) { S.res[s] = rlo[s]; S.done[s] = 1; }
                S.ncand[s] = 0;
            }
        }
        if (mode[0] == 1 || mode[1] == 1)
            for (int j = tid; j < 2 * kSelBins; j += kSelThreads) (&S.hist[0][0])[j] = 0;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < KPT; ++k) {
            if (tid + kSelThreads * k >= n) continue;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const uint32_t key = s ? k1[k] : k0[k];
                if (!mode[s] || key < rlo[s] || key > rhi[s]) continue;
                if (mode[s] == 1) {
                    atomicAdd(&S.hist[s][(key - rlo[s]) >> shift[s]], 1);
                } else {
                    const int j = atomicAdd(&S.ncand[s], 1);
                    S.cand[s][j] = key;
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (mode[s] == 2) {
                const int nc = S.ncand[s];
                for (int t = tid; t < nc; t += kSelThreads) {
                    const uint32_t v = S.cand[s][t];
                    int g = 0, e = 0;
                    for (int u = 0; u < nc; ++u) {
                        const uint32_t w = S.cand[s][u];
                        g += w > v;
                        e += w == v;
                    }
                    if (g < want[s] && want[s] <= g + e) { S.res[s] = v; S.done[s] = 1; }
                }
            } else if (mode[s] == 1) {
                // thread t owns bins [2t, 2t + 2); count the keys in higher bins
                const int c_lo = S.hist[s][2 * tid], c_hi = S.hist[s][2 * tid + 1];
                const int above = block_suffix_excl(c_lo + c_hi, S.wtmp);
                const int cnts[2] = {c_hi, c_lo};
                int ab = above;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int cc = cnts[u];
                    if (ab < want[s] && want[s] <= ab + cc) {
                        const uint32_t bin = static_cast<uint32_t>(2 * tid + 1 - u);
                        const uint32_t lo = rlo[s] + (bin << shift[s]);
                        const uint32_t w1 = (1u << shift[s]) - 1u;
                        S.want[s] = want[s] - ab;
                        S.cnt[s] = cc;
                        S.lo[s] = lo;
                        S.hi[s] = lo + min(w1, rhi[s] - lo);
                    }
                    ab += cc;
                }
            }
        }
        __syncthreads();
    }
    out0 = S.res[0];
    out1 = S.res[1];
}

template <int KPT>
__global__ void __launch_bounds__(kSelThreads, 1)
    pivot_select_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, int K, const float* __restrict__ lo_g,
                        const float* __restrict__ hi_g, const double* __restrict__ mean64,
                        int* __restrict__ band_idx_g, double* __restrict__ band_score_g,
                        int32_t* __restrict__ idx_out, int32_t* status, int exact)
{
    __shared__ SelShared S;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();   // the scores of the score kernel
    // a pruned attention chained after this kernel (var_pruned_step) may set up
    // beside it now; it reads the index list only after this grid completes
    pdl_launch_dependents();
    int32_t* out = idx_out + static_cast<size_t>(b) * K;
    if (K == N) {
        for (int j = tid; j < N; j += kSelThreads) out[j] = j;
        return;
    }
    uint32_t ka[KPT], kh[KPT];
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        const int i = tid + kSelThreads * k;
        ka[k] = kh[k] = 0u;
        if (i < N) {
            ka[k] = f32_key(__ldcg(lo_g + static_cast<size_t>(b) * N + i));
            kh[k] = f32_key(__ldcg(hi_g + static_cast<size_t>(b) * N + i));
        }
    }
    uint32_t t_lo, t_hi;
    dual_kth_largest(ka, kh, N, K, K + 1, S, t_lo, t_hi);

    // classify: 1 certainly kept, 2 band, 0 certainly dropped.  Block (k, w) =
    // the 32 consecutive tokens kSelThreads*k + 32w + [0, 32) held by warp w,
    // so blocks in (k, w) order are in token order.
    uint32_t fin = 0u, fband = 0u;    // bit k: token k of this thread kept / in the band
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        if (tid + kSelThreads * k < N) {
            if (ka[k] > t_hi) fin |= 1u << k;
            else if (!(kh[k] < t_lo)) fband |= 1u << k;
        }
    }
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        const int ci = __popc(__ballot_sync(0xffffffffu, (fin >> k) & 1u));
        const int cb = __popc(__ballot_sync(0xffffffffu, (fband >> k) & 1u));
        if (lane == 0) S.blk[k * kSelWarps + warp] = (ci << 16) | cb;
    }
    __syncthreads();
    // offsets of the blocks: thread j < KPT*kSelWarps owns block j
    int tot;
    {
        const int v = tid < KPT * kSelWarps ? S.blk[tid] : 0;
        const int off = block_prefix_excl(v, S.wtmp, &tot);
        __syncthreads();
        if (tid < KPT * kSelWarps) S.blk[tid] = off;
        __syncthreads();
    }
    const int tot_in = tot >> 16, tot_band = tot & 0xFFFF;
    const int need = K - tot_in;
    if (need < 0 || need > tot_band) {
        if (tid == 0) atomicCAS(status, 0, VAR_ERR_NUMERIC);
        return;
    }
    if (need == 0 || need == tot_band) {
        // the band is decided by count alone
        const bool keep_band = need > 0;
#pragma unroll
        for (int k = 0; k < KPT; ++k) {
            const int off = S.blk[k * kSelWarps + warp];
            const bool kept = ((fin >> k) & 1u) || (keep_band && ((fband >> k) & 1u));
            const uint32_t mi = __ballot_sync(0xffffffffu, (fin >> k) & 1u);
            const uint32_t mb = __ballot_sync(0xffffffffu, (fband >> k) & 1u);
            const uint32_t m = keep_band ? (mi | mb) : mi;
            const int pos = (off >> 16) + (keep_band ? (off & 0xFFFF) : 0) + __popc(m & lt);
            if (kept) out[pos] = tid + kSelThreads * k;
        }
        return;
    }
    // the band's exact scores: fp64 re-score in the exact evaluation order, or
    // (exact keys, lo = hi) the key value itself
    int* band_idx = band_idx_g + static_cast<size_t>(b) * N;
    double* band_score = band_score_g + static_cast<size_t>(b) * N;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        const uint32_t mb = __ballot_sync(0xffffffffu, (fband >> k) & 1u);
        if ((fband >> k) & 1u) band_idx[(S.blk[k * kSelWarps + warp] & 0xFFFF) + __popc(mb & lt)] = tid + kSelThreads * k;
    }
    __syncthreads();
    if (exact) {
        for (int j = tid; j < tot_band; j += kSelThreads)
            band_score[j] = static_cast<double>(__ldcg(lo_g + static_cast<size_t>(b) * N + band_idx[j]));
    } else {
        const int q = C / 32;
        const double* mb64 = mean64 + static_cast<size_t>(b) * C;
        for (int j = warp; j < tot_band; j += kSelWarps) {
            const int i = band_idx[j];
            const __nv_bfloat16* row = x + (static_cast<size_t>(b) * N + i) * C;
            double v = tree64(row + lane * q, mb64 + lane * q, q);
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) v = __dadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0) band_score[j] = v;
        }
    }
    __syncthreads();
    for (int j = tid; j < tot_band; j += kSelThreads) {
        const double sj = band_score[j];
        const int ij = band_idx[j];
        int better = 0;
        for (int t = 0; t < tot_band && better < need; ++t) {
            const double st = band_score[t];
            better += (st > sj) || (st == sj && band_idx[t] < ij);
        }
        S.keep_band[ij] = better < need ? 1 : 0;
    }
    __syncthreads();
    uint32_t fsel = fin;
#pragma unroll
    for (int k = 0; k < KPT; ++k)
        if (((fband >> k) & 1u) && S.keep_band[tid + kSelThreads * k]) fsel |= 1u << k;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        const int cs = __popc(__ballot_sync(0xffffffffu, (fsel >> k) & 1u));
        if (lane == 0) S.blk[k * kSelWarps + warp] = cs;
    }
    __syncthreads();
    {
        const int v = tid < KPT * kSelWarps ? S.blk[tid] : 0;
        const int off = block_prefix_excl(v, S.wtmp, &tot);
        __syncthreads();
        if (tid < KPT * kSelWarps) S.blk[tid] = off;
        __syncthreads();
    }
    if (tid == 0 && tot != K) atomicCAS(status, 0, VAR_ERR_NUMERIC);
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
        const uint32_t m = __ballot_sync(0xffffffffu, (fsel >> k) & 1u);
        const int pos = S.blk[k * kSelWarps + warp] + __popc(m & lt);
        if (((fsel >> k) & 1u) && pos < K) out[pos] = tid + kSelThreads * k;
    }
}

}  // namespace

size_t pivot_workspace_bytes(int B, int N, int C) { return pivot_ws_layout(B, N, C).total; }

int launch_pivot_select(int B, int N, int C, const void* xv, int keep_k, int32_t* idx, float* scores,
                        void* ws, size_t ws_bytes, cudaStream_t st, int32_t* status)
{
    const PivotWs w = pivot_ws_layout(B, N, C);
    if (ws_bytes < w.total) return VAR_ERR_WORKSPACE;
    if (N > kMaxN || C > 16384) return VAR_ERR_UNSUPPORTED;
    if (ensure_smem_attr(pivot_colsum_kernel, kRingBytes) != cudaSuccess ||
        ensure_smem_attr(pivot_score_kernel, 16384 * 4) != cudaSuccess)
        return VAR_ERR_CUDA;
    auto* base = static_cast<uint8_t*>(ws);
    auto* m64 = reinterpret_cast<double*>(base + w.mean64);
    auto* m32 = reinterpret_cast<float*>(base + w.mean32);
    auto* lok = reinterpret_cast<float*>(base + w.lok);
    auto* hik = reinterpret_cast<float*>(base + w.hik);
    auto* bidx = reinterpret_cast<int*>(base + w.band_idx);
    auto* bsc = reinterpret_cast<double*>(base + w.band_score);
    const auto* x = static_cast<const __nv_bfloat16*>(xv);

    if (launch_kernel(pivot_colsum_kernel, dim3(kSlabs, (C + kChunk - 1) / kChunk, B), dim3(kSumThreads), kRingBytes,
                      st, false, x, N, C, m64, m32, status) != cudaSuccess)
        return VAR_ERR_CUDA;
    // the score and select kernels start as programmatic dependents of their predecessor
    if (launch_kernel(pivot_score_kernel, dim3((N + kScoreTok - 1) / kScoreTok, B, 1), dim3(kScoreThreads),
                      static_cast<size_t>(C) * 4, st, true, x, N, C, m32, lok, hik, scores, status) != cudaSuccess)
        return VAR_ERR_CUDA;
    if (keep_k > 0) {
        auto* fn = N <= 4 * kSelThreads ? pivot_select_kernel<4>
                   : N <= 8 * kSelThreads ? pivot_select_kernel<8>
                                          : pivot_select_kernel<kMaxKeysPerThread>;
        if (launch_kernel(fn, dim3(B), dim3(kSelThreads), 0, st, true, x, N, C, keep_k, lok, hik, m64, bidx, bsc, idx,
                          status, 0) != cudaSuccess)
            return VAR_ERR_CUDA;
    }
    return VAR_OK;
}

int launch_select_exact(int B, int N, int keep_k, const float* keys_lo, const float* keys_hi, int* band_idx,
                        double* band_score, int32_t* idx, cudaStream_t st, int32_t* status)
{
    if (N > kMaxN) return VAR_ERR_UNSUPPORTED;
    auto* fn = N <= 4 * kSelThreads ? pivot_select_kernel<4>
               : N <= 8 * kSelThreads ? pivot_select_kernel<8>
                                      : pivot_select_kernel<kMaxKeysPerThread>;
    const __nv_bfloat16* no_x = nullptr;
    const double* no_mean = nullptr;
    // a programmatic dependent of the kernel that wrote the keys (it waits for
    // that grid before reading them)
    return cuda_status(launch_kernel(fn, dim3(B), dim3(kSelThreads), 0, st, true, no_x, N, 32, keep_k, keys_lo,
                                     keys_hi, no_mean, band_idx, band_score, idx, status, 1));
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
    if (current_device(&dev) != cudaSuccess) return nullptr;
    void* p = nullptr;
    if (rt_mocked())
        return rt().get_symbol_address(&p, reinterpret_cast<const void*>(g_pivot_scratch)) == cudaSuccess
                   ? static_cast<uint8_t*>(p)
                   : nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        if (rt().get_symbol_address(&p, reinterpret_cast<const void*>(g_pivot_scratch)) != cudaSuccess || !p)
            return nullptr;
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
    StepGeom g;
    if (int rc = check_pivot_args(p, step, x, channels, keep_k, idx, &g)) return rc;
    if (g.B > kNoAllocMaxB || g.N > kNoAllocMaxN || channels > kNoAllocMaxC) return VAR_ERR_WORKSPACE;
    if (pivot_workspace_bytes(g.B, g.N, channels) > kNoAllocBytes) return VAR_ERR_WORKSPACE;
    int32_t* status = status_word(p);
    if (!status) return VAR_ERR_CUDA;
    uint8_t* ws = pivot_scratch_ptr();
    if (!ws) return VAR_ERR_CUDA;
    // Nothing in the scratch needs clearing: every word is written before it
    // is read within a call.
    return launch_pivot_select(g.B, g.N, channels, x, keep_k, idx, scores, ws, kNoAllocBytes,
                               static_cast<cudaStream_t>(stream), status);
}
