// Pivot selection for cached token pruning on sm_103a.
//
// "FastVAR: Linear Visual Autoregressive Modeling via Cached Token Pruning"
// (abstract): only pivotal tokens are forwarded; "ARVAR" Key Design 2: Top-K
// indices gather them.  Score of token i of batch element b:
//     score[b,i] = || x[b,i,:] - mean_i x[b,i,:] ||_2^2
// The K largest are kept (equal scores: lower index first), returned ascending.
//
// The ranking reproduces the fp64 evaluation (mean = fp64 channel sum / N,
// score = fp64 pairwise-halving tree over channels of rounded squared
// differences) while doing nearly all work in fp32:
//   1. colsum    exact channel sums in 64-bit fixed point (two accumulators:
//                LSB 2^-24 for |x| >= 2^-17, LSB 2^-60 below), int64 atomics;
//                integer addition is exact and order-free, so the sum is the
//                exact one and its fp64 rounding is deterministic.
//   2. finalize  fp64 mean (one correctly rounded conversion, IEEE division),
//                and its fp32 rounding for the fast path.
//   3. score     fp32 scores, one warp per token, plus a rigorous bound
//                eps_i >= |fp32 score - fp64 score| (see bound below); stores
//                lo_i = score - eps (rounded down), hi_i = score + eps (up).
//   4. select    one CTA per batch element: T_lo = K-th largest lo,
//                T_hi = (K+1)-th largest hi (radix select).  lo_i > T_hi => i is
//                certainly kept; hi_i < T_lo => certainly dropped; the band in
//                between is re-scored in fp64 in the exact evaluation order and
//                the remaining slots go to the best band tokens by (score desc,
//                index asc).  Output compaction keeps ascending order.
// Error bound for step 3: with a_c = |x_c| + |m_c|, the fp32 difference, square
// and FMA accumulation of q = C/32 terms per lane plus a 5-level shuffle tree
// err <= (q + 9.1) u sum a_c^2 (u = 2^-24); eps uses 4u (q + 16) sum a_c^2.
#include <cfloat>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace varattn {

namespace {

constexpr int kColRows = 128;      // rows per colsum CTA
constexpr int kScoreTok = 32;      // tokens per score CTA
constexpr int kSelThreads = 1024;

struct PivotWs {
    size_t hi, lo, mean64, mean32, lok, hik, band_idx, band_score, flags, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline PivotWs pivot_ws_layout(int B, int N, int C)
{
    PivotWs w;
    size_t o = 0;
    w.hi = o;         o = align256(o + sizeof(long long) * B * C);
    w.lo = o;         o = align256(o + sizeof(long long) * B * C);
    w.mean64 = o;     o = align256(o + sizeof(double) * B * C);
    w.mean32 = o;     o = align256(o + sizeof(float) * B * C);
    w.lok = o;        o = align256(o + sizeof(float) * B * N);
    w.hik = o;        o = align256(o + sizeof(float) * B * N);
    w.band_idx = o;   o = align256(o + sizeof(int) * B * N);
    w.band_score = o; o = align256(o + sizeof(double) * B * N);
    w.flags = o;      o = align256(o + sizeof(int) * B * N);
    w.total = o;
    return w;
}

// ------------------------------------------------------------------ 1. colsum

__device__ __forceinline__ void accum_fixed(uint32_t h, long long& hi, long long& lo, bool& bad)
{
    const uint32_t e = (h >> 7) & 0xFFu;
    const long long m = static_cast<long long>((h & 0x7Fu) | 0x80u);
    if (e >= 110u) {                          // |x| >= 2^-17: exponent of the LSB >= -24
        if (e >= 147u) bad = true;             // |x| >= 2^20, inf or nan
        const long long v = m << min(e - 110u, 36u);
        hi += (h & 0x8000u) ? -v : v;
    } else if (e >= 74u) {                    // 2^-53 <= |x| < 2^-17
        const long long v = m << (e - 74u);
        lo += (h & 0x8000u) ? -v : v;
    }
    // |x| < 2^-53 (and zeros, subnormals): contributes nothing
}

__global__ void __launch_bounds__(256)
    pivot_colsum_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, long long* __restrict__ hi_out,
                        long long* __restrict__ lo_out, int32_t* status)
{
    __shared__ long long red[2][8][256];
    const int b = blockIdx.z;
    const int c0 = blockIdx.x * 256;
    const int r0 = blockIdx.y * kColRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    long long hi[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lo[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    bool bad = false;
    const int c = c0 + lane * 8;
    if (c < C) {
        const int r1 = min(N, r0 + kColRows);
        const __nv_bfloat16* base = x + static_cast<size_t>(b) * N * C + c;
#pragma unroll 4
        for (int r = r0 + warp; r < r1; r += 8) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(base + static_cast<size_t>(r) * C));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                accum_fixed(w[e] & 0xFFFFu, hi[2 * e], lo[2 * e], bad);
                accum_fixed(w[e] >> 16, hi[2 * e + 1], lo[2 * e + 1], bad);
            }
        }
    }
    if (bad) atomicCAS(status, 0, VAR_ERR_NUMERIC);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        red[0][warp][lane * 8 + e] = hi[e];
        red[1][warp][lane * 8 + e] = lo[e];
    }
    __syncthreads();
    const int t = threadIdx.x;
    if (c0 + t < C) {
        long long sh = 0, sl = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            sh += red[0][w][t];
            sl += red[1][w][t];
        }
        if (sh) atomicAdd(reinterpret_cast<unsigned long long*>(hi_out + static_cast<size_t>(b) * C + c0 + t),
                          static_cast<unsigned long long>(sh));
        if (sl) atomicAdd(reinterpret_cast<unsigned long long*>(lo_out + static_cast<size_t>(b) * C + c0 + t),
                          static_cast<unsigned long long>(sl));
    }
}

// ------------------------------------------------------------------ 2. finalize

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

__global__ void pivot_finalize_kernel(const long long* __restrict__ hi, const long long* __restrict__ lo,
                                      int BC, int N, double* __restrict__ mean64, float* __restrict__ mean32)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= BC) return;
    // exact sum = hi * 2^-24 + lo * 2^-60 = (hi * 2^36 + lo) * 2^-60
    const __int128 t = static_cast<__int128>(hi[i]) * (static_cast<__int128>(1) << 36) +
                       static_cast<__int128>(lo[i]);
    const double s = i128_to_f64_rn(t) * 0x1p-60;       // exact power-of-two scaling
    const double m = __ddiv_rn(s, static_cast<double>(N));
    mean64[i] = m;
    mean32[i] = __double2float_rn(m);
}

// ------------------------------------------------------------------ 3. score

__global__ void __launch_bounds__(256)
    pivot_score_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, const float* __restrict__ mean32,
                       float* __restrict__ lok, float* __restrict__ hik, float* __restrict__ scores)
{
    extern __shared__ float m_s[];   // [C]
    const int b = blockIdx.y;
    for (int c = threadIdx.x; c < C; c += blockDim.x) m_s[c] = mean32[static_cast<size_t>(b) * C + c];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float eps_scale = static_cast<float>(C / 32 + 16) * 0x1p-22f;
    for (int tk = warp; tk < kScoreTok; tk += 8) {
        const int i = blockIdx.x * kScoreTok + tk;
        if (i >= N) break;
        const uint4* row = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(b) * N + i) * C);
        float acc = 0.f, accA = 0.f;
        for (int ch = lane; ch < C / 8; ch += 32) {
            const uint4 v = __ldg(row + ch);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = __uint_as_float(w[e] << 16), x1 = __uint_as_float(w[e] & 0xFFFF0000u);
                const float m0 = m_s[ch * 8 + 2 * e], m1 = m_s[ch * 8 + 2 * e + 1];
                const float d0 = x0 - m0, d1 = x1 - m1;
                acc = fmaf(d0, d0, acc);
                acc = fmaf(d1, d1, acc);
                const float a0 = fabsf(x0) + fabsf(m0), a1 = fabsf(x1) + fabsf(m1);
                accA = fmaf(a0, a0, accA);
                accA = fmaf(a1, a1, accA);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
            accA += __shfl_xor_sync(0xffffffffu, accA, off);
        }
        if (lane == 0) {
            const float eps = __fmul_ru(accA, eps_scale);
            lok[static_cast<size_t>(b) * N + i] = __fsub_rd(acc, eps);
            hik[static_cast<size_t>(b) * N + i] = __fadd_ru(acc, eps);
            if (scores) scores[static_cast<size_t>(b) * N + i] = acc;
        }
    }
}

// ------------------------------------------------------------------ 4. select

// Order-preserving map float -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// K-th largest (1-based rank `rank`) of keys[0..n) by 8-bit radix select.
// All threads of the CTA call it; returns the key value.
__device__ uint32_t radix_select_desc(const uint32_t* keys, int n, int rank, int* hist, int* shared_out)
{
    uint32_t prefix = 0, mask = 0;
    int want = rank;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t k = keys[i];
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l owns digits 255-8l .. 248-8l (descending)
            const int l = threadIdx.x;
            int cnt[8];
            int tot = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                cnt[q] = hist[255 - 8 * l - q];
                tot += cnt[q];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, off);
                if (l >= off) incl += v;
            }
            const int excl = incl - tot;
            if (excl < want && want <= incl) {
                int run = excl;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (run < want && want <= run + cnt[q]) {
                        shared_out[0] = 255 - 8 * l - q;
                        shared_out[1] = want - run;
                    }
                    run += cnt[q];
                }
            }
        }
        __syncthreads();
        const uint32_t d = static_cast<uint32_t>(shared_out[0]);
        want = shared_out[1];
        prefix |= d << shift;
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    return prefix;
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

__global__ void __launch_bounds__(kSelThreads)
    pivot_select_kernel(const __nv_bfloat16* __restrict__ x, int N, int C, int K, const float* __restrict__ lok,
                        const float* __restrict__ hik, const double* __restrict__ mean64,
                        int* __restrict__ band_idx_g, double* __restrict__ band_score_g, int* __restrict__ flags_g,
                        int32_t* __restrict__ idx_out, int32_t* status)
{
    extern __shared__ uint32_t sel_smem[];
    uint32_t* klo = sel_smem;          // [N]
    uint32_t* khi = sel_smem + N;      // [N]
    __shared__ int hist[256];
    __shared__ int sh_out[2];
    __shared__ int counts[kSelThreads / 32];
    __shared__ int sh_misc[4];
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    int* flags = flags_g + static_cast<size_t>(b) * N;
    int* band_idx = band_idx_g + static_cast<size_t>(b) * N;
    double* band_score = band_score_g + static_cast<size_t>(b) * N;
    int32_t* out = idx_out + static_cast<size_t>(b) * K;

    if (K == 0) return;
    for (int i = tid; i < N; i += blockDim.x) {
        klo[i] = f32_key(lok[static_cast<size_t>(b) * N + i]);
        khi[i] = f32_key(hik[static_cast<size_t>(b) * N + i]);
    }
    __syncthreads();
    const uint32_t t_lo = radix_select_desc(klo, N, K, hist, sh_out);
    const uint32_t t_hi = (K < N) ? radix_select_desc(khi, N, K + 1, hist, sh_out) : 0u;

    // classify: 1 = certainly kept, 2 = band, 0 = certainly dropped
    for (int i = tid; i < N; i += blockDim.x) {
        int f;
        if (K == N || klo[i] > t_hi) f = 1;
        else if (khi[i] < t_lo) f = 0;
        else f = 2;
        flags[i] = f;
    }
    __syncthreads();

    // ordered compaction helpers: each thread owns a contiguous chunk of i
    const int chunk = (N + blockDim.x - 1) / blockDim.x;
    const int i0 = min(N, tid * chunk), i1 = min(N, i0 + chunk);
    auto block_excl_scan = [&](int v, int* total) -> int {
        const int lane = tid & 31, warp = tid >> 5;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += u;
        }
        if (lane == 31) counts[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = lane < kSelThreads / 32 ? counts[lane] : 0;
            int wi = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += u;
            }
            if (lane < kSelThreads / 32) counts[lane] = wi - w;
            if (lane == 31) sh_misc[3] = wi;
        }
        __syncthreads();
        const int r = counts[warp] + incl - v;
        *total = sh_misc[3];
        __syncthreads();
        return r;
    };

    int n_in = 0, n_band = 0;
    for (int i = i0; i < i1; ++i) {
        n_in += flags[i] == 1;
        n_band += flags[i] == 2;
    }
    int tot_in, tot_band;
    const int pos_in = block_excl_scan(n_in, &tot_in);
    (void)pos_in;
    const int pos_band = block_excl_scan(n_band, &tot_band);
    {
        int p = pos_band;
        for (int i = i0; i < i1; ++i)
            if (flags[i] == 2) band_idx[p++] = i;
    }
    const int need = K - tot_in;
    if (need < 0 || need > tot_band) {
        if (tid == 0) atomicCAS(status, 0, VAR_ERR_NUMERIC);
        return;
    }
    __syncthreads();

    if (need > 0 && need < tot_band) {
        // fp64 re-score of the band, one warp per token
        const int warp = tid >> 5, lane = tid & 31;
        const int q = C / 32;
        const double* mb = mean64 + static_cast<size_t>(b) * C;
        for (int j = warp; j < tot_band; j += kSelThreads / 32) {
            const int i = band_idx[j];
            const __nv_bfloat16* row = x + (static_cast<size_t>(b) * N + i) * C;
            double v = tree64(row + lane * q, mb + lane * q, q);
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) v = __dadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0) band_score[j] = v;
        }
        __syncthreads();
        // rank inside the band by (score desc, index asc); keep the first `need`
        for (int j = tid; j < tot_band; j += blockDim.x) {
            const double sj = band_score[j];
            const int ij = band_idx[j];
            int better = 0;
            for (int t = 0; t < tot_band && better < need; ++t) {
                const double st = band_score[t];
                better += (st > sj) || (st == sj && band_idx[t] < ij);
            }
            flags[ij] = better < need ? 1 : 0;
        }
    } else {
        for (int j = tid; j < tot_band; j += blockDim.x) flags[band_idx[j]] = need > 0 ? 1 : 0;
    }
    __syncthreads();

    int n_sel = 0;
    for (int i = i0; i < i1; ++i) n_sel += flags[i] == 1;
    int tot_sel;
    int p = block_excl_scan(n_sel, &tot_sel);
    for (int i = i0; i < i1; ++i)
        if (flags[i] == 1 && p < K) out[p++] = i;
    if (tid == 0 && tot_sel != K) atomicCAS(status, 0, VAR_ERR_NUMERIC);
}

}  // namespace

size_t pivot_workspace_bytes(int B, int N, int C) { return pivot_ws_layout(B, N, C).total; }

int launch_pivot_select(int B, int N, int C, const void* xv, int keep_k, int32_t* idx, float* scores,
                        void* ws, size_t ws_bytes, cudaStream_t st)
{
    const PivotWs w = pivot_ws_layout(B, N, C);
    if (ws_bytes < w.total) return VAR_ERR_WORKSPACE;
    int32_t* status = device_status_ptr();
    if (!status) return VAR_ERR_CUDA;
    auto* base = static_cast<uint8_t*>(ws);
    auto* hi = reinterpret_cast<long long*>(base + w.hi);
    auto* lo = reinterpret_cast<long long*>(base + w.lo);
    auto* m64 = reinterpret_cast<double*>(base + w.mean64);
    auto* m32 = reinterpret_cast<float*>(base + w.mean32);
    auto* lok = reinterpret_cast<float*>(base + w.lok);
    auto* hik = reinterpret_cast<float*>(base + w.hik);
    auto* bidx = reinterpret_cast<int*>(base + w.band_idx);
    auto* bsc = reinterpret_cast<double*>(base + w.band_score);
    auto* flg = reinterpret_cast<int*>(base + w.flags);
    const auto* x = static_cast<const __nv_bfloat16*>(xv);

    if (cudaMemsetAsync(base + w.hi, 0, w.mean64 - w.hi, st) != cudaSuccess) return VAR_ERR_CUDA;
    {
        const dim3 grid((C + 255) / 256, (N + kColRows - 1) / kColRows, B);
        pivot_colsum_kernel<<<grid, 256, 0, st>>>(x, N, C, hi, lo, status);
    }
    pivot_finalize_kernel<<<(B * C + 255) / 256, 256, 0, st>>>(hi, lo, B * C, N, m64, m32);
    {
        const size_t smem = sizeof(float) * C;
        static bool attr = false;
        if (!attr) {
            if (cudaFuncSetAttribute(pivot_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     64 * 1024) != cudaSuccess)
                return VAR_ERR_CUDA;
            attr = true;
        }
        const dim3 grid((N + kScoreTok - 1) / kScoreTok, B);
        pivot_score_kernel<<<grid, 256, smem, st>>>(x, N, C, m32, lok, hik, scores);
    }
    if (keep_k > 0) {
        const size_t smem = sizeof(uint32_t) * 2 * N;
        static bool attr = false;
        if (!attr) {
            if (cudaFuncSetAttribute(pivot_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * 16384 * 4) != cudaSuccess)
                return VAR_ERR_CUDA;
            attr = true;
        }
        pivot_select_kernel<<<B, kSelThreads, smem, st>>>(x, N, C, keep_k, lok, hik, m64, bidx, bsc, flg,
                                                          idx, status);
    }
    return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  Some callers cannot allocate device memory at the
// point where they select pivots: an engine that hands out all device memory
// itself and gives a plug-in no workspace, or a latency-critical stream where
// cudaMalloc (which may synchronise the device) is not allowed after start-up.
// For them the workspace lives in this file-scope array instead, sized for
// B <= 4, N <= 16384, C <= 4096 (about 1.9 MB).  Every GPU that loads the
// library holds it until the process exits.

constexpr int kNoAllocMaxB = 4;
constexpr int kNoAllocMaxN = 16384;
constexpr int kNoAllocMaxC = 4096;

constexpr size_t noalloc_align(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kNoAllocBytes =
    noalloc_align(sizeof(long long) * kNoAllocMaxB * kNoAllocMaxC) * 2 +   // hi, lo
    noalloc_align(sizeof(double) * kNoAllocMaxB * kNoAllocMaxC) +          // mean64
    noalloc_align(sizeof(float) * kNoAllocMaxB * kNoAllocMaxC) +           // mean32
    noalloc_align(sizeof(float) * kNoAllocMaxB * kNoAllocMaxN) * 2 +       // lo/hi keys
    noalloc_align(sizeof(int) * kNoAllocMaxB * kNoAllocMaxN) +             // band indices
    noalloc_align(sizeof(double) * kNoAllocMaxB * kNoAllocMaxN) +          // band scores
    noalloc_align(sizeof(int) * kNoAllocMaxB * kNoAllocMaxN);              // flags

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
    // launch_pivot_select clears the accumulators it needs zeroed (cudaMemsetAsync,
    // no allocation); everything else in the scratch is written before it is read.
    return launch_pivot_select(B, N, channels, x, keep_k, idx, scores, ws, kNoAllocBytes,
                               static_cast<cudaStream_t>(stream));
}
