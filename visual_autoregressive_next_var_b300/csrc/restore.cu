// Structural reconstruction for sm_103a ("ARVAR" Key Design 3, Eq. (8)-(9)):
//   out = Scatter(Up(prev; s, s), idx, o_compact)
// Up is bilinear with half-pixel centres and edge clamp; the scatter overwrites
// the kept rows.
//
// Scatter mode: restore_rows_kernel, one 256-thread CTA per output grid row y
// and (b, h).  One thread issues two bulk copies (cp.async.bulk, completion on
// an mbarrier) of the source rows y0, y1 of prev (2 x s' tokens, contiguous)
// into shared memory.  Meanwhile the CTA finds the kept tokens of row y: index
// lists of up to 4,096 entries are read whole (each thread keeps four loads in
// flight, the first issued before the CTA fills its per-token tap tables; an
// entry in row y marks its token and joins the row's kept list), longer ones by
// two 32-ary searches for the row's slice.  Then the warps split: four copy the
// kept tokens' rows of o_compact (they need no source row, two loads in flight
// per thread) while the other four blend every other token from four staged
// taps once the source rows have landed.  Every row of out is written once,
// with 16-byte stores.
//
// Fill mode (var_restore_fill, var_pruned_in_place: the in-place pruned
// attention writes the kept rows, maybe concurrently, so they must not be
// touched): the same kernel with every warp blending and no kept copies.  In
// var_pruned_in_place it is launched as a programmatic dependent of that
// call's attention, which lets it start at once: its CTAs take the SMs the
// attention leaves free, and one thread of CTA 0 waits for the attention
// before its CTA exits, so the grid completes after it.
#include "internal.h"
#include "ptx.cuh"

namespace varattn {

namespace {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Source coordinate of output pixel d of an axis from an n_in-wide one
// (half-pixel centres, clamped to 0; ratio = n_in / n_out): taps i0, i1 and
// the weight of i1.
__device__ __forceinline__ void axis_taps(int d, float ratio, int n_in, int& i0, int& i1, float& w1)
{
    const float src = fmaxf((static_cast<float>(d) + 0.5f) * ratio - 0.5f, 0.f);
    i0 = min(static_cast<int>(src), n_in - 1);
    i1 = min(i0 + 1, n_in - 1);
    w1 = src - static_cast<float>(i0);
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// bilinear blend of four 16-byte groups (8 bf16 each), two elements per
// packed f32x2 operation
__device__ __forceinline__ uint4 blend4(const uint4& a, const uint4& b, const uint4& c, const uint4& d, float w00,
                                        float w01, float w10, float w11)
{
    const uint32_t* A = &a.x;
    const uint32_t* Bw = &b.x;
    const uint32_t* Cw = &c.x;
    const uint32_t* Dw = &d.x;
    const uint64_t W00 = f2_pack(w00, w00), W01 = f2_pack(w01, w01), W10 = f2_pack(w10, w10),
                   W11 = f2_pack(w11, w11);
    uint4 r;
    uint32_t* R = &r.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        uint64_t t = f2_mul(W00, f2_pack(bf_lo(A[e]), bf_hi(A[e])));
        t = f2_fma(W01, f2_pack(bf_lo(Bw[e]), bf_hi(Bw[e])), t);
        t = f2_fma(W10, f2_pack(bf_lo(Cw[e]), bf_hi(Cw[e])), t);
        t = f2_fma(W11, f2_pack(bf_lo(Dw[e]), bf_hi(Dw[e])), t);
        float lo, hi;
        f2_unpack(t, lo, hi);
        R[e] = pack_bf16x2(lo, hi);
    }
    return r;
}

// ------------------------------------------------------------------ index search

// First index of a[0, n) (ascending) whose value is >= key; every lane of the
// warp calls it and gets the result.
__device__ __forceinline__ int warp_lower_bound(const int32_t* a, int n, int key)
{
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = n;                    // the answer lies in [lo, hi]
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) >> 5;
        const int i = lo + (lane + 1) * step - 1;
        const bool below = i < hi && __ldg(a + i) < key;
        const int c = __popc(__ballot_sync(0xffffffffu, below));
        const int ic = lo + (c + 1) * step - 1;
        lo += c * step;
        if (c < 32 && ic < hi) hi = ic;
    }
    const int i = lo + lane;
    const bool below = i < hi && __ldg(a + i) < key;
    return lo + __popc(__ballot_sync(0xffffffffu, below));
}

// ------------------------------------------------------------------ row kernel

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

constexpr int kScanMax = 4096;   // index lists up to this length are read whole by every CTA

constexpr int kRowThreads = 256;
constexpr int kKeptWarps = 4;    // warps that copy the kept tokens; the other four blend
constexpr int kIdxBatch = 4;     // index entries each thread has in flight
constexpr int kKeptBatch = 2;    // compact-row loads each kept-copy thread has in flight

template <int D, bool FILL>
__global__ void __launch_bounds__(kRowThreads)
    restore_rows_kernel(const __nv_bfloat16* __restrict__ prev, const __nv_bfloat16* __restrict__ oc,
                        const int32_t* __restrict__ idx, int keep_k, __nv_bfloat16* __restrict__ out, int H, int sp,
                        int s, float ratio, int32_t* status)
{
    constexpr int LPT = D / 8;
    // fill mode: the kept rows are not this kernel's (the in-place attention
    // writes them), every warp blends
    constexpr int KW = FILL ? 0 : kKeptWarps;
    // [2][sp][LPT] source rows y0, y1; then per token x of the row: the four
    // tap weights, its two source columns (times LPT), an entry of the kept
    // list (token, compact row) and its compact row or -1
    extern __shared__ __align__(128) uint4 stage[];
    __shared__ __align__(8) uint64_t full;
    __shared__ int range[2], nkept;
    const int y = blockIdx.x, bh = blockIdx.y, b = bh / H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_row = sp * LPT;
    float4* tw = reinterpret_cast<float4*>(stage + 2 * per_row);
    int2* toff = reinterpret_cast<int2*>(tw + s);
    int2* klist = toff + s;
    int* slot = reinterpret_cast<int*>(klist + s);
    int y0, y1;
    float ly;
    axis_taps(y, ratio, sp, y0, y1, ly);
    const uint4* P = reinterpret_cast<const uint4*>(prev + static_cast<size_t>(bh) * sp * sp * D);
    const uint32_t bar = smem_u32(&full);
    const uint32_t row_bytes = static_cast<uint32_t>(per_row) * 16u;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, (y1 != y0 ? 2u : 1u) * row_bytes);
        bulk_g2s(smem_u32(stage), P + static_cast<size_t>(y0) * per_row, row_bytes, bar);
        if (y1 != y0) bulk_g2s(smem_u32(stage + per_row), P + static_cast<size_t>(y1) * per_row, row_bytes, bar);
        nkept = 0;
    }
    const int32_t* ib = idx + static_cast<size_t>(b) * keep_k;
    const int lo = y * s;
    // the first entries of a whole-list read are in flight while the tables fill
    int tk[kIdxBatch];
#pragma unroll
    for (int i = 0; i < kIdxBatch; ++i) {
        const int j = i * kRowThreads + threadIdx.x;
        tk[i] = (keep_k <= kScanMax && j < keep_k) ? __ldg(ib + j) - lo : -1;
    }
    for (int x = threadIdx.x; x < s; x += blockDim.x) {
        slot[x] = -1;
        int x0, x1;
        float lx;
        axis_taps(x, ratio, sp, x0, x1, lx);
        tw[x] = make_float4((1.f - ly) * (1.f - lx), (1.f - ly) * lx, ly * (1.f - lx), ly * lx);
        toff[x] = make_int2(x0 * LPT, x1 * LPT);
    }
    if (keep_k > kScanMax && warp < 2) {
        const int r = warp_lower_bound(ib, keep_k, lo + warp * s);
        if (lane == 0) range[warp] = r;
    }
    __syncthreads();
    // token t of the row is kept as compact row j (at most s entries are listed:
    // more only for a list that is not strictly ascending)
    auto mark = [&](int t, int j) {
        slot[t] = j;
        if (FILL) return;
        const int n = atomicAdd(&nkept, 1);
        if (n < s) klist[n] = make_int2(t, j);
    };
    if (keep_k <= kScanMax) {
#pragma unroll
        for (int i = 0; i < kIdxBatch; ++i)
            if (tk[i] >= 0 && tk[i] < s) mark(tk[i], i * kRowThreads + threadIdx.x);
        for (int j0 = kIdxBatch * kRowThreads; j0 < keep_k; j0 += kIdxBatch * kRowThreads) {
#pragma unroll
            for (int i = 0; i < kIdxBatch; ++i) {
                const int j = j0 + i * kRowThreads + threadIdx.x;
                tk[i] = j < keep_k ? __ldg(ib + j) - lo : -1;
            }
#pragma unroll
            for (int i = 0; i < kIdxBatch; ++i)
                if (tk[i] >= 0 && tk[i] < s) mark(tk[i], j0 + i * kRowThreads + threadIdx.x);
        }
    } else {
        const int j0 = range[0], nk = min(range[1] - range[0], s);
        if (threadIdx.x == 0 && range[1] - range[0] > s) atomicCAS(status, 0, VAR_ERR_INVALID_ARG);
        for (int t = threadIdx.x; t < nk; t += blockDim.x) {
            const int x = __ldg(ib + j0 + t) - lo;
            if (x >= 0 && x < s) mark(x, j0 + t);
        }
    }
    __syncthreads();
    uint4* O = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * s * s + static_cast<size_t>(lo)) * D);
    const uint4* Cb = reinterpret_cast<const uint4*>(oc + static_cast<size_t>(bh) * keep_k * D);
    if (warp < KW) {
        // kept tokens: copies of their compact rows, which need no source row
        const int nk = min(nkept, s);
        for (int k0 = threadIdx.x; k0 < nk * LPT; k0 += kKeptBatch * 32 * KW) {
            uint4 v[kKeptBatch];
            unsigned got = 0;
#pragma unroll
            for (int i = 0; i < kKeptBatch; ++i) {
                const int k = k0 + i * 32 * KW;
                if (k < nk * LPT) {
                    const int item = k / LPT, part = k - item * LPT;
                    v[i] = __ldg(Cb + static_cast<size_t>(klist[item].y) * LPT + part);
                    got |= 1u << i;
                }
            }
#pragma unroll
            for (int i = 0; i < kKeptBatch; ++i)
                if (got >> i & 1u) {
                    const int k = k0 + i * 32 * KW;
                    const int item = k / LPT, part = k - item * LPT;
                    O[klist[item].x * LPT + part] = v[i];
                }
        }
        return;
    }
    // every other token: the blend of four staged taps, once the source rows
    // landed (a run-time stride: unrolling this loop measured slower)
    if (!mbar_wait(bar, 0, nullptr)) {
        if (threadIdx.x == 32 * KW) atomicCAS(status, 0, VAR_ERR_TIMEOUT);
        mbar_wait(bar, 0, nullptr);          // the copy must land before the CTA leaves
        return;
    }
    const uint4* S1 = stage + (y1 != y0 ? per_row : 0);
    for (int e = threadIdx.x - 32 * KW; e < s * LPT; e += blockDim.x - 32 * KW) {
        const int x = e / LPT, part = e - x * LPT;
        if (slot[x] >= 0) continue;
        const int2 o = toff[x];
        const float4 w = tw[x];
        O[e] = blend4(stage[o.x + part], stage[o.y + part], S1[o.x + part], S1[o.y + part], w.x, w.y, w.z, w.w);
    }
    // a fill launched beside the in-place attention (programmatic dependent)
    // completes only after it, so later work on the stream sees both
    if (FILL && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) pdl_wait();
}

template <int D>
int launch_restore_d(int B, int H, int sp, int s, const __nv_bfloat16* P, const __nv_bfloat16* C,
                     const int32_t* idx, int keep_k, __nv_bfloat16* O, cudaStream_t st, int32_t* status,
                     bool fill_only, bool beside)
{
    constexpr int LPT = D / 8;
    const float ratio = static_cast<float>(sp) / static_cast<float>(s);
    const size_t smem = 2ull * sp * LPT * sizeof(uint4) + (sizeof(float4) + 2 * sizeof(int2) + sizeof(int)) * s;
    if (smem > 200 * 1024) return VAR_ERR_UNSUPPORTED;
    auto kern = fill_only ? restore_rows_kernel<D, true> : restore_rows_kernel<D, false>;
    // eight CTAs per SM (about 27 KB each at 48x48 -> 64x64) need the largest carveout
    if (ensure_smem_attr(kern, static_cast<int>(smem), true) != cudaSuccess) return VAR_ERR_CUDA;
    return cuda_status(launch_kernel(kern, dim3(s, B * H), dim3(kRowThreads), smem, st, fill_only && beside, P,
                                     fill_only ? nullptr : C, idx, keep_k, O, H, sp, s, ratio, status));
}

}  // namespace

int launch_restore_scatter(int B, int H, int D, int sp, int s, const void* prev, const void* oc,
                           const int32_t* idx, int keep_k, void* out, cudaStream_t st, int32_t* status,
                           bool fill_only, bool beside)
{
    if (B * H > 65535) return VAR_ERR_UNSUPPORTED;
    auto* P = static_cast<const __nv_bfloat16*>(prev);
    auto* C = static_cast<const __nv_bfloat16*>(oc);
    auto* O = static_cast<__nv_bfloat16*>(out);
    if (D == 128) return launch_restore_d<128>(B, H, sp, s, P, C, idx, keep_k, O, st, status, fill_only, beside);
    if (D == 64) return launch_restore_d<64>(B, H, sp, s, P, C, idx, keep_k, O, st, status, fill_only, beside);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
