// Structural reconstruction for sm_103a ("ARVAR" Key Design 3, Eq. (8)-(9)):
//   out = Scatter(Up(prev; s, s), idx, o_compact)
// Up is bilinear with half-pixel centres and edge clamp; the scatter overwrites
// the kept rows.
//
// Scatter mode: restore_rows_kernel, one CTA per output grid row y and (b, h).
// The two source rows y0, y1 of prev (2 x s' tokens) are staged in shared
// memory with cp.async; while they are in flight two warps find the slice of
// the ascending index list that falls in row y (32-ary searches: all lanes
// probe at once, one load round per factor of 32 of the list's length) and the
// kept rows of o_compact named by the slice are staged too.  Every output
// token of the row is then either its staged o_compact row (kept) or a blend of
// four staged taps, written with 16-byte stores: each row of out written once.
//
// Fill mode (the kept rows are written by the in-place pruned attention, maybe
// concurrently, so they must not be touched): fill_rows_kernel, one CTA per 64
// tokens of a (b, h); two warps find the chunk's slice of the ascending index
// list with 32-ary searches (all lanes probing at once, one load round per
// factor of 32 of the list's length), the slice is marked in shared memory,
// and the other tokens are blended from prev.
#include "internal.h"
#include "ptx.cuh"

namespace varattn {

namespace {

constexpr int kFillTok = 64;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}


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

// bilinear blend of four 16-byte groups (8 bf16 each)
__device__ __forceinline__ uint4 blend4(const uint4& a, const uint4& b, const uint4& c, const uint4& d, float w00,
                                        float w01, float w10, float w11)
{
    const uint32_t* A = &a.x;
    const uint32_t* Bw = &b.x;
    const uint32_t* Cw = &c.x;
    const uint32_t* Dw = &d.x;
    uint4 r;
    uint32_t* R = &r.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float lo = w00 * bf_lo(A[e]) + w01 * bf_lo(Bw[e]) + w10 * bf_lo(Cw[e]) + w11 * bf_lo(Dw[e]);
        const float hi = w00 * bf_hi(A[e]) + w01 * bf_hi(Bw[e]) + w10 * bf_hi(Cw[e]) + w11 * bf_hi(Dw[e]);
        R[e] = pack_bf16x2(lo, hi);
    }
    return r;
}

// ------------------------------------------------------------------ fill mode

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

// ------------------------------------------------------------------ scatter mode

template <int D>
__global__ void __launch_bounds__(256)
    restore_rows_kernel(const __nv_bfloat16* __restrict__ prev, const __nv_bfloat16* __restrict__ oc,
                        const int32_t* __restrict__ idx, int keep_k, __nv_bfloat16* __restrict__ out, int H, int sp,
                        int s, float ratio, int32_t* status)
{
    constexpr int LPT = D / 8;              // 16-byte groups per token row
    // [2][sp][LPT] source rows y0, y1, then [s][LPT] kept rows of o_compact, then [s] int
    extern __shared__ __align__(16) uint4 stage[];
    __shared__ int range[2];
    const int y = blockIdx.x, bh = blockIdx.y, b = bh / H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_row = sp * LPT;
    uint4* kst = stage + 2 * per_row;
    int* slot = reinterpret_cast<int*>(kst + s * LPT);   // token x -> staged kept row, or -1
    int y0, y1;
    float ly;
    axis_taps(y, ratio, sp, y0, y1, ly);
    const uint4* P = reinterpret_cast<const uint4*>(prev + static_cast<size_t>(bh) * sp * sp * D);
    for (int e = threadIdx.x; e < 2 * per_row; e += blockDim.x) {
        const int r = e / per_row, o = e - r * per_row;
        cp_async16(smem_u32(stage + e), P + static_cast<size_t>(r ? y1 : y0) * per_row + o);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int x = threadIdx.x; x < s; x += blockDim.x) slot[x] = -1;
    const int32_t* ib = idx + static_cast<size_t>(b) * keep_k;
    if (warp < 2) {
        const int r = keep_k ? warp_lower_bound(ib, keep_k, (y + warp) * s) : 0;
        if (lane == 0) range[warp] = r;
    }
    __syncthreads();
    // kept tokens of this row: idx[j0, j0 + nk); more than s means the list is
    // not strictly ascending (reported, and cut to the row's s tokens)
    const int j0 = range[0], nk = min(range[1] - range[0], s);
    if (threadIdx.x == 0 && range[1] - range[0] > s) atomicCAS(status, 0, VAR_ERR_INVALID_ARG);
    for (int t = threadIdx.x; t < nk; t += blockDim.x) {
        const int x = __ldg(ib + j0 + t) - y * s;          // in [0, s) for an ascending list
        if (x >= 0 && x < s) slot[x] = t;
    }
    const uint4* Cp = reinterpret_cast<const uint4*>(oc + (static_cast<size_t>(bh) * keep_k + j0) * D);
    for (int e = threadIdx.x; e < nk * LPT; e += blockDim.x) cp_async16(smem_u32(kst + e), Cp + e);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    uint4* O = reinterpret_cast<uint4*>(out + (static_cast<size_t>(bh) * s * s + static_cast<size_t>(y) * s) * D);
    for (int e = threadIdx.x; e < s * LPT; e += blockDim.x) {
        const int x = e / LPT, part = e - x * LPT;
        const int t = slot[x];
        if (t >= 0) {
            O[e] = kst[t * LPT + part];
        } else {
            int x0, x1;
            float lx;
            axis_taps(x, ratio, sp, x0, x1, lx);
            const float w00 = (1.f - ly) * (1.f - lx), w01 = (1.f - ly) * lx;
            const float w10 = ly * (1.f - lx), w11 = ly * lx;
            O[e] = blend4(stage[x0 * LPT + part], stage[x1 * LPT + part], stage[per_row + x0 * LPT + part],
                          stage[per_row + x1 * LPT + part], w00, w01, w10, w11);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256)
    fill_rows_kernel(const __nv_bfloat16* __restrict__ prev, const int32_t* __restrict__ idx, int keep_k,
                     __nv_bfloat16* __restrict__ out, int H, int sp, int s, float ratio)
{
    constexpr int LPT = D / 8;            // lanes per token row (16 B each)
    constexpr int TPW = 32 / LPT;         // token rows per warp step
    __shared__ uint8_t kept[kFillTok];
    __shared__ int range[2];
    const int N = s * s;
    const int bh = blockIdx.y;
    const int b = bh / H;
    const int n0 = blockIdx.x * kFillTok;
    const int n1 = min(N, n0 + kFillTok);
    const int32_t* ib = idx + static_cast<size_t>(b) * keep_k;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x < kFillTok) kept[threadIdx.x] = 0;
    if (warp < 2) {
        const int r = keep_k ? warp_lower_bound(ib, keep_k, warp ? n1 : n0) : 0;
        if (lane == 0) range[warp] = r;
    }
    __syncthreads();
    for (int j = range[0] + threadIdx.x; j < range[1]; j += blockDim.x) {
        const int t = __ldg(ib + j) - n0;   // in [0, n1-n0) for an ascending list
        if (t >= 0 && t < kFillTok) kept[t] = 1;
    }
    __syncthreads();

    const int sub = lane / LPT, part = lane % LPT;
    const uint4* P = reinterpret_cast<const uint4*>(prev + static_cast<size_t>(bh) * sp * sp * D);
    uint4* O = reinterpret_cast<uint4*>(out + static_cast<size_t>(bh) * N * D);
    for (int n = n0 + warp * TPW + sub; n < n1; n += 8 * TPW) {
        if (kept[n - n0]) continue;
        const int y = n / s, x = n - y * s;
        int y0, y1, x0, x1;
        float ly, lx;
        axis_taps(y, ratio, sp, y0, y1, ly);
        axis_taps(x, ratio, sp, x0, x1, lx);
        const uint4 a = __ldg(P + static_cast<size_t>(y0 * sp + x0) * LPT + part);
        const uint4 bq = __ldg(P + static_cast<size_t>(y0 * sp + x1) * LPT + part);
        const uint4 c = __ldg(P + static_cast<size_t>(y1 * sp + x0) * LPT + part);
        const uint4 d = __ldg(P + static_cast<size_t>(y1 * sp + x1) * LPT + part);
        O[static_cast<size_t>(n) * LPT + part] = blend4(a, bq, c, d, (1.f - ly) * (1.f - lx), (1.f - ly) * lx,
                                                        ly * (1.f - lx), ly * lx);
    }
}

template <int D>
int launch_restore_d(int B, int H, int sp, int s, const __nv_bfloat16* P, const __nv_bfloat16* C,
                     const int32_t* idx, int keep_k, __nv_bfloat16* O, cudaStream_t st, int32_t* status,
                     bool fill_only)
{
    constexpr int LPT = D / 8;
    const int N = s * s;
    const float ratio = static_cast<float>(sp) / static_cast<float>(s);
    if (fill_only) {
        const dim3 grid((N + kFillTok - 1) / kFillTok, B * H);
        return cuda_status(launch_kernel(fill_rows_kernel<D>, grid, dim3(256), 0, st, false, P, idx, keep_k, O, H,
                                         sp, s, ratio));
    }
    const size_t smem = (2ull * sp + s) * LPT * sizeof(uint4) + sizeof(int) * s;
    if (smem > 200 * 1024) return VAR_ERR_UNSUPPORTED;
    if (ensure_smem_attr(restore_rows_kernel<D>, static_cast<int>(smem)) != cudaSuccess) return VAR_ERR_CUDA;
    return cuda_status(launch_kernel(restore_rows_kernel<D>, dim3(s, B * H), dim3(256), smem, st, false, P, C, idx,
                                     keep_k, O, H, sp, s, ratio, status));
}

}  // namespace

int launch_restore_scatter(int B, int H, int D, int sp, int s, const void* prev, const void* oc,
                           const int32_t* idx, int keep_k, void* out, cudaStream_t st, int32_t* status,
                           bool fill_only)
{
    if (B * H > 65535) return VAR_ERR_UNSUPPORTED;
    auto* P = static_cast<const __nv_bfloat16*>(prev);
    auto* C = static_cast<const __nv_bfloat16*>(oc);
    auto* O = static_cast<__nv_bfloat16*>(out);
    if (D == 128) return launch_restore_d<128>(B, H, sp, s, P, C, idx, keep_k, O, st, status, fill_only);
    if (D == 64) return launch_restore_d<64>(B, H, sp, s, P, C, idx, keep_k, O, st, status, fill_only);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
