// Structural reconstruction for sm_103a ("ARVAR" Key Design 3, Eq. (8)-(9)):
//   out = Scatter(Up(prev; s, s), idx, o_compact)
// In fill mode the kept rows are left as they are (the pruned attention has
// written them in place) and only the upsampled rows are written.
// Up is bilinear with half-pixel centres and edge clamp; the scatter overwrites
// the kept rows.  One pass: every output row is written exactly once, either
// copied from o_compact (kept token) or blended from four rows of prev.
//
// Grid: (token chunks of TOK, B*H).  A chunk's kept rows are found by two
// binary searches in the ascending index list and mapped in shared memory.
// D/8 lanes handle one token row with 16-byte loads and stores.
#include "internal.h"
#include "ptx.cuh"

namespace varattn {

constexpr int kRestoreTok = 64;

__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int n, int key)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a + mid) < key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D>
__global__ void __launch_bounds__(256)
    restore_scatter_kernel(const __nv_bfloat16* __restrict__ prev, const __nv_bfloat16* __restrict__ oc,
                           const int32_t* __restrict__ idx, int keep_k, __nv_bfloat16* __restrict__ out,
                           int H, int sp, int s, float ratio, int fill_only)
{
    constexpr int LPT = D / 8;            // lanes per token row (16 B each)
    constexpr int TPW = 32 / LPT;         // token rows per warp step
    __shared__ int inv[kRestoreTok];
    __shared__ int range[2];
    const int N = s * s;
    const int bh = blockIdx.y;
    const int b = bh / H;
    const int n0 = blockIdx.x * kRestoreTok;
    const int n1 = min(N, n0 + kRestoreTok);
    const int32_t* ib = idx + static_cast<size_t>(b) * keep_k;

    if (threadIdx.x < kRestoreTok) inv[threadIdx.x] = -1;
    if (threadIdx.x == 0) range[0] = keep_k ? lower_bound_i32(ib, keep_k, n0) : 0;
    if (threadIdx.x == 32) range[1] = keep_k ? lower_bound_i32(ib, keep_k, n1) : 0;
    __syncthreads();
    for (int j = range[0] + threadIdx.x; j < range[1]; j += blockDim.x) {
        const int t = __ldg(ib + j) - n0;   // in [0, n1-n0) for an ascending list
        if (t >= 0 && t < kRestoreTok) inv[t] = j;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPT, part = lane % LPT;
    const int Np = sp * sp;
    const uint4* P = reinterpret_cast<const uint4*>(prev + static_cast<size_t>(bh) * Np * D);
    const uint4* C = reinterpret_cast<const uint4*>(oc + static_cast<size_t>(bh) * keep_k * D);
    uint4* O = reinterpret_cast<uint4*>(out + static_cast<size_t>(bh) * N * D);
    for (int n = n0 + warp * TPW + sub; n < n1; n += 8 * TPW) {
        const int j = inv[n - n0];
        uint4 r;
        if (j >= 0) {
            if (fill_only) continue;
            r = __ldg(C + static_cast<size_t>(j) * LPT + part);
        } else {
            const int y = n / s, x = n - y * s;
            const float sy = fmaxf((static_cast<float>(y) + 0.5f) * ratio - 0.5f, 0.f);
            const float sx = fmaxf((static_cast<float>(x) + 0.5f) * ratio - 0.5f, 0.f);
            const int y0 = min(static_cast<int>(sy), sp - 1), x0 = min(static_cast<int>(sx), sp - 1);
            const int y1 = min(y0 + 1, sp - 1), x1 = min(x0 + 1, sp - 1);
            const float ly = sy - static_cast<float>(y0), lx = sx - static_cast<float>(x0);
            const float w00 = (1.f - ly) * (1.f - lx), w01 = (1.f - ly) * lx;
            const float w10 = ly * (1.f - lx), w11 = ly * lx;
            const uint4 a = __ldg(P + static_cast<size_t>(y0 * sp + x0) * LPT + part);
            const uint4 bq = __ldg(P + static_cast<size_t>(y0 * sp + x1) * LPT + part);
            const uint4 c = __ldg(P + static_cast<size_t>(y1 * sp + x0) * LPT + part);
            const uint4 d = __ldg(P + static_cast<size_t>(y1 * sp + x1) * LPT + part);
            const uint32_t* A = &a.x;
            const uint32_t* Bw = &bq.x;
            const uint32_t* Cw = &c.x;
            const uint32_t* Dw = &d.x;
            uint32_t* R = &r.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = w00 * bf_lo(A[e]) + w01 * bf_lo(Bw[e]) + w10 * bf_lo(Cw[e]) + w11 * bf_lo(Dw[e]);
                const float hi = w00 * bf_hi(A[e]) + w01 * bf_hi(Bw[e]) + w10 * bf_hi(Cw[e]) + w11 * bf_hi(Dw[e]);
                R[e] = pack_bf16x2(lo, hi);
            }
        }
        O[static_cast<size_t>(n) * LPT + part] = r;
    }
}

int launch_restore_scatter(int B, int H, int D, int sp, int s, const void* prev, const void* oc,
                           const int32_t* idx, int keep_k, void* out, cudaStream_t st, int32_t* status,
                           bool fill_only)
{
    (void)status;
    const int N = s * s;
    const dim3 grid((N + kRestoreTok - 1) / kRestoreTok, B * H);
    if (B * H > 65535) return VAR_ERR_UNSUPPORTED;
    const float ratio = static_cast<float>(sp) / static_cast<float>(s);
    auto* P = static_cast<const __nv_bfloat16*>(prev);
    auto* C = static_cast<const __nv_bfloat16*>(oc);
    auto* O = static_cast<__nv_bfloat16*>(out);
    const int fill = fill_only ? 1 : 0;
    if (D == 128)
        return cuda_status(launch_kernel(restore_scatter_kernel<128>, grid, dim3(256), 0, st, false, P, C, idx, keep_k,
                                         O, H, sp, s, ratio, fill));
    if (D == 64)
        return cuda_status(launch_kernel(restore_scatter_kernel<64>, grid, dim3(256), 0, st, false, P, C, idx, keep_k,
                                         O, H, sp, s, ratio, fill));
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
