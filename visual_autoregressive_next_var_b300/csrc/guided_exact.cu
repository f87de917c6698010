// Attention-guided pivot selection decided in fp64 ("ARVAR" Key Design 2:
// attention retrospect).  The fast path (saliency.cu) ranks positions by
// fp32 values, so near-ties at the K-th value may fall either way compared
// with the fp64 definition; this path evaluates the definition itself in fp64
// on the device, in its own order, and ranks on those values:
//
//   row_stats_kernel   per (b, h) and source query i: s_j = (q_i . k_j
//                      summed over channels in order) * scale for the L'
//                      keys, mx = max_j s_j, l = sum_j exp(s_j - mx) added
//                      in key order.
//   saliency_kernel    per (b, h) and source token j: sal = sum_i exp(s_ij -
//                      mx_i) / l_i added in query order (s_ij with key
//                      L' - N' + j, the source step's own scale).
//   topk_kernel        per b: the head sum of sal added in head order,
//                      divided by H N', interpolated bilinearly (half-pixel
//                      centres, edge clamp) term by term, and the keep_k
//                      largest (equal values: lower index first) written in
//                      ascending order.
// bf16 x bf16 products are exact in fp64, so a fused multiply-add rounds as
// the definition's separate multiply and add.  Every other operation is an
// IEEE fp64 operation in the definition's order; exp is CUDA's double exp,
// which may differ from another library's in the last bit, so two values
// closer than that can still be ordered differently from a CPU evaluation.
//
// Cost: one fp64 dot product of head_dim per (query, key) pair of the source
// step, plus one per (query, self-block key) pair.  B300 runs fp64 at a small
// fraction of its fp32 rate, so this path is for callers that need the exact
// ranking, not the fast one.
#include <cuda_bf16.h>

#include "internal.h"

namespace varattn {

namespace {

constexpr int kRowWarps = 4;       // row_stats_kernel: one warp per query row
constexpr int kRowMaxKeys = 6144;  // keys whose scores a warp keeps in shared memory (48 KB)
constexpr int kSalThreads = 128;   // saliency_kernel: one thread per source token
constexpr int kSalQTile = 16;      // query rows staged per round

__device__ __forceinline__ double bf(uint32_t w, int hi)
{
    return static_cast<double>(__uint_as_float(hi ? (w & 0xFFFF0000u) : (w << 16)));
}

// q (fp64 in shared memory, D values) . k_j (bf16 row in global memory), in channel order, times scale
template <int D>
__device__ __forceinline__ double score(const double* qd, const __nv_bfloat16* kr, double scale)
{
    const uint4* k4 = reinterpret_cast<const uint4*>(kr);
    double dot = 0.0;
#pragma unroll 4
    for (int c0 = 0; c0 < D / 8; ++c0) {
        const uint4 v = __ldg(k4 + c0);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            dot = __fma_rn(qd[8 * c0 + 2 * h], bf(w[h], 0), dot);
            dot = __fma_rn(qd[8 * c0 + 2 * h + 1], bf(w[h], 1), dot);
        }
    }
    return __dmul_rn(dot, scale);
}

template <int D>
__global__ void __launch_bounds__(kRowWarps * 32)
    row_stats_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int BH, int Np,
                     int L, int cap, double scale, double* __restrict__ mx_out, double* __restrict__ l_out)
{
    extern __shared__ double shd[];                       // per warp: q[D], s[min(L, kRowMaxKeys)]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowWarps + warp;         // (b, h, i) flat
    if (row >= BH * Np) return;
    const int bh = row / Np;
    const bool keep = L <= kRowMaxKeys;
    double* qd = shd + warp * (D + (keep ? L : 0));
    double* sv = qd + D;
    for (int c = lane; c < D; c += 32) qd[c] = static_cast<double>(__bfloat162float(q[static_cast<size_t>(row) * D + c]));
    __syncwarp();
    const __nv_bfloat16* kb = k + static_cast<size_t>(bh) * cap * D;
    double mx = -INFINITY;
    for (int j = lane; j < L; j += 32) {
        const double s = score<D>(qd, kb + static_cast<size_t>(j) * D, scale);
        if (keep) sv[j] = s;
        mx = fmax(mx, s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    __syncwarp();
    double l = 0.0;
    for (int j0 = 0; j0 < L; j0 += 32) {
        const int j = j0 + lane;
        double e = 0.0;
        if (j < L) e = exp(__dsub_rn(keep ? sv[j] : score<D>(qd, kb + static_cast<size_t>(j) * D, scale), mx));
        const int n = min(32, L - j0);
        for (int t = 0; t < n; ++t) l = __dadd_rn(l, __shfl_sync(0xffffffffu, e, t));
    }
    if (lane == 0) {
        mx_out[row] = mx;
        l_out[row] = l;
    }
}

template <int D>
__global__ void __launch_bounds__(kSalThreads)
    exact_saliency_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k, int Np, int L,
                          int cap, double scale, const double* __restrict__ mx, const double* __restrict__ lsum,
                          double* __restrict__ sal)
{
    __shared__ double qt[kSalQTile][D];
    __shared__ double st[kSalQTile][2];
    const int bh = blockIdx.y;
    const int j = blockIdx.x * kSalThreads + threadIdx.x;
    const bool valid = j < Np;
    const __nv_bfloat16* kr = k + (static_cast<size_t>(bh) * cap + (L - Np) + (valid ? j : 0)) * D;
    double acc = 0.0;
    for (int i0 = 0; i0 < Np; i0 += kSalQTile) {
        const int ni = min(kSalQTile, Np - i0);
        __syncthreads();
        for (int e = threadIdx.x; e < ni * D; e += kSalThreads) {
            const int ii = e / D, c = e - ii * D;
            qt[ii][c] = static_cast<double>(__bfloat162float(q[(static_cast<size_t>(bh) * Np + i0 + ii) * D + c]));
        }
        if (threadIdx.x < ni) {
            st[threadIdx.x][0] = mx[static_cast<size_t>(bh) * Np + i0 + threadIdx.x];
            st[threadIdx.x][1] = lsum[static_cast<size_t>(bh) * Np + i0 + threadIdx.x];
        }
        __syncthreads();
        if (valid) {
            for (int ii = 0; ii < ni; ++ii) {
                const double s = score<D>(qt[ii], kr, scale);
                acc = __dadd_rn(acc, __ddiv_rn(exp(__dsub_rn(s, st[ii][0])), st[ii][1]));
            }
        }
    }
    if (valid) sal[static_cast<size_t>(bh) * Np + j] = acc;
}

// per batch element: head sum, bilinear values, exact Top-K by counting
__global__ void __launch_bounds__(1024)
    exact_topk_kernel(const double* __restrict__ sal, int H, int sp, int s, int K, double* __restrict__ values,
                      int32_t* __restrict__ idx)
{
    extern __shared__ double sm[];                     // m[sp*sp], v[s*s], then int flags
    __shared__ int wsum[32];
    const int b = blockIdx.x;
    const int Np = sp * sp, N = s * s;
    double* m = sm;
    double* v = sm + Np;
    const int tid = threadIdx.x;
    const double den = static_cast<double>(H) * static_cast<double>(Np);
    for (int j = tid; j < Np; j += blockDim.x) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h) acc = __dadd_rn(acc, sal[(static_cast<size_t>(b) * H + h) * Np + j]);
        m[j] = __ddiv_rn(acc, den);
    }
    __syncthreads();
    auto axis = [&](int d, int& i0, int& i1, double& lam) {
        double src = __dsub_rn(__ddiv_rn(__dmul_rn(__dadd_rn(static_cast<double>(d), 0.5), static_cast<double>(sp)),
                                         static_cast<double>(s)),
                               0.5);
        src = fmax(src, 0.0);
        int a = static_cast<int>(floor(src));
        a = min(a, sp - 1);
        i0 = a;
        i1 = min(a + 1, sp - 1);
        lam = __dsub_rn(src, static_cast<double>(a));
    };
    for (int t = tid; t < N; t += blockDim.x) {
        const int y = t / s, x = t - y * s;
        int y0, y1, x0, x1;
        double ly, lx;
        axis(y, y0, y1, ly);
        axis(x, x0, x1, lx);
        const double ox = __dsub_rn(1.0, lx), oy = __dsub_rn(1.0, ly);
        const double top = __dadd_rn(__dmul_rn(m[y0 * sp + x0], ox), __dmul_rn(m[y0 * sp + x1], lx));
        const double bot = __dadd_rn(__dmul_rn(m[y1 * sp + x0], ox), __dmul_rn(m[y1 * sp + x1], lx));
        const double val = __dadd_rn(__dmul_rn(top, oy), __dmul_rn(bot, ly));
        v[t] = val;
        if (values) values[static_cast<size_t>(b) * N + t] = val;
    }
    __syncthreads();
    if (K <= 0) return;
    // rank of t: the tokens before it in (value descending, index ascending) order
    int* kept = reinterpret_cast<int*>(v + N);
    for (int t = tid; t < N; t += blockDim.x) {
        const double vt = v[t];
        int rank = 0;
        for (int u = 0; u < N && rank < K; ++u) {
            const double vu = v[u];
            rank += (vu > vt) || (vu == vt && u < t);
        }
        kept[t] = rank < K;
    }
    __syncthreads();
    // ascending compaction: each thread owns a contiguous run of tokens
    const int per = (N + blockDim.x - 1) / blockDim.x;
    const int t0 = min(N, tid * per), t1 = min(N, t0 + per);
    int cnt = 0;
    for (int t = t0; t < t1; ++t) cnt += kept[t];
    const int lane = tid & 31, warp = tid >> 5;
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wsum[w];
    int pos = before + incl - cnt;
    for (int t = t0; t < t1; ++t)
        if (kept[t]) {
            if (pos < K) idx[static_cast<size_t>(b) * K + pos] = t;
            ++pos;
        }
}

struct ExactWs {
    size_t mx, l, sal, total;
};

inline ExactWs exact_ws_layout(int BH, int Np)
{
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    ExactWs w{};
    size_t o = 0;
    w.mx = o;  o = al(o + sizeof(double) * BH * Np);
    w.l = o;   o = al(o + sizeof(double) * BH * Np);
    w.sal = o; o = al(o + sizeof(double) * BH * Np);
    w.total = o;
    return w;
}

template <int D>
int launch_exact_d(const StepGeom& g_src, int H, int B, int s, const void* q_src, const void* k, double scale64,
                   int keep_k, int32_t* idx, double* values, void* ws, cudaStream_t st)
{
    const int BH = B * H, Np = g_src.N, L = g_src.L, sp = g_src.side;
    const ExactWs w = exact_ws_layout(BH, Np);
    auto* base = static_cast<uint8_t*>(ws);
    auto* mx = reinterpret_cast<double*>(base + w.mx);
    auto* ls = reinterpret_cast<double*>(base + w.l);
    auto* sal = reinterpret_cast<double*>(base + w.sal);
    const auto* qp = static_cast<const __nv_bfloat16*>(q_src);
    const auto* kp = static_cast<const __nv_bfloat16*>(k);
    const size_t rsm = sizeof(double) * kRowWarps * (D + (L <= kRowMaxKeys ? L : 0));
    if (ensure_smem_attr(row_stats_kernel<D>, static_cast<int>(rsm)) != cudaSuccess) return VAR_ERR_CUDA;
    const int rows = BH * Np;
    if (launch_kernel(row_stats_kernel<D>, dim3((rows + kRowWarps - 1) / kRowWarps), dim3(kRowWarps * 32), rsm, st,
                      false, qp, kp, BH, Np, L, g_src.cap, scale64, mx, ls) != cudaSuccess)
        return VAR_ERR_CUDA;
    if (launch_kernel(exact_saliency_kernel<D>, dim3((Np + kSalThreads - 1) / kSalThreads, BH), dim3(kSalThreads), 0,
                      st, false, qp, kp, Np, L, g_src.cap, scale64, static_cast<const double*>(mx),
                      static_cast<const double*>(ls), sal) != cudaSuccess)
        return VAR_ERR_CUDA;
    const int N = s * s;
    const size_t tsm = sizeof(double) * (Np + N) + sizeof(int) * N;
    if (ensure_smem_attr(exact_topk_kernel, static_cast<int>(tsm)) != cudaSuccess) return VAR_ERR_CUDA;
    return cuda_status(launch_kernel(exact_topk_kernel, dim3(B), dim3(1024), tsm, st, false,
                                     static_cast<const double*>(sal), H, sp, s, keep_k, values, idx));
}

}  // namespace

size_t guided_exact_workspace_bytes(int BH, int Np) { return exact_ws_layout(BH, Np).total; }

int launch_guided_exact(const StepGeom& g_src, int B, int H, int s, const void* q_src, const void* k, double scale64,
                        int keep_k, int32_t* idx, double* values, void* ws, size_t ws_bytes, cudaStream_t st)
{
    if (ws_bytes < guided_exact_workspace_bytes(B * H, g_src.N)) return VAR_ERR_WORKSPACE;
    const int N = s * s;
    if (sizeof(double) * (g_src.N + N) + sizeof(int) * N > 200 * 1024) return VAR_ERR_UNSUPPORTED;
    if (g_src.D == 128) return launch_exact_d<128>(g_src, H, B, s, q_src, k, scale64, keep_k, idx, values, ws, st);
    if (g_src.D == 64) return launch_exact_d<64>(g_src, H, B, s, q_src, k, scale64, keep_k, idx, values, ws, st);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
