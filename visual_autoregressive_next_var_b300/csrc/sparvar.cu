// Dynamic sparse attention pattern ("SparVAR" abstract: the sparse attention
// pattern of later high-resolution scales is predicted from a sparse decision
// scale and carried to them by index mapping).
//
// Block scores of the decision step on the GPU: the attention mass a unit of
// 64 keys receives from query i is sum_{j in unit} softmax_j(q_i . k_j * scale),
// which is the attention output of query i with the value rows replaced by
// the unit's indicator: V[j][c] = 1 if key j belongs to unit u0 + c, else 0.
// The dense attention kernel computes it on the tensor cores, head_dim units
// per pass; a second kernel averages it over each 8x8 query block, the heads
// and the batch, in a fixed order, so the scores are reproducible.
// The selection and the index mapping run on the host (api.cu).
#include <cuda_bf16.h>

#include "internal.h"

namespace varattn {

namespace {

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

// V_ind[bh][j][c] = 1 (bf16) where key j belongs to unit u0 + c; 8 columns per thread.
template <int D>
__global__ void __launch_bounds__(256) unit_indicator_kernel(const UnitMap m, int BH, int u0, __nv_bfloat16* v)
{
    const long long per_bh = static_cast<long long>(m.L) * (D / 8);
    const long long n = per_bh * BH;
    for (long long t = blockIdx.x * 256ll + threadIdx.x; t < n; t += static_cast<long long>(gridDim.x) * 256) {
        const long long r = t % per_bh;
        const int j = static_cast<int>(r / (D / 8));
        const int c0 = static_cast<int>(r % (D / 8)) * 8;
        const int c = unit_of(m, j) - u0 - c0;
        // bf16 1.0 in column c of the eight (element 2i in the low half of word i)
        const uint32_t one = (c & 1) ? 0x3F800000u : 0x00003F80u;
        reinterpret_cast<uint4*>(v)[t] = make_uint4(c >> 1 == 0 ? one : 0u, c >> 1 == 1 ? one : 0u,
                                                    c >> 1 == 2 ? one : 0u, c >> 1 == 3 ? one : 0u);
    }
}

// scores[qb][u0 + c] = mean over the batch, the heads and the 64 queries of query
// block qb of O[b][h][i][c].  Thread (c, part) sums each (b, h) pair part,
// part + 8, ... over the block's 64 queries in fp32 (64 terms in [0, 1]: a
// relative error of at most 64 * 2^-24, far below the bf16 rounding of the
// terms) and those sums in fp64; the eight parts are added in order.
template <int D>
__global__ void __launch_bounds__(8 * D) unit_score_kernel(const __nv_bfloat16* o, int BH, int side, int n_units,
                                                       int u0, double* scores)
{
    __shared__ double part[8][D];
    const int c = threadIdx.x % D, pr = threadIdx.x / D;
    const int nb = side / 8;
    const int qb = blockIdx.x, by = qb / nb, bx = qb - by * nb;
    const int N = side * side;
    double acc = 0.0;
    for (int bh = pr; bh < BH; bh += 8) {
        const __nv_bfloat16* base = o + static_cast<size_t>(bh) * N * D + c;
        float f = 0.f;
        for (int y = 0; y < 8; ++y)
#pragma unroll
            for (int x = 0; x < 8; ++x)
                f += __bfloat162float(base[static_cast<size_t>((by * 8 + y) * side + bx * 8 + x) * D]);
        acc += static_cast<double>(f);
    }
    part[pr][c] = acc;
    __syncthreads();
    if (pr == 0 && u0 + c < n_units) {
        double t = 0.0;
        for (int k = 0; k < 8; ++k) t += part[k][c];
        scores[static_cast<size_t>(qb) * n_units + u0 + c] = t / (static_cast<double>(BH) * 64.0);
    }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t sparvar_workspace_bytes(const StepGeom& g)
{
    const size_t BH = static_cast<size_t>(g.B) * g.H;
    return align256(BH * g.L * g.D * 2) + align256(BH * g.N * g.D * 2);
}

int launch_sparvar_scores(const StepGeom& g, const UnitMap& m, const void* q, const void* k, void* ws,
                          size_t ws_bytes, double* scores, cudaStream_t st, int32_t* status)
{
    if (ws_bytes < sparvar_workspace_bytes(g)) return VAR_ERR_WORKSPACE;
    const int BH = g.B * g.H;
    auto* v_ind = static_cast<__nv_bfloat16*>(ws);
    auto* o = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) +
                                              align256(static_cast<size_t>(BH) * g.L * g.D * 2));
    for (int u0 = 0; u0 < m.U; u0 += g.D) {
        const long long n = static_cast<long long>(BH) * g.L * (g.D / 8);
        const unsigned blocks = static_cast<unsigned>(std::min<long long>((n + 255) / 256, 148ll * 16));
        const cudaError_t e1 = g.D == 128
                                   ? launch_kernel(unit_indicator_kernel<128>, dim3(blocks), dim3(256), 0, st, false,
                                                   m, BH, u0, v_ind)
                                   : launch_kernel(unit_indicator_kernel<64>, dim3(blocks), dim3(256), 0, st, false,
                                                   m, BH, u0, v_ind);
        if (e1 != cudaSuccess) return VAR_ERR_CUDA;
        if (int rc = launch_attn_dense_vcap(g, q, k, v_ind, g.L, o, st, status)) return rc;
        const unsigned nqb = static_cast<unsigned>((g.side / 8) * (g.side / 8));
        const cudaError_t e2 = g.D == 128 ? launch_kernel(unit_score_kernel<128>, dim3(nqb), dim3(8 * 128), 0, st,
                                                          false, o, BH, g.side, m.U, u0, scores)
                                          : launch_kernel(unit_score_kernel<64>, dim3(nqb), dim3(8 * 64), 0, st, false,
                                                          o, BH, g.side, m.U, u0, scores);
        if (e2 != cudaSuccess) return VAR_ERR_CUDA;
    }
    return VAR_OK;
}

}  // namespace varattn
