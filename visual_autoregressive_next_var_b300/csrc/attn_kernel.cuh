// Cross-scale attention kernel for sm_103a, shared by the dense, pruned
// (gathered-query) and block-sparse entry points.
//
// Computes, per (b, h) and query row i, softmax(q_i K^T * scale) V over the
// cached tokens of scales 0..step ("SparVAR" abstract: every step attends to
// all tokens of the historical scales), optionally restricted to a key set:
//   MODE_DENSE   all L keys, query rows in order
//   MODE_GATHER  all L keys, query rows taken from an index list ("FastVAR"
//                abstract, cached token pruning; "ARVAR" Key Design 2)
//   MODE_SPARSE  the attention sinks plus the key blocks the block mask lists
//                for the row's 8x8 query block ("SparVAR" abstract:
//                attention sinks, cross-scale locality, block-wise kernel)
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
// only moved (and O rescaled) when a new maximum exceeds it by 2^8.  Dense and
// block-sparse tiles leave through the idle K ring: each softmax thread writes
// its normalised row into a swizzled staging tile and one thread per group
// stores it with tensor-map stores (gathered rows, which may scatter, are
// written by their threads).
//
// Block-sparse CTAs own a 2x2 square of 8x8 query blocks (tile t = block row
// t of the square, two blocks side by side).  Before the pipeline starts, the
// CTA merges the four blocks' sorted key-block lists into one deduplicated
// list of 64-key units in shared memory (sink chunks first), each with the
// bit set of the query blocks that keep it and its valid extent at the scale
// edge.  A 128-key tile is two consecutive units; rows mask the units their
// own block does not keep.
#pragma once
#include <cfloat>
#include <climits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace varattn {

enum : int { MODE_DENSE = 0, MODE_GATHER = 1, MODE_SPARSE = 2 };

struct DenseMaps {
    CUtensorMap q, k, v;   // 3-D (D, rows, B*H), box (64, 128, 1)
    CUtensorMap o;         // dense: 3-D (D, n_rows, B*H), box (64, 128, 1); the epilogue's tile stores
};

struct SparseMaps {
    CUtensorMap q;                     // 4-D (D, s_q, s_q, B*H), box (64, 8, 8, 1)
    CUtensorMap k_sink, v_sink;        // 3-D (D, sink_len, B*H), box (64, 64, 1)
    CUtensorMap k_sc[VAR_MAX_SCALES];  // 4-D (D, s, s, B*H) per non-sink scale, box (64, 8, 8, 1)
    CUtensorMap v_sc[VAR_MAX_SCALES];
    CUtensorMap o;                     // 4-D (D, s_q, s_q, B*H), box (64, 8, 8, 1): the epilogue's block stores
};

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
    static constexpr int B_PF = B_SF + 2;        // [4]  P_t written up to half h, at 2t + h (O_t rescaled first)
    static constexpr int B_OF = B_PF + 4;        // [1]  all products done
    static constexpr int B_DR = B_OF + 1;        // [1]  drain before teardown
    static constexpr int NBAR = B_DR + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // tmem slot, abort flag, unit count
    static constexpr int OFF_U = OFF_MISC + 16;           // block-sparse unit list
    static constexpr int MAXU = SPARSE_MAX_UNITS;         // units per block-sparse CTA
    static constexpr int MAXL = 512;                      // entries per query-block list
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;              // + alignment slack
    static constexpr int SMEM_BYTES_SPARSE = OFF_U + MAXU * 8 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
    // staging for the list merge (aliases the V ring, unused until the merge ends)
    static constexpr int STG_L = OFF_V;                               // int [4][MAXL]
    static constexpr int STG_P = STG_L + 4 * MAXL * 4;                // int [4][MAXL + 1]
    static constexpr int STG_M = STG_P + 4 * (MAXL + 1) * 4;          // u8  [4][MAXL]
    static constexpr int STG_N = STG_M + 4 * MAXL;                    // int [8]
    static_assert(STG_N + 32 <= OFF_BAR, "merge staging must fit in the V ring");
};

struct AttnArgs {
    int32_t n_rows;         // output rows per (b,h): N (dense) or keep_k (pruned)
    int32_t n_q;            // rows of the Q tensor per (b,h)
    int32_t L;              // visible cached keys
    int32_t heads;
    // CTA schedule (dense, gather).  A (b,h) has tiles_per_bh 128-row query
    // tiles, grouped into pair slots (tiles 2k, 2k+1).  CTAs [0, n_pair_ctas)
    // take pair slots in order; the other CTAs take one tile each ("split"
    // CTAs: the two softmax groups share that tile and take alternate key
    // tiles): first both tiles of the remaining pair slots, then the last tile
    // of each (b,h) when tiles_per_bh is odd.
    int32_t tiles_per_bh;
    int32_t slots_per_bh;   // tiles_per_bh / 2
    int32_t n_pair_ctas;
    int32_t n_conv_slots;   // pair slots taken by two split CTAs
    int32_t n_kv;           // ceil(L / 128)                   (dense, gather)
    float scale_log2;       // softmax scale * log2(e)
    const __nv_bfloat16* q; // gather source (pruned)
    const int32_t* idx;     // [B][n_rows] (pruned)
    __nv_bfloat16* o;       // [B][H][n_rows][D], or [B][H][n_q][D] when scatter is set
    int64_t o_repeat;       // non-zero: each output row is also written this many elements further
                            // (branch halving: the conditional half's rows repeated into the
                            // unconditional half)
    int32_t scatter;        // gather mode: write query idx[b][j]'s row of a full-grid output
    float* lse;             // dense mode, optional: [B][H][n_rows] row log2-sum-exp of the scaled
                            // scores (log2 of sum_j 2^(s_ij * scale * log2 e))
    int32_t* status;
    // block-sparse
    int32_t side_q;         // query grid side
    int32_t nb;             // query blocks per grid row
    int32_t nsq;            // 2x2 squares per grid row, ceil(nb / 2)
    int32_t sink_len;       // leading cache tokens every query keeps
    int32_t sink_extent;    // rows of the sink tensor maps (>= 1)
    int32_t nnz;            // entries[] length
    uint32_t map_ok;        // bit sc: scale sc has a per-scale tensor map
    const int32_t* row_ptr; // [n_qblocks + 1]
    const int32_t* entries; // packed (scale << 24) | (u << 12) | v
    const int32_t* sq_ptr;  // optional host-built plan: units of square q
    const int2* sq_units;
    const int32_t* sq_order;// squares in the order CTAs take them (heaviest first)
    int32_t n_bh;           // B * H
    int32_t head_group;     // planned order: heads per group (1 .. n_bh); groups run one after the
                            // other, inside a group the squares in sq_order, all its heads together
    int32_t plan_units;     // entries of sq_units
    int32_t sides[VAR_MAX_SCALES];
};


__device__ __forceinline__ void record_fault(volatile int* abort_flag, int32_t* status, int code)
{
    *abort_flag = 1;
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ bool list_contains(const int* a, int n, int key)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < key) lo = mid + 1;
        else hi = mid;
    }
    return lo < n && a[lo] == key;
}

__device__ __forceinline__ int list_lower_bound(const int* a, int n, int key)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Block-sparse schedule of the CTA owning the square with top-left block
// (by0, bx0): merge the four blocks' lists into unit list U; all threads call
// it.  Returns the number of units.  Malformed masks are recorded in the
// status word and their entries replaced by empty units.
template <int D>
__device__ int build_units(uint8_t* smem, const AttnArgs& a, int by0, int bx0)
{
    using Lay = AttnLayout<D>;
    constexpr int MAXL = Lay::MAXL, MAXU = Lay::MAXU;
    int* Ls = reinterpret_cast<int*>(smem + Lay::STG_L);
    int* Ps = reinterpret_cast<int*>(smem + Lay::STG_P);
    uint8_t* Ms = smem + Lay::STG_M;
    int* nn = reinterpret_cast<int*>(smem + Lay::STG_N);   // n[4], base[4]
    int2* U = reinterpret_cast<int2*>(smem + Lay::OFF_U);
    const int tid = threadIdx.x, nt = blockDim.x;

    for (int i = tid; i < MAXU; i += nt) U[i] = make_int2(INT_MAX, 0);
    if (tid < 4) {
        const int by = by0 + (tid >> 1), bx = bx0 + (tid & 1);
        int n = 0, base = 0;
        if (by < a.nb && bx < a.nb) {
            const int qb = by * a.nb + bx;
            base = __ldg(a.row_ptr + qb);
            const int end = __ldg(a.row_ptr + qb + 1);
            n = end - base;
            if (base < 0 || n < 0 || end > a.nnz) {
                atomicCAS(a.status, 0, VAR_ERR_INVALID_ARG);
                n = 0;
                base = 0;
            } else if (n > MAXL) {
                atomicCAS(a.status, 0, VAR_ERR_UNSUPPORTED);
                n = MAXL;
            }
        }
        nn[tid] = n;
        nn[4 + tid] = base;
    }
    __syncthreads();
    for (int idx = tid; idx < 4 * MAXL; idx += nt) {
        const int t = idx / MAXL, i = idx - t * MAXL;
        if (i < nn[t]) {
            int e = __ldg(a.entries + nn[4 + t] + i);
            const int sc = e >> 24, u = (e >> 12) & 0xFFF, v = e & 0xFFF;
            bool ok = e >= 0 && sc < VAR_MAX_SCALES && ((a.map_ok >> sc) & 1u);
            if (ok) {
                const int nbk = (a.sides[sc] + 7) >> 3;
                ok = u < nbk && v < nbk;
            }
            if (!ok) {
                atomicCAS(a.status, 0, VAR_ERR_INVALID_ARG);
                e = INT_MAX;
            }
            Ls[t * MAXL + i] = e;
        }
    }
    __syncthreads();
    // which blocks keep each entry; the first list holding a value owns it
    for (int idx = tid; idx < 4 * MAXL; idx += nt) {
        const int t = idx / MAXL, i = idx - t * MAXL;
        if (i < nn[t]) {
            const int e = Ls[t * MAXL + i];
            uint32_t m = 1u << t;
            int own = 1;
            for (int t2 = 0; t2 < 4; ++t2) {
                if (t2 == t) continue;
                if (list_contains(Ls + t2 * MAXL, nn[t2], e)) {
                    m |= 1u << t2;
                    if (t2 < t) own = 0;
                }
            }
            Ms[t * MAXL + i] = static_cast<uint8_t>(m);
            Ps[t * (MAXL + 1) + i + 1] = own;
        }
    }
    if (tid < 4) Ps[tid * (MAXL + 1)] = 0;
    __syncthreads();
    // per-list inclusive scan of the ownership flags (warp t scans list t)
    if (tid < 128) {
        const int w = tid >> 5, lane = tid & 31;
        int carry = 0;
        for (int base = 0; base < nn[w]; base += 32) {
            const int i = base + lane;
            int v = i < nn[w] ? Ps[w * (MAXL + 1) + i + 1] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += y;
            }
            if (i < nn[w]) Ps[w * (MAXL + 1) + i + 1] = v + carry;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
    const int n_sink = (a.sink_len + 63) >> 6;
    int total = n_sink;
    for (int t = 0; t < 4; ++t) total += Ps[t * (MAXL + 1) + nn[t]];
    if (total > MAXU && tid == 0) atomicCAS(a.status, 0, VAR_ERR_UNSUPPORTED);
    // each owned value lands at its rank among the distinct values
    for (int idx = tid; idx < 4 * MAXL; idx += nt) {
        const int t = idx / MAXL, i = idx - t * MAXL;
        if (i < nn[t] && Ps[t * (MAXL + 1) + i + 1] != Ps[t * (MAXL + 1) + i]) {
            const int e = Ls[t * MAXL + i];
            int rank = Ps[t * (MAXL + 1) + i];
            for (int t2 = 0; t2 < 4; ++t2)
                if (t2 != t) rank += Ps[t2 * (MAXL + 1) + list_lower_bound(Ls + t2 * MAXL, nn[t2], e)];
            uint32_t meta = 0;
            if (e != INT_MAX) {
                const int s = a.sides[e >> 24], u = (e >> 12) & 0xFFF, v = e & 0xFFF;
                const uint32_t rows = static_cast<uint32_t>(min(8, s - 8 * u));
                const uint32_t cols = static_cast<uint32_t>(min(8, s - 8 * v));
                meta = Ms[t * MAXL + i] | (rows << 8) | (cols << 12) |
                       ((rows == 8 && cols == 8) ? META_FULL : 0u);
            }
            const int pos = n_sink + rank;
            if (pos < MAXU) U[pos] = make_int2(e, static_cast<int>(meta));
        }
    }
    for (int c = tid; c < n_sink && c < MAXU; c += nt) {
        const uint32_t cnt = static_cast<uint32_t>(min(64, a.sink_len - 64 * c));
        U[c] = make_int2(-1 - c, static_cast<int>(0xFu | META_SINK | (cnt == 64 ? META_FULL : 0u) | (cnt << 16)));
    }
    __syncthreads();
    return min(total, MAXU);
}

template <int D, int MODE, typename Maps>
__global__ void __launch_bounds__(384, 1) attn_kernel(const __grid_constant__ Maps maps, const AttnArgs args)
{
    using Lay = AttnLayout<D>;
    constexpr int NS = Lay::NS;
    constexpr bool GATHER = MODE == MODE_GATHER;
    constexpr bool SPARSE = MODE == MODE_SPARSE;
    // Publish P per 64-key half (the PV of the first half overlaps the second
    // half's exponentials).  Measured: faster for the block-sparse kernel, a
    // little slower for the dense and gathered ones, whose PV then waits once.
    constexpr bool P_HALVES = SPARSE;
    // Free K/V ring slots from a softmax thread that has seen the next S (no
    // tensor-core commit in the issue stream) or by commits after the last
    // product that reads them (the slot frees sooner).  Measured: the first is
    // faster for the gathered kernel, the second for the dense one, whose
    // two-slot ring then feeds the next value tile sooner.
    constexpr bool SOFT_RELEASE = GATHER;
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
    const int2* U = reinterpret_cast<const int2*>(smem + Lay::OFF_U);

    int bh, row0 = 0, by0 = 0, bx0 = 0;
    bool split = false;        // one query tile; group g takes key tiles j = g (mod 2)
    if constexpr (SPARSE) {
        const int nsq2 = args.nsq * args.nsq;
        int sq;
        if (args.sq_order) {
            // planned: head groups in turn (their K/V stay in L2 while the group
            // runs); inside a group the squares heaviest first, all its heads together
            const int G = args.head_group;
            const int g = blockIdx.x / (G * nsq2);
            const int o = blockIdx.x - g * G * nsq2;
            const int gs = min(G, args.n_bh - g * G);
            const int rnk = o / gs;
            bh = g * G + (o - rnk * gs);
            sq = min(max(__ldg(args.sq_order + rnk), 0), nsq2 - 1);
        } else {
            bh = blockIdx.x / nsq2;
            sq = blockIdx.x - bh * nsq2;
        }
        by0 = 2 * (sq / args.nsq);
        bx0 = 2 * (sq % args.nsq);
    } else {
        const int c = static_cast<int>(blockIdx.x);
        if (c < args.n_pair_ctas) {
            bh = c / args.slots_per_bh;
            row0 = (c - bh * args.slots_per_bh) * 256;
        } else {
            split = true;
            const int sgl = c - args.n_pair_ctas;
            const int n_conv = args.n_conv_slots;            // pair slots taken as two split CTAs
            if (sgl < 2 * n_conv) {
                const int slot = args.n_pair_ctas + sgl / 2;
                bh = slot / args.slots_per_bh;
                row0 = (slot - bh * args.slots_per_bh) * 256 + (sgl & 1) * 128;
            } else {
                bh = sgl - 2 * n_conv;
                row0 = (args.tiles_per_bh - 1) * 128;
            }
        }
    }

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) mbar_init(bar(Lay::B_QF + t), GATHER ? 128 : 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(Lay::B_KF + s), 1);
            mbar_init(bar(Lay::B_KE + s), 1);
            mbar_init(bar(Lay::B_VF + s), 1);
            mbar_init(bar(Lay::B_VE + s), 1);
        }
        for (int t = 0; t < 2; ++t) mbar_init(bar(Lay::B_SF + t), 1);
        for (int t = 0; t < 4; ++t) mbar_init(bar(Lay::B_PF + t), 128);
        mbar_init(bar(Lay::B_OF), 1);
        mbar_init(bar(Lay::B_DR), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        if constexpr (SPARSE) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.k_sink);
            tma_prefetch_desc(&maps.v_sink);
        } else {
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(&maps.v);
            if (!GATHER) tma_prefetch_desc(&maps.q);
        }
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent (the gathered attention of
    // var_pruned_step, behind the pivot selection), every thread waits here,
    // after the set-up and before anything reads an input; an ordinary launch
    // returns at once.
    pdl_wait();
    // In place (gathered rows scattered into the full grid): from here on the
    // fill of the other rows may start beside this grid -- the indices are
    // final, and it reads and writes none of this grid's rows.
    if (GATHER && args.scatter) pdl_launch_dependents();

    int n_kv = args.n_kv;
    int n_units = 0;
    if constexpr (SPARSE) {
        if (args.sq_units) {
            // the host-built plan: copy this square's units
            const int sq = (by0 >> 1) * args.nsq + (bx0 >> 1);
            const int u0 = min(max(__ldg(args.sq_ptr + sq), 0), args.plan_units);
            const int u1 = min(max(__ldg(args.sq_ptr + sq + 1), u0), args.plan_units);
            n_units = min(max(u1 - u0, 0), Lay::MAXU);
            if (threadIdx.x == 0 && u1 - u0 > Lay::MAXU) atomicCAS(args.status, 0, VAR_ERR_UNSUPPORTED);
            int2* Uw = reinterpret_cast<int2*>(smem + Lay::OFF_U);
            for (int i = threadIdx.x; i < n_units; i += blockDim.x) Uw[i] = __ldg(args.sq_units + u0 + i);
            __syncthreads();
        } else {
            n_units = build_units<D>(smem, args, by0, bx0);
        }
        n_kv = (n_units + 1) >> 1;
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            if constexpr (SPARSE) {
                for (int t = 0; t < 2; ++t) {
                    mbar_arrive_expect_tx(bar(Lay::B_QF + t), Lay::TILE_BYTES);
                    for (int hb = 0; hb < 2; ++hb)
                        for (int hh = 0; hh < Lay::HALVES; ++hh)
                            tma_load_4d(sbase + Lay::OFF_Q + t * Lay::TILE_BYTES + hh * Lay::HALF_BYTES +
                                            hb * (Lay::HALF_BYTES / 2),
                                        &maps.q, hh * 64, (bx0 + hb) * 8, (by0 + t) * 8, bh,
                                        bar(Lay::B_QF + t));
                }
            } else if constexpr (!GATHER) {
                for (int t = 0; t < (split ? 1 : 2); ++t) {
                    mbar_arrive_expect_tx(bar(Lay::B_QF + t), Lay::TILE_BYTES);
                    for (int hh = 0; hh < Lay::HALVES; ++hh)
                        tma_load_3d(sbase + Lay::OFF_Q + t * Lay::TILE_BYTES + hh * Lay::HALF_BYTES,
                                    &maps.q, hh * 64, row0 + t * 128, bh, bar(Lay::B_QF + t));
                }
            }
            // one 128-key tile of K or V into the slot at `dst`
            auto load_tile = [&](bool is_v, uint32_t dst, int j, uint32_t b) {
                if constexpr (SPARSE) {
                    const CUtensorMap* flat = is_v ? &maps.v_sink : &maps.k_sink;
                    const CUtensorMap* per = is_v ? maps.v_sc : maps.k_sc;
                    for (int hb = 0; hb < 2; ++hb) {
                        const int unit = 2 * j + hb;
                        const int e = unit < n_units ? U[unit].x : INT_MAX;
                        const int sc = e >> 24;
                        const bool blk = e >= 0 && e != INT_MAX && sc < VAR_MAX_SCALES &&
                                         ((args.map_ok >> sc) & 1u);
                        for (int hh = 0; hh < Lay::HALVES; ++hh) {
                            const uint32_t d = dst + hh * Lay::HALF_BYTES + hb * (Lay::HALF_BYTES / 2);
                            if (e < 0)          // sink chunk -1-e
                                tma_load_3d(d, flat, hh * 64, 64 * (-1 - e), bh, b);
                            else if (blk)
                                tma_load_4d(d, per + sc, hh * 64, (e & 0xFFF) * 8, ((e >> 12) & 0xFFF) * 8,
                                            bh, b);
                            else                // no unit: rows past the sink extent read as zeros
                                tma_load_3d(d, flat, hh * 64, args.sink_extent, bh, b);
                        }
                    }
                } else {
                    const CUtensorMap* m = is_v ? &maps.v : &maps.k;
                    for (int hh = 0; hh < Lay::HALVES; ++hh)
                        tma_load_3d(dst + hh * Lay::HALF_BYTES, m, hh * 64, j * 128, bh, b);
                }
            };
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % NS;
                const uint32_t ph = (j / NS) & 1;
                if (!mbar_wait(bar(Lay::B_KE + s), ph ^ 1, abort_flag)) {
                    record_fault(abort_flag, args.status, VAR_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(bar(Lay::B_KF + s), Lay::TILE_BYTES);
                load_tile(false, sbase + Lay::OFF_K + s * Lay::TILE_BYTES, j, bar(Lay::B_KF + s));
                ++k_issued;
                if (!mbar_wait(bar(Lay::B_VE + s), ph ^ 1, abort_flag)) {
                    record_fault(abort_flag, args.status, VAR_ERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(bar(Lay::B_VF + s), Lay::TILE_BYTES);
                load_tile(true, sbase + Lay::OFF_V + s * Lay::TILE_BYTES, j, bar(Lay::B_VF + s));
                ++v_issued;
            }
            // Every copy this thread started must land before the CTA may exit.
            for (int j = (k_issued > NS ? k_issued - NS : 0); j < k_issued; ++j)
                mbar_wait(bar(Lay::B_KF + j % NS), (j / NS) & 1, nullptr);
            for (int j = (v_issued > NS ? v_issued - NS : 0); j < v_issued; ++j)
                mbar_wait(bar(Lay::B_VF + j % NS), (j / NS) & 1, nullptr);
            if (!GATHER)
                for (int t = 0; t < (split ? 1 : 2); ++t) mbar_wait(bar(Lay::B_QF + t), 0, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
            auto qk = [&](int t, int s, int qt) {   // S_t = Q_qt K_s^T
                const uint32_t qa = sbase + Lay::OFF_Q + qt * Lay::TILE_BYTES;
                const uint32_t kb = sbase + Lay::OFF_K + s * Lay::TILE_BYTES;
                const uint32_t dst = tmem + (t ? Lay::COL_S1 : Lay::COL_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * Lay::HALF_BYTES + (kk % 4) * 32;
                    umma_ss(dst, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                            IDESC_QK, kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V_s.  With P_HALVES each 64-key half is issued as soon as
            // the softmax has written that half of P; otherwise once all of P is
            // written (the wait on phase `ph` of the barrier)
            auto pv = [&](int t, int s, bool acc, uint32_t ph) -> bool {
                const uint32_t vb = sbase + Lay::OFF_V + s * Lay::TILE_BYTES;
                const uint32_t dst = tmem + (t ? Lay::COL_O1 : Lay::COL_O0);
                const uint32_t pa = tmem + (t ? Lay::COL_S1 : Lay::COL_S0);
                for (int h = 0; h < 2; ++h) {
                    if (P_HALVES || h == 0) {   // without halves: one wait, for all of P
                        if (!mbar_wait(bar(Lay::B_PF + 2 * t + (P_HALVES ? h : 1)), ph, abort_flag)) return false;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const int kk = 4 * h + k4;
                        umma_ts(dst, pa + kk * 8, sdesc_sw128(vb + kk * 2048, Lay::HALF_BYTES, 1024),
                                IDESC_PV, (acc || kk > 0) ? 1u : 0u);
                    }
                }
                return true;
            };
            bool ok = mbar_wait(bar(Lay::B_QF + 0), 0, abort_flag) &&
                      (split || mbar_wait(bar(Lay::B_QF + 1), 0, abort_flag));
            if (split) {
                // one query tile; group g takes key tiles j = g, g + 2, ...: its
                // S_g = Q_0 K_j^T, O_g += P_g V_j; each K / V tile is used once
                for (int g0 = 0; g0 < 2 && ok && g0 < n_kv; ++g0) {
                    if (!(ok = mbar_wait(bar(Lay::B_KF + g0 % NS), (g0 / NS) & 1, abort_flag))) break;
                    tc_fence_after();
                    qk(g0, g0 % NS, 0);
                    umma_commit(bar(Lay::B_SF + g0));
                    if (!SOFT_RELEASE) umma_commit(bar(Lay::B_KE + g0 % NS));
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int g1 = j & 1, jj = j >> 1;
                    const int s = j % NS;
                    if (!(ok = mbar_wait(bar(Lay::B_VF + s), (j / NS) & 1, abort_flag) &&
                               pv(g1, s, jj > 0, jj & 1)))
                        break;
                    if (!SOFT_RELEASE) umma_commit(bar(Lay::B_VE + s));
                    const int jn = j + 2;
                    if (jn < n_kv) {
                        if (!(ok = mbar_wait(bar(Lay::B_KF + jn % NS), (jn / NS) & 1, abort_flag))) break;
                        tc_fence_after();
                        qk(g1, jn % NS, 0);
                        umma_commit(bar(Lay::B_SF + g1));
                        if (!SOFT_RELEASE) umma_commit(bar(Lay::B_KE + jn % NS));
                    }
                }
            } else {
                if (ok && n_kv > 0) {
                    ok = mbar_wait(bar(Lay::B_KF + 0), 0, abort_flag);
                    if (ok) {
                        tc_fence_after();
                        qk(0, 0, 0);
                        umma_commit(bar(Lay::B_SF + 0));
                        qk(1, 0, 1);
                        umma_commit(bar(Lay::B_SF + 1));
                        if (!SOFT_RELEASE) umma_commit(bar(Lay::B_KE + 0));
                    }
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int s = j % NS;
                    const uint32_t ph = (j / NS) & 1;
                    const bool more = j + 1 < n_kv;
                    const int s1 = (j + 1) % NS;
                    const uint32_t ph1 = ((j + 1) / NS) & 1;
                    ok = mbar_wait(bar(Lay::B_VF + s), ph, abort_flag) && pv(0, s, j > 0, j & 1);
                    if (!ok) break;
                    if (more) {
                        if (!(ok = mbar_wait(bar(Lay::B_KF + s1), ph1, abort_flag))) break;
                        tc_fence_after();
                        qk(0, s1, 0);
                        umma_commit(bar(Lay::B_SF + 0));
                    }
                    if (!(ok = pv(1, s, j > 0, j & 1))) break;
                    if (!SOFT_RELEASE) umma_commit(bar(Lay::B_VE + s));
                    if (more) {
                        qk(1, s1, 1);
                        umma_commit(bar(Lay::B_SF + 1));
                        if (!SOFT_RELEASE) umma_commit(bar(Lay::B_KE + s1));
                    }
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
        const int q4 = 2 * g + (r >> 6);     // block of the square (block-sparse); warp-uniform
        int tok_row = 0;                     // gather mode: the grid token of this query row

        if (GATHER && !(split && g == 1)) {
            // This thread's query row, gathered by index, into the swizzled tile.
            const int b = bh / args.heads;
            uint8_t* qs = smem + Lay::OFF_Q + g * Lay::TILE_BYTES;
            uint4 chunk[D / 8];
            if (qrow < args.n_rows) {
                int tok = __ldg(args.idx + static_cast<size_t>(b) * args.n_rows + qrow);
                tok = min(max(tok, 0), args.n_q - 1);
                tok_row = tok;
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
        // a split CTA's group g takes key tiles j = g, g + 2, ...
        const int n_local = split ? (n_kv + 1 - g) / 2 : n_kv;
        for (int jj = 0; jj < n_local; ++jj) {
            const int j = split ? 2 * jj + g : jj;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(Lay::B_SF + g), jj & 1, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // SOFT_RELEASE: ring slots this S proves free.  The products that last
            // read K_j (this step's QK of both tiles) and the V of the step before
            // were issued ahead of the QK whose completion this wait observed, and
            // the tensor core completes its work in issue order.
            if (SOFT_RELEASE && r == 0 && (split || g == 1)) {
                const int jv = split ? j - 2 : j - 1;
                mbar_arrive(bar(Lay::B_KE + j % NS));
                if (jv >= 0) mbar_arrive(bar(Lay::B_VE + jv % NS));
            }
            uint32_t s[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
            tmem_wait_ld();
            if constexpr (SPARSE) {
                // keep set of each 64-key unit for this row's query block
                uint32_t keep[4];
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    const int unit = 2 * j + hb;
                    const uint32_t meta = unit < n_units ? static_cast<uint32_t>(U[unit].y) : 0u;
                    uint64_t kp;
                    if (!((meta >> q4) & 1u)) {
                        kp = 0ull;
                    } else if (meta & META_FULL) {
                        kp = ~0ull;
                    } else if (meta & META_SINK) {
                        kp = (1ull << ((meta >> 16) & 63u)) - 1ull;          // count < 64 here
                    } else {
                        const uint32_t rows = (meta >> 8) & 15u, cols = (meta >> 12) & 15u;
                        const uint64_t rowbits = rows >= 8 ? ~0ull : (1ull << (8 * rows)) - 1ull;
                        const uint64_t colbits = static_cast<uint64_t>((1u << cols) - 1u) * 0x0101010101010101ull;
                        kp = rowbits & colbits;
                    }
                    keep[2 * hb] = static_cast<uint32_t>(kp);
                    keep[2 * hb + 1] = static_cast<uint32_t>(kp >> 32);
                }
                if ((keep[0] & keep[1] & keep[2] & keep[3]) != 0xffffffffu) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (!((keep[c >> 5] >> (c & 31)) & 1u)) s[c >> 5][c & 31] = __float_as_uint(-INFINITY);
                }
            } else {
                const int valid = args.L - j * 128;
                if (valid < 128) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= valid) s[c >> 5][c & 31] = __float_as_uint(-INFINITY);
                }
            }
            // row maximum: eight independent chains of 3-input max
            float mc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int base = q * 16;      // chain q covers columns [16q, 16q + 16)
                float m = __uint_as_float(s[base >> 5][base & 31]);
#pragma unroll
                for (int c = 1; c < 15; c += 2)
                    m = fmax3(m, __uint_as_float(s[(base + c) >> 5][(base + c) & 31]),
                              __uint_as_float(s[(base + c + 1) >> 5][(base + c + 1) & 31]));
                mc[q] = fmaxf(m, __uint_as_float(s[(base + 15) >> 5][(base + 15) & 31]));
            }
            const float mx = fmax3(fmax3(mc[0], mc[1], mc[2]), fmax3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
            const float m_tile = mx * sl2;
            const bool need = m_tile > m_run + 8.0f;
            const float m_new = need ? m_tile : m_run;
            const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
            l_run *= alpha;
            m_run = m_new;
            // P = exp2(S * scale*log2e - m), packed to bf16 pairs, 16 columns at a
            // time; each 64-key half is published as soon as it is written, so the
            // PV of the first half overlaps the exponentials of the second
            const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
            const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(neg_m, neg_m);
            uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[cc][2 * c]), __uint_as_float(s[cc][2 * c + 1])),
                                               sc2, nm2);
                    float x0, x1;
                    f2_unpack(x2, x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    sum2 = f2_add(sum2, f2_pack(p0, p1));
                    pk[c] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tS + cc * 16, pk);
                if (cc == 1 && __any_sync(0xffffffffu, need && jj > 0)) {
                    // O_t *= alpha where the running maximum moved, before the first half
                    // of this step's P is published (every earlier PV of this tile has
                    // completed: it was issued ahead of the QK whose S this thread
                    // waited for)
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
                if (cc == 3 || (P_HALVES && cc == 1)) {
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(bar(Lay::B_PF + 2 * g + (cc >> 1)));
                }
            }
            {
                float a0, a1;
                f2_unpack(sum2, a0, a1);
                l_run += a0 + a1;
            }
        }
        if (ok) ok = mbar_wait(bar(Lay::B_OF), 0, abort_flag);
        // split CTA: group 1 hands its row's (m, l) to group 0, which merges
        // O_0 and O_1 (both in its tensor-memory lanes) into the output
        float2* comb = reinterpret_cast<float2*>(smem + Lay::OFF_V);   // the V ring is idle now
        float a0 = 1.f, a1 = 0.f;
        if (split) {
            if (g == 1) {
                if (ok) comb[r] = make_float2(m_run, l_run);
                named_bar_arrive(1, 256);
            } else {
                named_bar_sync(1, 256);
                const float2 ml = comb[r];
                const float mm = fmaxf(m_run, ml.x);
                a0 = l_run > 0.f ? ex2_approx(m_run - mm) : 0.f;
                a1 = ml.y > 0.f ? ex2_approx(ml.x - mm) : 0.f;
                l_run = l_run * a0 + ml.y * a1;
                m_run = mm;
            }
        }
        if (!ok) record_fault(abort_flag, args.status, VAR_ERR_TIMEOUT);
        if (!split || g == 0) {
            tc_fence_after();
            // destination row of this thread, or none
            __nv_bfloat16* dst = nullptr;
            if constexpr (SPARSE) {
                const int by = by0 + (q4 >> 1), bx = bx0 + (q4 & 1);
                if (by < args.nb && bx < args.nb) {
                    const int y = by * 8 + ((r & 63) >> 3), x = bx * 8 + (r & 7);
                    dst = args.o + (static_cast<size_t>(bh) * args.n_q + y * args.side_q + x) * D;
                }
            } else if (qrow < args.n_rows) {
                dst = (GATHER && args.scatter)
                          ? args.o + (static_cast<size_t>(bh) * args.n_q + tok_row) * D
                          : args.o + (static_cast<size_t>(bh) * args.n_rows + qrow) * D;
            }
            const bool any = l_run > 0.f;            // a row that kept no key is written as zeros
            const float inv = any ? 1.0f / l_run : 0.f;
            if (ok && !SPARSE && !GATHER && args.lse && qrow < args.n_rows)
                args.lse[static_cast<size_t>(bh) * args.n_rows + qrow] = any ? m_run + log2f(l_run) : -INFINITY;
            const uint32_t tO1 = tmem + lane_base + Lay::COL_O1;
            // dense and block-sparse: the normalised tile is staged in the idle K ring
            // (128-byte swizzle, as the loads) and written by tensor-map stores
            uint8_t* st_tile = smem + Lay::OFF_K + g * Lay::TILE_BYTES;
#pragma unroll
            for (int c0 = 0; c0 < D && ok; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c0, o);
                if (split) {
                    uint32_t o1[32];
                    tmem_ld32(tO1 + c0, o1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        o[c] = __float_as_uint(__uint_as_float(o[c]) * a0 +
                                               (a1 != 0.f ? __uint_as_float(o1[c]) * a1 : 0.f));
                }
                tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    w[c] = any ? pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv)
                               : 0u;
                if constexpr (GATHER) {
                    if (dst) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                        for (int c = 0; c < 4; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int col = c0 + 8 * c;          // first of the 8 columns of this 16-byte chunk
                        const int hh = col >> 6, cc = (col & 63) >> 3;
                        *reinterpret_cast<uint4*>(st_tile + hh * Lay::HALF_BYTES + r * 128 + ((cc ^ (r & 7)) << 4)) =
                            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    }
                }
            }
            if constexpr (!GATHER) {
                // every thread of the group arrives, whatever its status; the tile is
                // stored only if all of it was written
                fence_proxy_async_smem();
                const bool all_ok = bar_red_and(2 + g, 128, ok);
                if (all_ok && r == 0) {
                    const uint32_t src = smem_u32(st_tile);
                    if constexpr (SPARSE) {
                        for (int hb = 0; hb < 2; ++hb) {
                            const int by = by0 + g, bx = bx0 + hb;
                            if (by >= args.nb || bx >= args.nb) continue;
                            for (int hh = 0; hh < Lay::HALVES; ++hh)
                                tma_store_4d(&maps.o, hh * 64, bx * 8, by * 8, bh,
                                             src + hh * Lay::HALF_BYTES + hb * (Lay::HALF_BYTES / 2));
                        }
                    } else {
                        const int bh_rep = args.o_repeat ? static_cast<int>(args.o_repeat / (static_cast<int64_t>(args.n_rows) * D)) : 0;
                        for (int rep = 0; rep < (args.o_repeat ? 2 : 1); ++rep)
                            for (int hh = 0; hh < Lay::HALVES; ++hh)
                                tma_store_3d(&maps.o, hh * 64, row0 + g * 128, bh + rep * bh_rep,
                                             src + hh * Lay::HALF_BYTES);
                    }
                    bulk_commit();
                    bulk_wait_read0();
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

}  // namespace varattn
