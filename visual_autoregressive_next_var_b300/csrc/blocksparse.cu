// Block-sparse cross-scale attention ("SparVAR" abstract: attention sinks,
// cross-scale local windows, a block-wise sparse kernel): host launcher of the
// shared kernel in attn_kernel.cuh.
//
// Key tiles are built from 64-key units: flat 64-token chunks of the sink
// range (the leading scales kept by every query) read through a 3-D tensor
// map, and 8x8 key blocks of the other scales read through one 4-D tensor map
// per scale (D, x, y, b*h), so a block is a single TMA box whatever the
// scale's row stride.  Query tiles are two 8x8 query blocks, loaded the same
// way from a 4-D map of the query grid.
#include <cstring>

#include "attn_kernel.cuh"

namespace varattn {

template <int D>
static int launch_sparse(const StepGeom& g, const int32_t* sides, int step, const void* q, const void* k,
                         const void* v, const var_block_mask* mask, void* o, cudaStream_t st, int32_t* status)
{
    using Lay = AttnLayout<D>;
    auto kern = attn_kernel<D, MODE_SPARSE, SparseMaps>;

    // The sink range must end exactly at a scale boundary of the leading scales.
    int first_local = 0;
    long long cum = 0;
    while (first_local <= step && cum < mask->sink_len) {
        cum += static_cast<long long>(sides[first_local]) * sides[first_local];
        ++first_local;
    }
    if (cum != mask->sink_len) return VAR_ERR_INVALID_ARG;
    if (ensure_smem_attr(kern, Lay::SMEM_BYTES_SPARSE) != cudaSuccess) return VAR_ERR_CUDA;

    SparseMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const uint64_t BH = static_cast<uint64_t>(g.B) * g.H;
    const uint64_t row_bytes = D * 2ull;
    const uint64_t bh_bytes = static_cast<uint64_t>(g.cap) * row_bytes;
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(g.side),
                                  static_cast<uint64_t>(g.side), BH};
        const uint64_t strides[3] = {row_bytes, g.side * row_bytes, static_cast<uint64_t>(g.N) * row_bytes};
        const uint32_t box[4] = {64, 8, 8, 1};
        if (int rc = encode_tmap_bf16(&maps.q, q, 4, dims, strides, box)) return rc;
    }
    {
        // the output grid, for the epilogue's 8x8 block stores
        const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(g.side),
                                  static_cast<uint64_t>(g.side), BH};
        const uint64_t strides[3] = {row_bytes, g.side * row_bytes, static_cast<uint64_t>(g.N) * row_bytes};
        const uint32_t box[4] = {64, 8, 8, 1};
        if (int rc = encode_tmap_bf16(&maps.o, o, 4, dims, strides, box)) return rc;
    }
    const int sink_extent = mask->sink_len > 0 ? mask->sink_len : 1;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(sink_extent), BH};
        const uint64_t strides[2] = {row_bytes, bh_bytes};
        const uint32_t box[3] = {64, 64, 1};
        if (int rc = encode_tmap_bf16(&maps.k_sink, k, 3, dims, strides, box)) return rc;
        if (int rc = encode_tmap_bf16(&maps.v_sink, v, 3, dims, strides, box)) return rc;
    }
    uint32_t map_ok = 0;
    long long off = cum;
    for (int sc = first_local; sc <= step; ++sc) {
        const uint64_t s = static_cast<uint64_t>(sides[sc]);
        const uint64_t dims[4] = {static_cast<uint64_t>(D), s, s, BH};
        const uint64_t strides[3] = {row_bytes, s * row_bytes, bh_bytes};
        const uint32_t box[4] = {64, 8, 8, 1};
        const uint8_t* kb = static_cast<const uint8_t*>(k) + off * row_bytes;
        const uint8_t* vb = static_cast<const uint8_t*>(v) + off * row_bytes;
        if (int rc = encode_tmap_bf16(&maps.k_sc[sc], kb, 4, dims, strides, box)) return rc;
        if (int rc = encode_tmap_bf16(&maps.v_sc[sc], vb, 4, dims, strides, box)) return rc;
        map_ok |= 1u << sc;
        off += static_cast<long long>(s * s);
    }

    AttnArgs a = {};
    a.n_rows = g.N;
    a.n_q = g.N;
    a.L = g.L;
    a.heads = g.H;
    a.scale_log2 = g.scale * 1.4426950408889634f;
    a.o = static_cast<__nv_bfloat16*>(o);
    a.status = status;
    a.side_q = g.side;
    a.nb = g.side / 8;
    a.nsq = (a.nb + 1) / 2;
    a.sink_len = mask->sink_len;
    a.sink_extent = sink_extent;
    a.nnz = mask->nnz;
    a.map_ok = map_ok;
    a.row_ptr = mask->row_ptr;
    a.entries = mask->entries;
    for (int i = 0; i <= step; ++i) a.sides[i] = sides[i];
    a.n_bh = static_cast<int32_t>(BH);
    if (mask->n_squares > 0) {
        if (mask->n_squares != a.nsq * a.nsq || !mask->sq_ptr || !mask->sq_units || !mask->sq_order ||
            mask->plan_units < 0)
            return VAR_ERR_INVALID_ARG;
        a.sq_ptr = mask->sq_ptr;
        a.sq_units = reinterpret_cast<const int2*>(mask->sq_units);
        a.sq_order = mask->sq_order;
        a.plan_units = mask->plan_units;
    }
    // Heads per group: as many heads' K/V (read over the group's lifetime) as fit
    // in three eighths of L2 -- three quarters of one of the two dies' halves --
    // so each K/V byte crosses HBM about once.  Measured on the 2K workload:
    // groups sized to 3/4 of the whole L2 (4 heads) re-read 61 % of the K/V,
    // groups of 2 heads 2 %, in the same kernel time.
    {
        const long long l2 = l2_bytes();
        if (l2 <= 0) return VAR_ERR_CUDA;
        const long long per_head = 2ll * g.L * D * 2;
        const long long fit = (3 * l2 / 8) / (per_head > 0 ? per_head : 1);
        a.head_group = static_cast<int32_t>(fit < 1 ? 1 : (fit > a.n_bh ? a.n_bh : fit));
    }
    const uint64_t ctas = BH * static_cast<uint64_t>(a.nsq) * a.nsq;
    if (ctas > 0x7fffffffull) return VAR_ERR_UNSUPPORTED;
    return cuda_status(launch_kernel(kern, dim3(static_cast<unsigned>(ctas)), dim3(384), Lay::SMEM_BYTES_SPARSE, st,
                                     false, maps, a));
}

int launch_attn_blocksparse(const StepGeom& g, const int32_t* sides, int n_scales, int step, const void* q,
                            const void* k, const void* v, const var_block_mask* mask, void* o, cudaStream_t st,
                            int32_t* status)
{
    (void)n_scales;
    if (mask->qblock_side != 8) return VAR_ERR_UNSUPPORTED;
    if (g.side % 8 != 0) return VAR_ERR_UNSUPPORTED;
    if (g.D == 128) return launch_sparse<128>(g, sides, step, q, k, v, mask, o, st, status);
    if (g.D == 64) return launch_sparse<64>(g, sides, step, q, k, v, mask, o, st, status);
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
