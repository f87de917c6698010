// Internal declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/varattn.h"
#include "rt.h"

namespace varattn {

// Block-sparse unit metadata (the kernel's unit list and the host plan share
// it): bits 0-3 the square's query blocks that keep the unit, bit 4 a sink
// chunk, bit 5 every key valid, bits 8-11 valid key rows, 12-15 valid key
// columns, 16-22 valid keys of a sink chunk.
constexpr uint32_t META_SINK = 1u << 4;
constexpr uint32_t META_FULL = 1u << 5;
constexpr int SPARSE_MAX_UNITS = 1024;   // units per square

// Resolved problem geometry for one step.
struct StepGeom {
    int B, H, D;
    int side;        // s = side[step]
    int N;           // s*s queries
    int L;           // cached tokens of scales 0..step
    int cap;         // rows per (b,h) in K/V
    float scale;     // softmax scale
};

// Validate the problem and resolve the geometry of `step` (host only, no CUDA call).
int resolve(const var_problem* p, int32_t step, StepGeom* g);

// Device address of this library's status word on the current device (0 on error).
int32_t* device_status_ptr();

// The status word the kernels of a call with problem p record faults in: the
// caller's p->status, else the per-device word (0 on error).
int32_t* status_word(const var_problem* p);

// The argument checks of pivot selection, shared by the workspace and the
// allocation-free entry points (geometry in *g).
int check_pivot_args(const var_problem* p, int32_t step, const void* x, int32_t channels, int32_t keep_k,
                     const int32_t* idx, StepGeom* g);

// 3-D / 4-D bf16 tensor maps with 128-byte swizzle, box inner extent 64 elements.
// dims/strides as cuTensorMapEncodeTiled takes them (strides in bytes, rank-1 of them).
int encode_tmap_bf16(CUtensorMap* out, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box);

// Launchers: `status` is the device status word of the call.
int launch_attn_dense(const StepGeom& g, const void* q, const void* k, const void* v, void* o,
                      cudaStream_t st, int32_t* status, float* lse = nullptr);
// after_select: launch as a programmatic dependent of the pivot selection
// kernel just launched on `st` (which lets it set up beside the selection).
int launch_attn_pruned(const StepGeom& g, const void* q, const void* k, const void* v,
                       const int32_t* idx, int keep_k, void* o, cudaStream_t st, int32_t* status, bool scatter,
                       bool after_select = false);
int launch_attn_dense_halved(const StepGeom& g, const void* q, const void* k, const void* v, void* o,
                             cudaStream_t st, int32_t* status);
int launch_attn_blocksparse(const StepGeom& g, const int32_t* sides, int n_scales, int step,
                            const void* q, const void* k, const void* v,
                            const var_block_mask* mask, void* o, cudaStream_t st, int32_t* status);
size_t pivot_workspace_bytes(int B, int N, int C);
int launch_pivot_select(int B, int N, int C, const void* x, int keep_k, int32_t* idx,
                        float* scores, void* ws, size_t ws_bytes, cudaStream_t st, int32_t* status);
int launch_select_exact(int B, int N, int keep_k, const float* keys_lo, const float* keys_hi, int* band_idx,
                        double* band_score, int32_t* idx, cudaStream_t st, int32_t* status);
int launch_saliency(const StepGeom& g, int n_src, int L_src, const void* q, const void* k, const float* lse,
                    float* sal, cudaStream_t st, int32_t* status);
size_t guided_workspace_bytes(int B, int N);
// Attention-guided pivots decided in fp64 (guided_exact.cu): g_src is the source step.
size_t guided_exact_workspace_bytes(int BH, int Np);
int launch_guided_exact(const StepGeom& g_src, int B, int H, int s, const void* q_src, const void* k, double scale64,
                        int keep_k, int32_t* idx, double* values, void* ws, size_t ws_bytes, cudaStream_t st);
int launch_guided_pivot(int B, int H, int sp, int s, const float* sal, int keep_k, int32_t* idx, float* scores,
                        void* ws, size_t ws_bytes, cudaStream_t st, int32_t* status);
// The decision step's 64-key units (dynamic sparse pattern): the sink range
// [0, sink_len) in 64-token chunks (units [0, n_sink)), then every 8x8 key block
// of each later scale up to the decision scale, row-major, scale by scale.
struct UnitMap {
    int L, U, sink_len, n_sink, n_sc;
    int sc[VAR_MAX_SCALES];      // schedule index of each non-sink scale
    int off[VAR_MAX_SCALES];     // its first flat key
    int side[VAR_MAX_SCALES];
    int ubase[VAR_MAX_SCALES];   // its first unit
};
size_t sparvar_workspace_bytes(const StepGeom& g, int U);
// One-thread kernel whose wait gives up after limit_us and records VAR_ERR_TIMEOUT.
int launch_wait_timeout(int limit_us, cudaStream_t st, int32_t* status);
// Block scores of the decision step, exact enough to decide the selection at
// tau as the fp64 definition does (certified fp32, fp64 re-score of unsettled
// blocks; force: re-score every block).  scale64: the softmax scale in fp64.
int launch_sparvar_scores(const StepGeom& g, const UnitMap& m, const void* q, const void* k, double tau, int force,
                          double scale64, void* ws, size_t ws_bytes, double* scores, int32_t* rescored,
                          cudaStream_t st);
// Block scores from the decision step's row log2-sum-exp on the tensor cores
// (fp32, deterministic, no error bound).
int launch_sparvar_scores_fast(const StepGeom& g, const UnitMap& m, const void* q, const void* k, const float* lse,
                               void* ws, size_t ws_bytes, double* scores, cudaStream_t st, int32_t* status);
// fill_only: the rows not in idx only (oc unused).  beside: launch as a
// programmatic dependent of the preceding kernel, which must be the in-place
// attention of the same step (it lets the fill start beside itself).
int launch_restore_scatter(int B, int H, int D, int sp, int s, const void* prev, const void* oc,
                           const int32_t* idx, int keep_k, void* out, cudaStream_t st, int32_t* status,
                           bool fill_only, bool beside = false);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? VAR_OK : VAR_ERR_CUDA; }

#ifdef VAR_DEBUG
// Debug build: check an index list on the device (entries in [0, N), strictly
// ascending per batch element if asked); a bad list records VAR_ERR_INVALID_ARG.
int debug_check_indices(const int32_t* idx, int B, int K, int N, bool ascending, int32_t* status, cudaStream_t st);
#define VAR_DEBUG_CHECK_INDICES(idx, B, K, N, asc, status, st)                                  \
    do {                                                                                        \
        if (int rc_ = debug_check_indices((idx), (B), (K), (N), (asc), (status), (st))) return rc_; \
    } while (0)
#else
#define VAR_DEBUG_CHECK_INDICES(idx, B, K, N, asc, status, st) \
    do {                                                       \
    } while (0)
#endif

// SM count of the current device (0 if it cannot be read).
int sm_count();
// L2 cache bytes of the current device (0 if it cannot be read).
long long l2_bytes();

}  // namespace varattn
