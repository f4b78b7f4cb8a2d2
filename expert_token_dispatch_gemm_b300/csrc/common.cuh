// Shared device helpers and internal launcher declarations of libmoe (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Tokens per histogram segment. The routing kernel and the standalone histogram kernel
// both count expert ids per segment of this many tokens; the scan turns the per-segment
// counts into the stable rank base of every segment.
constexpr int kSegTokens = 64;
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
// Gate rows per interleaved gate/up block of the packed weights: block b holds gate rows
// 64b..64b+63 followed by the matching up rows. The intermediate size is padded to
// kIpadAlign (two blocks: the 256 weight rows of one tensor-core tile).
constexpr int kGateUpBlock = 64;
constexpr int kIpadAlign = 128;

// Rows per M tile of the grouped GEMMs (tensor-core path and fp32 path).
constexpr int kTcBlockM = 128;
constexpr int kSimtBlockM = 128;

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// 16-byte vector of T: 8 bf16 or 4 fp32.
template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void to_float(const uint4 &v, float *f) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 p = __bfloat1622float2(h[i]);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
    __device__ __forceinline__ static uint4 from_float(const float *f) {
        uint4 v;
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        return v;
    }
};
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void to_float(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 from_float(const float *f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

// ----------------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel of the forward is launched so that it may
// start while the kernel before it in the stream finishes: it waits for that grid (and
// its memory) before its first access to global memory, then lets the next grid launch.
// Setup that touches no global memory (TMEM allocation, barrier initialisation) runs
// before the wait, overlapping the previous kernel's tail.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// ----------------------------------------------------------------------------------
// Internal launchers (host side). Each returns the cudaError_t of its launch(es).
// ----------------------------------------------------------------------------------
struct LayerDims {
    int N, H, I, Ipad, E, k, P;
    int capacity;      // INT32_MAX when unlimited
    int dtype;         // MOE_DTYPE_*
    int group_limit;   // partitions a token may use; 0 when unlimited
    const float *sel_bias;   // [E] selection-only bias or nullptr
    int slot_priority;       // 1: capacity ranks pairs slot-major (j*N + t)
    int training;            // 1: the forward keeps what the backward needs
};
// Histogram segments of the dispatch scan: ceil(N/64) token segments, or in slot-major
// priority k slots x ceil(N / 64k) token spans.
int num_segments(const LayerDims &d);
// Largest group limit and partition count of the group-limited routing.
constexpr int kMaxGroupLimit = 8;
constexpr int kMaxGroupPartitions = 64;

cudaError_t launch_route(const LayerDims &d, const void *x, const void *w_router,
                         const float *b_router, int32_t *topk_idx, float *topk_w,
                         float *logits /* [N, E] or nullptr */,
                         int32_t *seg_hist /* [nseg, E] or nullptr */, cudaStream_t s);

cudaError_t launch_update_selection_bias(const LayerDims &d, const int32_t *routed_counts,
                                        float *selection_bias, float gamma, cudaStream_t s);

cudaError_t launch_histogram(const LayerDims &d, const int32_t *topk_idx, int32_t *seg_hist,
                             int32_t *status, cudaStream_t s);
// scan + assign in one kernel (the scan's segment bases are not materialised)
cudaError_t launch_scan_assign(const LayerDims &d, const int32_t *topk_idx, const int32_t *seg_hist,
                               int32_t *routed_counts, int32_t *counts, int32_t *expert_offsets,
                               int32_t *part_offsets, int32_t *slot_pos, int32_t *perm,
                               int32_t *status, cudaStream_t s);
cudaError_t launch_permute(const LayerDims &d, const void *x, const int32_t *slot_pos,
                           void *send, cudaStream_t s);

cudaError_t launch_pack_gate_up(const LayerDims &d, const void *w_gate, const void *w_up,
                                void *packed, cudaStream_t s);

// Tensor-core (bf16) grouped GEMMs. h has row stride Ipad.
cudaError_t launch_tc_gate_up(const LayerDims &d, const void *send, const int32_t *expert_offsets,
                              int e_begin, int e_end, const void *packed, void *h,
                              void *gu /* [N*k, 2 Ipad] or nullptr */, int32_t *status,
                              int num_sms, cudaStream_t s);
cudaError_t launch_tc_down(const LayerDims &d, const void *h, const int32_t *expert_offsets,
                           int e_begin, int e_end, const void *w_down, const int32_t *perm,
                           const float *topk_w, void *out_slots, int32_t *status, int num_sms,
                           cudaStream_t s);

// Tensor-core (bf16) router: logits, top-k, softmax and segment histogram in one kernel.
// seg_hist and status may be null.
cudaError_t launch_tc_route(const LayerDims &d, const void *x, const void *w_router,
                            const float *bias, int32_t *topk_idx, float *topk_w,
                            float *logits, int32_t *seg_hist, int32_t *status, int num_sms,
                            cudaStream_t s);

// Router load statistics: per-block partial sums of the token softmax [kStatsBlocks, E]
// in `partials`, then load_frac / prob_mean. TP row split: ordered sum of tp padded
// outputs.
constexpr int kStatsBlocks = 256;

// Backward: grouped GEMMs (tensor cores for bf16, FFMA for fp32), then the router /
// combine kernels.
// The weight-gradient GEMMs' K-major operands are transposed copies of token rows in the
// send layout, [features][the 64-row blocks of every expert in turn] with this many
// columns (zero past each segment).
int64_t wgrad_t_cols(const LayerDims &d);
// dgrad-down writes dgu rows and (w a)^T in that transposed layout.
cudaError_t launch_tc_dgrad_down(const LayerDims &d, const void *dout_send, const int32_t *eoff,
                                 const void *w_down, const void *gu, const int32_t *perm,
                                 const float *topk_w, void *dgu, void *waT, float *dweight_part,
                                 int32_t *status, cudaStream_t s);
cudaError_t launch_tc_dgrad_gate_up(const LayerDims &d, const void *dgu, const int32_t *eoff,
                                    const void *packed, const int32_t *perm, void *dx_slots,
                                    int32_t *status, cudaStream_t s);
cudaError_t launch_tc_wgrad_gate_up(const LayerDims &d, const void *dgu, const void *xT,
                                    const int32_t *eoff, void *dw_gate, void *dw_up,
                                    int32_t *status, cudaStream_t s);
cudaError_t launch_tc_wgrad_down(const LayerDims &d, const void *dout_send, const void *waT,
                                 const int32_t *eoff, void *dw_down, int32_t *status,
                                 cudaStream_t s);
// x^T in the weight-gradient layout (ldt = wgrad_t_cols) from x [N, H] and perm; also zeroes
// rows [A, A + 64) of z0 [N*k, z0_cols] and z1 [N*k, z1_cols] (A = the kept rows).
cudaError_t launch_transpose_rows(const LayerDims &d, const void *src, const int32_t *eoff,
                                  const int32_t *perm, void *dstT, int64_t ldt, void *z0, int z0_cols,
                                  void *z1, int z1_cols, cudaStream_t s);
cudaError_t launch_simt_dgrad_down(const LayerDims &d, const float *dout_send, const int32_t *eoff,
                                   const float *w_down, const float *gu, const int32_t *perm,
                                   const float *topk_w, float *dgu, float *wa, float *dweight_part,
                                   cudaStream_t s);
cudaError_t launch_simt_dgrad_gate_up(const LayerDims &d, const float *dgu, const int32_t *eoff,
                                      const float *packed, const int32_t *perm, float *dx_slots,
                                      cudaStream_t s);
cudaError_t launch_simt_wgrad_gate_up(const LayerDims &d, const float *dgu, const float *send,
                                      const int32_t *eoff, float *dw_gate, float *dw_up,
                                      cudaStream_t s);
cudaError_t launch_simt_wgrad_down(const LayerDims &d, const float *dout_send, const float *wa,
                                   const int32_t *eoff, float *dw_down, cudaStream_t s);
int router_wgrad_splits(const LayerDims &d);
cudaError_t launch_router_dl(const LayerDims &d, const float *dweight_part, int m_tiles,
                             const int32_t *slot_pos, const float *topk_w, float *dl,
                             cudaStream_t s);
cudaError_t launch_dx_combine(const LayerDims &d, const void *dx_slots, const int32_t *slot_pos,
                              const int32_t *topk_idx, const float *dl, const void *w_router,
                              void *dx, cudaStream_t s);
cudaError_t launch_router_wgrad(const LayerDims &d, const int32_t *eoff_all, const int32_t *perm_all,
                                const float *dl, const void *x, float *partial, float *partial_db,
                                float *dw_router, float *db_router, cudaStream_t s);
cudaError_t launch_balance_stats(const LayerDims &d, const float *logits,
                                 const int32_t *routed_counts, float *partials, float *load_frac,
                                 float *prob_mean, cudaStream_t s);
cudaError_t launch_tp_reduce(const LayerDims &d, int tp_size, const void *padded, void *out,
                             cudaStream_t s);

// fp32 FFMA grouped FFN.
cudaError_t launch_simt_gate_up(const LayerDims &d, const float *send,
                                const int32_t *expert_offsets, int e_begin, int e_end,
                                const float *packed, float *h, float *gu /* [N*k, 2 Ipad] or nullptr */,
                                cudaStream_t s);
cudaError_t launch_simt_down(const LayerDims &d, const float *h, const int32_t *expert_offsets,
                             int e_begin, int e_end, const float *w_down, const int32_t *perm,
                             const float *topk_w, float *out_slots, cudaStream_t s);

cudaError_t launch_combine(const LayerDims &d, const void *out_slots, const int32_t *slot_pos,
                           void *out, cudaStream_t s);
cudaError_t launch_mask_sum(const LayerDims &d, const void *out_slots, const int32_t *topk_idx,
                            const int32_t *slot_pos, void *out, cudaStream_t s);

}  // namespace moe

namespace moe {

// Grouped-GEMM tile scheduling over variable-length expert segments.
// mtp[i] (i in [0, ne]) = number of BM-row tiles of experts e_begin .. e_begin+i-1 and
// eo[i] = expert_offsets[e_begin + i]; one warp builds both in shared memory.
__device__ inline void build_tile_tables(const int32_t *__restrict__ expert_offsets, int e_begin,
                                         int ne, int bm, int *eo, int *mtp) {
    const int lane = threadIdx.x & 31;
    const int per = (ne + 31) / 32;
    const int i0 = lane * per;
    int local = 0;
    for (int i = i0; i < i0 + per && i < ne; ++i) {
        const int a = expert_offsets[e_begin + i], b = expert_offsets[e_begin + i + 1];
        eo[i] = a;
        local += (b - a + bm - 1) / bm;
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int i = i0; i < i0 + per && i < ne; ++i) {
        mtp[i] = run;
        run += (expert_offsets[e_begin + i + 1] - expert_offsets[e_begin + i] + bm - 1) / bm;
    }
    if (lane == 31) {
        mtp[ne] = incl;
        eo[ne] = expert_offsets[e_begin + ne];
    }
}

// Tile t -> (expert index i in [0, ne), m tile, n tile). Tiles of one expert are ordered
// n-major with m fastest, so CTAs working at the same time share weight tiles in L2.
__device__ inline void decode_tile(int t, const int *mtp, int ne, int n_tiles, int &i, int &m,
                                   int &n) {
    int lo = 0, hi = ne - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mtp[mid] * n_tiles <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    i = lo;
    const int mt = mtp[lo + 1] - mtp[lo];
    const int local = t - mtp[lo] * n_tiles;
    n = local / mt;
    m = local - n * mt;
}

}  // namespace moe
