// The C ABI declared in include/moe.h: argument validation (complete before anything is
// enqueued), workspace layout, and the launch sequence of each step and of the layer.
#include <limits.h>
#include <stdarg.h>
#include <math.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>
#include <string>

#include "common.cuh"

namespace moe {
namespace {

thread_local std::string g_last_error;

moe_status_t fail(moe_status_t s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
moe_status_t fail(moe_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

// The error is reported to the caller here; the runtime's last-error state is cleared
// (for a non-sticky error) so that it is not reported again by a later launch check.
moe_status_t cuda_fail(cudaError_t e, const char *what) {
    (void)cudaGetLastError();
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_CUDA(call, what)                                 \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(e_, (what)); \
    } while (0)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates the sizes and derives the kernel-side dimensions.
moe_status_t check_config(const moe_config *cfg, LayerDims *d) {
    if (cfg == nullptr) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
    const int64_t N = cfg->num_tokens, H = cfg->hidden, I = cfg->intermediate;
    if (N < 0) return fail(MOE_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)N);
    if (H < 8 || H % 8) return fail(MOE_ERR_INVALID_ARG, "hidden must be a positive multiple of 8 (got %lld)", (long long)H);
    if (I < 8 || I % 8) return fail(MOE_ERR_INVALID_ARG, "intermediate must be a positive multiple of 8 (got %lld)", (long long)I);
    if (cfg->num_experts < 1) return fail(MOE_ERR_INVALID_ARG, "num_experts must be >= 1");
    if (cfg->num_experts > kMaxExperts)
        return fail(MOE_ERR_UNSUPPORTED, "num_experts %d exceeds %d", cfg->num_experts, kMaxExperts);
    if (cfg->top_k < 1 || cfg->top_k > cfg->num_experts)
        return fail(MOE_ERR_INVALID_ARG, "top_k must be in [1, num_experts] (got %d)", cfg->top_k);
    if (cfg->top_k > kMaxTopK)
        return fail(MOE_ERR_UNSUPPORTED, "top_k %d exceeds %d", cfg->top_k, kMaxTopK);
    if (cfg->ep_size < 1 || cfg->num_experts % cfg->ep_size)
        return fail(MOE_ERR_INVALID_ARG, "ep_size (%d) must divide num_experts (%d)", cfg->ep_size,
                    cfg->num_experts);
    if (isnan(cfg->capacity_factor)) return fail(MOE_ERR_INVALID_ARG, "capacity_factor is NaN");
    if (cfg->mode != MOE_MODE_DISPATCH && cfg->mode != MOE_MODE_MASK_SUM)
        return fail(MOE_ERR_INVALID_ARG, "unknown mode %d", cfg->mode);
    if (cfg->dtype != MOE_DTYPE_BF16 && cfg->dtype != MOE_DTYPE_FP32)
        return fail(MOE_ERR_INVALID_ARG, "unknown dtype %d", cfg->dtype);
    if (cfg->has_bias != 0 && cfg->has_bias != 1) return fail(MOE_ERR_INVALID_ARG, "has_bias must be 0 or 1");
    const int64_t pairs = N * cfg->top_k;
    const int64_t Ipad = (I + kIpadAlign - 1) / kIpadAlign * kIpadAlign;
    if (pairs > INT_MAX / 2 || H > (1 << 20) || Ipad > (1 << 20) ||
        pairs * std::max(H, Ipad) > ((int64_t)1 << 40))
        return fail(MOE_ERR_UNSUPPORTED, "sizes too large for 32-bit row indices");
    d->N = (int)N;
    d->H = (int)H;
    d->I = (int)I;
    d->Ipad = (int)Ipad;
    d->E = cfg->num_experts;
    d->k = cfg->top_k;
    d->P = cfg->ep_size;
    d->dtype = cfg->dtype;
    d->capacity = INT_MAX;
    if (cfg->group_limit < 0)
        return fail(MOE_ERR_INVALID_ARG, "group_limit must be >= 0 (got %d)", cfg->group_limit);
    d->group_limit = cfg->group_limit < cfg->ep_size ? cfg->group_limit : 0;
    if (d->group_limit > 0) {
        if ((int64_t)d->group_limit * (cfg->num_experts / cfg->ep_size) < cfg->top_k)
            return fail(MOE_ERR_INVALID_ARG,
                        "group_limit %d partitions of %d experts hold fewer than top_k = %d",
                        d->group_limit, cfg->num_experts / cfg->ep_size, cfg->top_k);
        if (d->group_limit > kMaxGroupLimit || cfg->ep_size > kMaxGroupPartitions)
            return fail(MOE_ERR_UNSUPPORTED,
                        "group-limited routing supports group_limit <= %d and ep_size <= %d",
                        kMaxGroupLimit, kMaxGroupPartitions);
    }
    if (cfg->selection_bias != nullptr && (reinterpret_cast<uintptr_t>(cfg->selection_bias) & 3u))
        return fail(MOE_ERR_INVALID_ARG, "selection_bias must be 4-byte aligned");
    d->sel_bias = cfg->selection_bias;
    if (cfg->capacity_priority != MOE_PRIORITY_TOKEN && cfg->capacity_priority != MOE_PRIORITY_SLOT)
        return fail(MOE_ERR_INVALID_ARG, "unknown capacity_priority %d", cfg->capacity_priority);
    d->slot_priority = cfg->capacity_priority == MOE_PRIORITY_SLOT;
    if (cfg->training != 0 && cfg->training != 1) return fail(MOE_ERR_INVALID_ARG, "training must be 0 or 1");
    d->training = cfg->training;
    if (cfg->capacity_factor > 0.f) {
        // cf * N * k is exact in double (24-bit cf times an integer below 2^29); if the
        // exact quotient by E is an integer the division returns it exactly, otherwise it
        // lies at least 1/E from the next integer, far beyond the rounding error, so
        // ceil() of the double equals the exact ceiling.
        const double c = ceil((double)cfg->capacity_factor * (double)N * cfg->top_k / cfg->num_experts);
        d->capacity = c >= (double)N ? (N > 0 ? (int)N : 0) : (int)c;
        if (d->capacity < 1 && N > 0) d->capacity = 1;
    }
    return MOE_OK;
}

size_t esize(const LayerDims &d) { return d.dtype == MOE_DTYPE_BF16 ? 2 : 4; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace layout, every region 256-byte aligned.
struct Workspace {
    int32_t *status;       // [8]
    int32_t *seg_hist;     // [num_segments, E]
    float *stats;          // [kStatsBlocks, E]
    int32_t *topk_idx;     // [N*k]
    float *topk_w;         // [N*k]
    int32_t *routed;       // [E]
    int32_t *counts;       // [E]
    int32_t *eoff;         // [E+1]
    int32_t *poff;         // [P+1]
    int32_t *perm;         // [N*k]
    int32_t *slot_pos;     // [N*k]
    void *send;            // [N*k, H]
    void *h;               // [N*k, Ipad]
    void *slots;           // [N*k, H]; the backward's dx slots
    // training only: state kept by the forward, buffers of the backward
    void *gu;              // [N*k, 2 Ipad] gate / up pre-activations
    void *dout_send;       // [N*k, H]
    void *dgu;             // [N*k, 2 Ipad]
    float *dweight_part;   // [Ipad / 128, N*k]
    float *dl;             // [N*k]
    void *xT;              // bf16: [H, wgrad_t_cols] x rows transposed per expert
    void *waT;             // bf16: [Ipad, wgrad_t_cols] (w a) rows transposed per expert
    int32_t *routed_all, *counts_all, *eoff_all, *poff_all, *slot_all, *perm_all;
    float *rw_partial;     // [Z, E, H]
    float *rw_partial_db;  // [Z, E]
    size_t bytes;
};

Workspace carve(const LayerDims &d, int mode, void *base) {
    Workspace w = {};
    uint8_t *p = static_cast<uint8_t *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        void *r = p ? p + off : nullptr;
        off += align256(bytes);
        return r;
    };
    const size_t nseg = (size_t)num_segments(d);
    const size_t pairs = (size_t)d.N * d.k;
    w.status = (int32_t *)take(8 * sizeof(int32_t));
    w.seg_hist = (int32_t *)take(nseg * d.E * sizeof(int32_t));
    w.stats = (float *)take((size_t)kStatsBlocks * d.E * sizeof(float));
    w.topk_idx = (int32_t *)take(pairs * sizeof(int32_t));
    w.topk_w = (float *)take(pairs * sizeof(float));
    w.routed = (int32_t *)take(d.E * sizeof(int32_t));
    w.counts = (int32_t *)take(d.E * sizeof(int32_t));
    w.eoff = (int32_t *)take((d.E + 1) * sizeof(int32_t));
    w.poff = (int32_t *)take((d.P + 1) * sizeof(int32_t));
    w.perm = (int32_t *)take(pairs * sizeof(int32_t));
    w.slot_pos = (int32_t *)take(pairs * sizeof(int32_t));
    w.send = take(pairs * d.H * esize(d));
    w.h = take(pairs * d.Ipad * esize(d));
    w.slots = take(pairs * d.H * esize(d));
    if (d.training) {
        const size_t Z = (size_t)router_wgrad_splits(d);
        w.gu = take(pairs * 2 * d.Ipad * esize(d));
        w.dout_send = take(pairs * d.H * esize(d));
        w.dgu = take(pairs * 2 * d.Ipad * esize(d));
        w.dweight_part = (float *)take((size_t)(d.Ipad / 64) * pairs * sizeof(float));
        w.dl = (float *)take(pairs * sizeof(float));
        if (d.dtype == MOE_DTYPE_BF16) {
            w.xT = take((size_t)d.H * wgrad_t_cols(d) * esize(d));
            w.waT = take((size_t)d.Ipad * wgrad_t_cols(d) * esize(d));
        }
        w.routed_all = (int32_t *)take(d.E * sizeof(int32_t));
        w.counts_all = (int32_t *)take(d.E * sizeof(int32_t));
        w.eoff_all = (int32_t *)take((d.E + 1) * sizeof(int32_t));
        w.poff_all = (int32_t *)take((d.P + 1) * sizeof(int32_t));
        w.slot_all = (int32_t *)take(pairs * sizeof(int32_t));
        w.perm_all = (int32_t *)take(pairs * sizeof(int32_t));
        w.rw_partial = (float *)take(Z * d.E * d.H * sizeof(float));
        w.rw_partial_db = (float *)take(Z * d.E * sizeof(float));
    }
    w.bytes = off;
    return w;
}

moe_status_t check_workspace(const LayerDims &d, int mode, void *ws, size_t ws_bytes,
                             Workspace *out) {
    const Workspace need = carve(d, mode, nullptr);
    if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return fail(MOE_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need.bytes)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", ws_bytes, need.bytes);
    *out = carve(d, mode, ws);
    return MOE_OK;
}

moe_status_t need_ptr(const void *p, const char *name, bool vec) {
    if (p == nullptr) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
    if (vec && !aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s must be 16-byte aligned", name);
    return MOE_OK;
}
#define NEED(p, vec)                                    \
    do {                                                \
        moe_status_t s_ = need_ptr((p), #p, (vec));     \
        if (s_ != MOE_OK) return s_;                    \
    } while (0)

int num_sms() {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

// --------------------------------------------------------------- step bodies
// bf16 layers route on the tensor cores; fp32 layers on the FFMA router (single-pass
// TF32 would round the fp32 inputs). `hist` (may be null) receives the segment
// histogram, `logits` (may be null) the logits, `status` (may be null) the device
// status bits.
moe_status_t run_route(const LayerDims &d, const void *x, const void *wr, const float *b,
                       int32_t *idx, float *w, float *logits, int32_t *hist, int32_t *status,
                       cudaStream_t s) {
    if (d.dtype == MOE_DTYPE_BF16)
        MOE_CUDA(launch_tc_route(d, x, wr, b, idx, w, logits, hist, status, num_sms(), s),
                 "tensor-core route kernel");
    else
        MOE_CUDA(launch_route(d, x, wr, b, idx, w, logits, hist, s), "route kernel");
    return MOE_OK;
}

moe_status_t run_dispatch_from_hist(const LayerDims &d, const int32_t *idx, const void *x,
                                    const Workspace &w, int32_t *routed, int32_t *counts,
                                    int32_t *eoff, int32_t *poff, int32_t *perm, int32_t *slot_pos,
                                    void *send, cudaStream_t s) {
    MOE_CUDA(launch_scan_assign(d, idx, w.seg_hist, routed, counts, eoff, poff, slot_pos, perm,
                                w.status, s),
             "scan/assign kernel");
    MOE_CUDA(launch_permute(d, x, slot_pos, send, s), "permute kernel");
    return MOE_OK;
}

moe_status_t run_gate_up(const LayerDims &d, const void *send, const int32_t *eoff, int e0, int e1,
                         const void *packed, const Workspace &w, cudaStream_t s, void *gu = nullptr) {
    if (d.dtype == MOE_DTYPE_BF16)
        MOE_CUDA(launch_tc_gate_up(d, send, eoff, e0, e1, packed, w.h, gu, w.status, num_sms(), s),
                 "tensor-core gate/up kernel");
    else
        MOE_CUDA(launch_simt_gate_up(d, (const float *)send, eoff, e0, e1, (const float *)packed,
                                     (float *)w.h, (float *)gu, s),
                 "fp32 gate/up kernel");
    return MOE_OK;
}

moe_status_t run_down(const LayerDims &d, const int32_t *eoff, int e0, int e1, const void *wd,
                      const int32_t *perm, const float *tw, void *slots, const Workspace &w,
                      cudaStream_t s) {
    if (d.dtype == MOE_DTYPE_BF16)
        MOE_CUDA(launch_tc_down(d, w.h, eoff, e0, e1, wd, perm, tw, slots, w.status, num_sms(), s),
                 "tensor-core down kernel");
    else
        MOE_CUDA(launch_simt_down(d, (const float *)w.h, eoff, e0, e1, (const float *)wd, perm, tw,
                                  (float *)slots, s),
                 "fp32 down kernel");
    return MOE_OK;
}

moe_status_t run_experts(const LayerDims &d, const void *send, const int32_t *eoff, int e0, int e1,
                         const void *packed, const void *wd, const int32_t *perm, const float *tw,
                         void *slots, const Workspace &w, cudaStream_t s) {
    moe_status_t st = run_gate_up(d, send, eoff, e0, e1, packed, w, s);
    if (st != MOE_OK) return st;
    return run_down(d, eoff, e0, e1, wd, perm, tw, slots, w, s);
}

moe_status_t run_combine(const LayerDims &d, int mode, const void *slots, const int32_t *idx,
                         const int32_t *slot_pos, void *out, const Workspace &w, cudaStream_t s) {
    if (mode == MOE_MODE_DISPATCH) {
        MOE_CUDA(launch_combine(d, slots, slot_pos, out, s), "combine kernel");
    } else {
        MOE_CUDA(launch_mask_sum(d, slots, idx, slot_pos, out, s), "mask-and-sum kernel");
    }
    return MOE_OK;
}

// ---------------------------------------------------------------- no-allocation dispatch
// Scratch of moe_dispatch_noalloc: a status word (padded to 256 bytes), then the
// per-segment histograms, up to kNoAllocMaxSegExperts ints. Every GPU that loads the
// library holds this 1 MiB until the process exits.
constexpr int kNoAllocMaxSegExperts = 1 << 18;
constexpr int kNoAllocStatusInts = 64;
__device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocStatusInts + kNoAllocMaxSegExperts];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
int32_t *g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once per device
// (the array's name is only a host-side stand-in in host code).
moe_status_t noalloc_scratch(int32_t **out) {
    int dev = 0;
    MOE_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        MOE_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

namespace moe {
cudaError_t launch_wait_timeout_check(int32_t *status, cudaStream_t s);
}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    }
    return "MOE_ERR_UNKNOWN";
}

const char *moe_last_error(void) { return g_last_error.c_str(); }

moe_status_t moe_workspace_size(const moe_config *cfg, size_t *bytes) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    if (bytes == nullptr) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = carve(d, cfg->mode, nullptr).bytes;
    g_last_error.clear();
    return MOE_OK;
}

moe_status_t moe_packed_gate_up_size(const moe_config *cfg, size_t *bytes) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    if (bytes == nullptr) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = (size_t)d.E * 2 * d.Ipad * d.H * esize(d);
    g_last_error.clear();
    return MOE_OK;
}

moe_status_t moe_pack_weights(const moe_config *cfg, const void *w_gate, const void *w_up,
                              void *w_gate_up_packed, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    NEED(w_gate, true);
    NEED(w_up, true);
    NEED(w_gate_up_packed, true);
    g_last_error.clear();
    MOE_CUDA(launch_pack_gate_up(d, w_gate, w_up, w_gate_up_packed, (cudaStream_t)stream),
             "pack kernel");
    return MOE_OK;
}

moe_status_t moe_route(const moe_config *cfg, const void *x, const void *w_router,
                       const float *b_router, int32_t *topk_idx, float *topk_w, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    if (d.N == 0) return MOE_OK;
    NEED(x, true);
    NEED(w_router, true);
    if (cfg->has_bias) NEED(b_router, false);
    NEED(topk_idx, false);
    NEED(topk_w, false);
    g_last_error.clear();
    return run_route(d, x, w_router, cfg->has_bias ? b_router : nullptr, topk_idx, topk_w, nullptr,
                     nullptr, nullptr, (cudaStream_t)stream);
}

moe_status_t moe_update_selection_bias(const moe_config *cfg, const int32_t *routed_counts,
                                       float *selection_bias, float gamma, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    if (isnan(gamma) || isinf(gamma)) return fail(MOE_ERR_INVALID_ARG, "gamma must be finite");
    NEED(routed_counts, false);
    NEED(selection_bias, false);
    g_last_error.clear();
    MOE_CUDA(launch_update_selection_bias(d, routed_counts, selection_bias, gamma,
                                          (cudaStream_t)stream),
             "selection bias update kernel");
    return MOE_OK;
}

moe_status_t moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                          int32_t *routed_counts, int32_t *counts, int32_t *expert_offsets,
                          int32_t *part_offsets, int32_t *perm, int32_t *slot_pos, void *send,
                          void *workspace, size_t workspace_bytes, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    NEED(routed_counts, false);
    NEED(counts, false);
    NEED(expert_offsets, false);
    NEED(part_offsets, false);
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (d.N == 0) {   // empty batch: zero counts and offsets, nothing else
        MOE_CUDA(cudaMemsetAsync(routed_counts, 0, d.E * sizeof(int32_t), s), "memset");
        MOE_CUDA(cudaMemsetAsync(counts, 0, d.E * sizeof(int32_t), s), "memset");
        MOE_CUDA(cudaMemsetAsync(expert_offsets, 0, (d.E + 1) * sizeof(int32_t), s), "memset");
        MOE_CUDA(cudaMemsetAsync(part_offsets, 0, (d.P + 1) * sizeof(int32_t), s), "memset");
        return MOE_OK;
    }
    NEED(topk_idx, false);
    NEED(x, true);
    NEED(perm, false);
    NEED(slot_pos, false);
    NEED(send, true);
    g_last_error.clear();
    MOE_CUDA(launch_histogram(d, topk_idx, w.seg_hist, w.status, s), "histogram kernel");
    return run_dispatch_from_hist(d, topk_idx, x, w, routed_counts, counts, expert_offsets,
                                  part_offsets, perm, slot_pos, send, s);
}

moe_status_t moe_expert_ffn(const moe_config *cfg, const void *send, const int32_t *expert_offsets,
                            int32_t expert_begin, int32_t expert_end, const void *w_gate_up_packed,
                            const void *w_down, const int32_t *perm, const float *topk_w,
                            void *out_slots, void *workspace, size_t workspace_bytes, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    if (expert_begin < 0 || expert_end > d.E || expert_begin >= expert_end)
        return fail(MOE_ERR_INVALID_ARG, "expert range [%d, %d) not inside [0, %d)", expert_begin,
                    expert_end, d.E);
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    if (d.N == 0) return MOE_OK;
    NEED(send, true);
    NEED(expert_offsets, false);
    NEED(w_gate_up_packed, true);
    NEED(w_down, true);
    NEED(perm, false);
    NEED(topk_w, false);
    NEED(out_slots, true);
    g_last_error.clear();
    return run_experts(d, send, expert_offsets, expert_begin, expert_end, w_gate_up_packed, w_down,
                       perm, topk_w, out_slots, w, (cudaStream_t)stream);
}

moe_status_t moe_combine(const moe_config *cfg, const void *out_slots, const int32_t *topk_idx,
                         const int32_t *slot_pos, void *out, void *workspace,
                         size_t workspace_bytes, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    if (d.N == 0) return MOE_OK;
    NEED(out_slots, true);
    NEED(slot_pos, false);
    if (cfg->mode == MOE_MODE_MASK_SUM) NEED(topk_idx, false);
    NEED(out, true);
    g_last_error.clear();
    return run_combine(d, cfg->mode, out_slots, topk_idx, slot_pos, out, w, (cudaStream_t)stream);
}

moe_status_t moe_layer_forward(const moe_config *cfg, const void *x, const void *w_router,
                               const float *b_router, const void *w_gate_up_packed,
                               const void *w_down, void *out, const moe_diagnostics *diag,
                               void *workspace, size_t workspace_bytes, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    moe_diagnostics none = {};
    const moe_diagnostics &g = diag ? *diag : none;
    // training: the routing state stays in the workspace for the backward and is copied
    // to the requested diagnostic buffers at the end
    const bool own = !d.training;
    int32_t *idx = own && g.topk_idx ? g.topk_idx : w.topk_idx;
    float *tw = own && g.topk_w ? g.topk_w : w.topk_w;
    int32_t *routed = own && g.routed_counts ? g.routed_counts : w.routed;
    int32_t *counts = own && g.counts ? g.counts : w.counts;
    int32_t *eoff = own && g.expert_offsets ? g.expert_offsets : w.eoff;
    int32_t *poff = own && g.part_offsets ? g.part_offsets : w.poff;
    int32_t *perm = own && g.perm ? g.perm : w.perm;
    int32_t *slot_pos = own && g.slot_pos ? g.slot_pos : w.slot_pos;
    if (d.N == 0) {
        g_last_error.clear();
        if (g.routed_counts) MOE_CUDA(cudaMemsetAsync(g.routed_counts, 0, d.E * 4, s), "memset");
        if (g.counts) MOE_CUDA(cudaMemsetAsync(g.counts, 0, d.E * 4, s), "memset");
        if (g.expert_offsets) MOE_CUDA(cudaMemsetAsync(g.expert_offsets, 0, (d.E + 1) * 4, s), "memset");
        if (g.part_offsets) MOE_CUDA(cudaMemsetAsync(g.part_offsets, 0, (d.P + 1) * 4, s), "memset");
        return MOE_OK;
    }
    NEED(x, true);
    NEED(w_router, true);
    if (cfg->has_bias) NEED(b_router, false);
    NEED(w_gate_up_packed, true);
    NEED(w_down, true);
    NEED(out, true);
    g_last_error.clear();
    void *const *ev = g.stage_events;
    auto mark = [&](int stage) -> moe_status_t {
        if (ev == nullptr) return MOE_OK;
        MOE_CUDA(cudaEventRecord((cudaEvent_t)ev[stage], s), "stage event record");
        return MOE_OK;
    };
#define MOE_MARK(i)                 \
    do {                            \
        st = mark(i);               \
        if (st != MOE_OK) return st; \
    } while (0)

    if (g.router_logits) NEED(g.router_logits, true);
    MOE_MARK(MOE_STAGE_ROUTE);
    // slot-major priority ranks pairs in another order than the router's per-token
    // segment histogram: its histograms come from the histogram kernel instead
    st = run_route(d, x, w_router, cfg->has_bias ? b_router : nullptr, idx, tw, g.router_logits,
                   d.slot_priority ? nullptr : w.seg_hist, w.status, s);
    if (st != MOE_OK) return st;
    MOE_MARK(MOE_STAGE_SCAN);
    if (d.slot_priority)
        MOE_CUDA(launch_histogram(d, idx, w.seg_hist, w.status, s), "histogram kernel");
    MOE_CUDA(launch_scan_assign(d, idx, w.seg_hist, routed, counts, eoff, poff, slot_pos, perm,
                                w.status, s),
             "scan/assign kernel");
    MOE_MARK(MOE_STAGE_ASSIGN);   // fused into the scan stage's kernel
    MOE_MARK(MOE_STAGE_PERMUTE);
    MOE_CUDA(launch_permute(d, x, slot_pos, w.send, s), "permute kernel");
    MOE_MARK(MOE_STAGE_GATE_UP);
    // Both forward rules run every partition's experts in one launch per GEMM: an
    // expert's rows never share a tile with another expert's, so its outputs are the
    // same as if its partition ran it alone.
    st = run_gate_up(d, w.send, eoff, 0, d.E, w_gate_up_packed, w, s, d.training ? w.gu : nullptr);
    if (st != MOE_OK) return st;
    MOE_MARK(MOE_STAGE_DOWN);
    st = run_down(d, eoff, 0, d.E, w_down, perm, tw, w.slots, w, s);
    if (st != MOE_OK) return st;
    MOE_MARK(MOE_STAGE_COMBINE);
    st = run_combine(d, cfg->mode, w.slots, idx, slot_pos, out, w, s);
    if (st != MOE_OK) return st;
    MOE_MARK(MOE_NUM_STAGES);
#undef MOE_MARK
    if (d.training) {
        const size_t pairs = (size_t)d.N * d.k;
        auto copy = [&](void *dst, const void *src, size_t bytes) -> moe_status_t {
            if (dst != nullptr)
                MOE_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s), "diagnostic copy");
            return MOE_OK;
        };
        const moe_status_t c[8] = {
            copy(g.topk_idx, idx, pairs * 4), copy(g.topk_w, tw, pairs * 4),
            copy(g.routed_counts, routed, d.E * 4), copy(g.counts, counts, d.E * 4),
            copy(g.expert_offsets, eoff, (d.E + 1) * 4), copy(g.part_offsets, poff, (d.P + 1) * 4),
            copy(g.perm, perm, pairs * 4), copy(g.slot_pos, slot_pos, pairs * 4)};
        for (moe_status_t x : c)
            if (x != MOE_OK) return x;
    }
    return MOE_OK;
}

moe_status_t moe_read_device_status(const moe_config *cfg, void *workspace, size_t workspace_bytes,
                                    int32_t *flags, int32_t reset, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    if (flags == nullptr) return fail(MOE_ERR_INVALID_ARG, "flags is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    int32_t v = 0;
    MOE_CUDA(cudaMemcpyAsync(&v, w.status, sizeof v, cudaMemcpyDeviceToHost, s), "status read");
    MOE_CUDA(cudaStreamSynchronize(s), "stream sync");
    if (reset) {
        MOE_CUDA(cudaMemsetAsync(w.status, 0, sizeof v, s), "status reset");
        MOE_CUDA(cudaStreamSynchronize(s), "stream sync");
    }
    *flags = v;
    g_last_error.clear();
    if (v & MOE_DEV_TIMEOUT) return fail(MOE_ERR_TIMEOUT, "a device-side wait timed out");
    return MOE_OK;
}

moe_status_t moe_dispatch_noalloc(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                                  int32_t *routed_counts, int32_t *counts,
                                  int32_t *expert_offsets, int32_t *part_offsets, int32_t *perm,
                                  int32_t *slot_pos, void *send, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    const int64_t seg_experts = (int64_t)num_segments(d) * d.E;
    if (seg_experts > kNoAllocMaxSegExperts)
        return fail(MOE_ERR_UNSUPPORTED,
                    "moe_dispatch_noalloc: %lld histogram segments x num_experts = %lld exceeds "
                    "its fixed scratch of %d; use moe_dispatch with a workspace",
                    (long long)num_segments(d), (long long)seg_experts, kNoAllocMaxSegExperts);
    NEED(routed_counts, false);
    NEED(counts, false);
    NEED(expert_offsets, false);
    NEED(part_offsets, false);
    if (d.N > 0) {
        NEED(topk_idx, false);
        NEED(x, true);
        NEED(perm, false);
        NEED(slot_pos, false);
        NEED(send, true);
    }
    int32_t *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != MOE_OK) return st;
    g_last_error.clear();
    cudaStream_t s = (cudaStream_t)stream;
    if (d.N == 0) {
        MOE_CUDA(cudaMemsetAsync(routed_counts, 0, d.E * sizeof(int32_t), s), "memset");
        MOE_CUDA(cudaMemsetAsync(counts, 0, d.E * sizeof(int32_t), s), "memset");
        MOE_CUDA(cudaMemsetAsync(expert_offsets, 0, (d.E + 1) * sizeof(int32_t), s), "memset");
        MOE_CUDA(cudaMemsetAsync(part_offsets, 0, (d.P + 1) * sizeof(int32_t), s), "memset");
        return MOE_OK;
    }
    // The histogram kernel writes every [segment, expert] entry, so only the status word
    // carries over from the previous call: clear it.
    int32_t *status = scratch;
    Workspace w = {};
    w.status = status;
    w.seg_hist = scratch + kNoAllocStatusInts;
    MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int32_t), s), "status reset");
    MOE_CUDA(launch_histogram(d, topk_idx, w.seg_hist, w.status, s), "histogram kernel");
    return run_dispatch_from_hist(d, topk_idx, x, w, routed_counts, counts, expert_offsets,
                                  part_offsets, perm, slot_pos, send, s);
}

moe_status_t moe_layer_backward(const moe_config *cfg, const void *x, const void *w_router,
                                const void *w_gate_up_packed, const void *w_down,
                                const void *dout, void *dx, float *dw_router, float *db_router,
                                void *dw_gate, void *dw_up, void *dw_down, void *workspace,
                                size_t workspace_bytes, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    if (!d.training)
        return fail(MOE_ERR_INVALID_ARG, "moe_layer_backward needs a config with training = 1");
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    NEED(dw_router, true);
    NEED(dw_gate, true);
    NEED(dw_up, true);
    NEED(dw_down, true);
    cudaStream_t s = (cudaStream_t)stream;
    g_last_error.clear();
    if (d.N == 0) {   // no tokens: every gradient is zero
        const size_t es = esize(d);
        MOE_CUDA(cudaMemsetAsync(dw_router, 0, (size_t)d.E * d.H * 4, s), "memset");
        if (db_router) MOE_CUDA(cudaMemsetAsync(db_router, 0, (size_t)d.E * 4, s), "memset");
        MOE_CUDA(cudaMemsetAsync(dw_gate, 0, (size_t)d.E * d.I * d.H * es, s), "memset");
        MOE_CUDA(cudaMemsetAsync(dw_up, 0, (size_t)d.E * d.I * d.H * es, s), "memset");
        MOE_CUDA(cudaMemsetAsync(dw_down, 0, (size_t)d.E * d.H * d.I * es, s), "memset");
        return MOE_OK;
    }
    NEED(x, true);
    NEED(w_router, true);
    NEED(w_gate_up_packed, true);
    NEED(w_down, true);
    NEED(dout, true);
    NEED(dx, true);
    // 1. the upstream gradient of every kept pair, in the send layout
    MOE_CUDA(launch_permute(d, dout, w.slot_pos, w.dout_send, s), "permute kernel");
    // 2. dgrad of the down projection with the SwiGLU backward: dgu, w*a, dweight parts
    // 3. dgrad of gate / up: every kept pair's dx into its slot
    // 4. weight gradients of the experts
    int dw_tiles;   // M tiles of the dweight partials
    if (d.dtype == MOE_DTYPE_BF16) {
        dw_tiles = d.Ipad / 128;
        // the weight-gradient GEMMs' K-major operands: x^T here, (w a)^T from dgrad-down;
        // the rows past the kept rows of their other operands (dgu, dout) are zeroed here
        MOE_CUDA(launch_transpose_rows(d, x, w.eoff, w.perm, w.xT, wgrad_t_cols(d), w.dgu,
                                       2 * d.Ipad, w.dout_send, d.H, s),
                 "transpose kernel");
        MOE_CUDA(launch_tc_dgrad_down(d, w.dout_send, w.eoff, w_down, w.gu, w.perm, w.topk_w,
                                      w.dgu, w.waT, w.dweight_part, w.status, s),
                 "tensor-core dgrad-down kernel");
        MOE_CUDA(launch_tc_dgrad_gate_up(d, w.dgu, w.eoff, w_gate_up_packed, w.perm, w.slots,
                                         w.status, s),
                 "tensor-core dgrad-gate/up kernel");
        MOE_CUDA(launch_tc_wgrad_gate_up(d, w.dgu, w.xT, w.eoff, dw_gate, dw_up, w.status, s),
                 "tensor-core wgrad-gate/up kernel");
        MOE_CUDA(launch_tc_wgrad_down(d, w.dout_send, w.waT, w.eoff, dw_down, w.status, s),
                 "tensor-core wgrad-down kernel");
    } else {
        dw_tiles = d.Ipad / 64;
        MOE_CUDA(launch_simt_dgrad_down(d, (const float *)w.dout_send, w.eoff, (const float *)w_down,
                                        (const float *)w.gu, w.perm, w.topk_w, (float *)w.dgu,
                                        (float *)w.h, w.dweight_part, s),
                 "fp32 dgrad-down kernel");
        MOE_CUDA(launch_simt_dgrad_gate_up(d, (const float *)w.dgu, w.eoff,
                                           (const float *)w_gate_up_packed, w.perm,
                                           (float *)w.slots, s),
                 "fp32 dgrad-gate/up kernel");
        MOE_CUDA(launch_simt_wgrad_gate_up(d, (const float *)w.dgu, (const float *)w.send, w.eoff,
                                           (float *)dw_gate, (float *)dw_up, s),
                 "fp32 wgrad-gate/up kernel");
        MOE_CUDA(launch_simt_wgrad_down(d, (const float *)w.dout_send, (const float *)w.h, w.eoff,
                                        (float *)dw_down, s),
                 "fp32 wgrad-down kernel");
    }
    // 5. routing-weight and logit gradients, dx
    MOE_CUDA(launch_router_dl(d, w.dweight_part, dw_tiles, w.slot_pos, w.topk_w, w.dl, s),
             "router logit-gradient kernel");
    MOE_CUDA(launch_dx_combine(d, w.slots, w.slot_pos, w.topk_idx, w.dl, w_router, dx, s),
             "dx combine kernel");
    // 6. router weight gradient over every routed pair (dropped ones too), grouped by
    //    expert in token order: the dispatch scan without a capacity
    LayerDims all = d;
    all.capacity = INT_MAX;
    all.slot_priority = 0;
    MOE_CUDA(launch_histogram(all, w.topk_idx, w.seg_hist, w.status, s), "histogram kernel");
    MOE_CUDA(launch_scan_assign(all, w.topk_idx, w.seg_hist, w.routed_all, w.counts_all, w.eoff_all,
                                w.poff_all, w.slot_all, w.perm_all, w.status, s),
             "scan/assign kernel");
    MOE_CUDA(launch_router_wgrad(d, w.eoff_all, w.perm_all, w.dl, x, w.rw_partial, w.rw_partial_db,
                                 dw_router, db_router, s),
             "router wgrad kernels");
    return MOE_OK;
}

moe_status_t moe_check_wait_timeout(const moe_config *cfg, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    g_last_error.clear();
    MOE_CUDA(launch_wait_timeout_check(w.status, (cudaStream_t)stream), "wait check kernel");
    return MOE_OK;
}

moe_status_t moe_balance_stats(const moe_config *cfg, const float *router_logits,
                               const int32_t *routed_counts, float *load_frac, float *prob_mean,
                               void *workspace, size_t workspace_bytes, void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    Workspace w;
    st = check_workspace(d, cfg->mode, workspace, workspace_bytes, &w);
    if (st != MOE_OK) return st;
    NEED(routed_counts, false);
    NEED(load_frac, false);
    NEED(prob_mean, false);
    cudaStream_t s = (cudaStream_t)stream;
    g_last_error.clear();
    if (d.N == 0) {   // no tokens: both statistics are zero
        MOE_CUDA(cudaMemsetAsync(load_frac, 0, d.E * sizeof(float), s), "memset");
        MOE_CUDA(cudaMemsetAsync(prob_mean, 0, d.E * sizeof(float), s), "memset");
        return MOE_OK;
    }
    NEED(router_logits, false);
    MOE_CUDA(launch_balance_stats(d, router_logits, routed_counts, w.stats, load_frac, prob_mean, s),
             "balance statistics kernels");
    return MOE_OK;
}

moe_status_t moe_tp_slice(int64_t num_tokens, int32_t tp_size, int32_t tp_rank, int64_t *begin,
                          int64_t *end) {
    if (num_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "num_tokens must be >= 0");
    if (tp_size < 1) return fail(MOE_ERR_INVALID_ARG, "tp_size must be >= 1 (got %d)", tp_size);
    if (tp_rank < 0 || tp_rank >= tp_size)
        return fail(MOE_ERR_INVALID_ARG, "tp_rank %d not in [0, %d)", tp_rank, tp_size);
    if (begin == nullptr || end == nullptr) return fail(MOE_ERR_INVALID_ARG, "begin/end is NULL");
    const int64_t q = num_tokens / tp_size, r = num_tokens % tp_size;
    *begin = tp_rank * q + std::min<int64_t>(tp_rank, r);
    *end = *begin + q + (tp_rank < r ? 1 : 0);
    g_last_error.clear();
    return MOE_OK;
}

moe_status_t moe_tp_reduce(const moe_config *cfg, int32_t tp_size, const void *padded, void *out,
                           void *stream) {
    LayerDims d;
    moe_status_t st = check_config(cfg, &d);
    if (st != MOE_OK) return st;
    if (tp_size < 1) return fail(MOE_ERR_INVALID_ARG, "tp_size must be >= 1 (got %d)", tp_size);
    if (d.N == 0) return MOE_OK;
    NEED(padded, true);
    NEED(out, true);
    g_last_error.clear();
    MOE_CUDA(launch_tp_reduce(d, tp_size, padded, out, (cudaStream_t)stream), "TP reduce kernel");
    return MOE_OK;
}

}  // extern "C"
