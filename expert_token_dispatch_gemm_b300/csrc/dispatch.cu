// Step 2 -- dispatch: the send layout grouped by expert, hence by partition (experts are
// split contiguously: partition = expert / (E / ep_size)), and the copy of every kept
// pair's hidden state into it. (Hugging Face "Expert parallelism" docs, section "Token
// dispatch"; Ultralytics glossary "Expert Parallelism", step 2 and section "Load
// balancing and capacity".)
//
// Pair p = t*k + j. Its rank within expert e is the number of earlier pairs (lower token
// index) routed to e; with a capacity C the pair is kept iff rank < C, and its send row
// is expert_offsets[e] + rank. The rank is computed without atomics on values:
//   1. per segment of kSegTokens tokens, a histogram of expert ids (fused into routing
//      for the whole layer, or histogram_kernel here);
//   2. one warp per segment (8 per CTA): each CTA sums the [segments x E] histogram
//      into the routed totals (hence kept counts, expert and partition offsets) and its
//      segments' bases (pairs of earlier segments per expert); the warp then walks its
//      pairs in order 32 at a time, and lanes holding the same expert find each other
//      with __match_any_sync, so a pair's rank is its segment base plus the number of
//      earlier pairs of that expert.
// Every step is deterministic, so counts, offsets, perm and slot_pos are bit-exact.
//
// Slot-major priority (GShard-style capacity, template SLOT): the pairs are ranked in
// the order j*N + t -- every token's first choice, then every token's second choice --
// and the same machinery runs over "virtual segments" of that order: segment v covers
// slot j = v / S of the tokens [s*64k, (s+1)*64k), s = v mod S, S = ceil(N / 64k), so
// a segment still holds at most 64k pairs. Its histograms come from histogram_kernel.
#include <limits.h>

#include "common.cuh"

namespace moe {
namespace {

// The pairs of segment v in priority order: count() of them, the i-th is pair(i).
template <bool SLOT>
struct SegWalk {
    int64_t p0;      // token order: first pair; slot order: first token
    int count;
    int k, j;
    __device__ SegWalk(int v, int N, int k_) : k(k_) {
        const int span = kSegTokens * k;
        if (SLOT) {
            const int S = (N + span - 1) / span;
            j = v / S;
            p0 = (int64_t)(v - j * S) * span;
            count = (int)min((int64_t)span, (int64_t)N - p0);
        } else {
            j = 0;
            p0 = (int64_t)v * span;
            count = (int)min((int64_t)span, (int64_t)N * k - p0);
        }
    }
    __device__ int64_t pair(int i) const { return SLOT ? (p0 + i) * k + j : p0 + i; }
};

template <bool SLOT>
__global__ void histogram_kernel(const int32_t *__restrict__ idx, int N, int k, int E,
                                 int32_t *__restrict__ seg_hist, int32_t *status) {
    grid_dep_wait();
    grid_dep_trigger();
    __shared__ int hs[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hs[e] = 0;
    __syncthreads();
    const SegWalk<SLOT> w(blockIdx.x, N, k);
    for (int i = threadIdx.x; i < w.count; i += blockDim.x) {
        const int e = idx[w.pair(i)];
        if (e >= 0 && e < E)
            atomicAdd(&hs[e], 1);
        else
            atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) seg_hist[(size_t)blockIdx.x * E + e] = hs[e];
}

// Counts, offsets and stable slots in one kernel: one warp per 64-token segment, 8 per
// CTA. Every CTA sums all segments' histograms (at most 256 x nseg ints, read from L2)
// into the experts' routed totals and its own segments' rank bases, derives the kept
// counts and the exclusive expert offsets, and assigns its segments' pairs exactly as
// the separate scan and assign kernels do; CTA 0 writes the counts and offsets.
template <bool SLOT>
__global__ void __launch_bounds__(256)
scan_assign_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ seg_hist, int N,
                   int nseg, int k, int E, int P, int capacity, int32_t *__restrict__ routed_counts,
                   int32_t *__restrict__ counts, int32_t *__restrict__ expert_offsets,
                   int32_t *__restrict__ part_offsets, int32_t *__restrict__ slot_pos,
                   int32_t *__restrict__ perm, int32_t *status) {
    grid_dep_wait();
    grid_dep_trigger();
    __shared__ int tot_s[kMaxExperts], before_s[kMaxExperts], off_s[kMaxExperts + 1];
    __shared__ int base_s[8][kMaxExperts];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int seg0 = blockIdx.x * 8;
    // routed totals and the counts of segments before this CTA's, per expert
    for (int e = tid; e < E; e += 256) {
        tot_s[e] = 0;
        before_s[e] = 0;
    }
    __syncthreads();
    if (E % 4 == 0) {
        // 16-byte loads of 4 experts; G threads per group of 4 experts, each with 8
        // rows in flight
        const int Q = E / 4, G = 256 / Q;
        const int q = tid % Q, g = tid / Q;
        if (g < G) {
            int4 tot = make_int4(0, 0, 0, 0), before = make_int4(0, 0, 0, 0);
            const int4 *h4 = reinterpret_cast<const int4 *>(seg_hist) + q;
            for (int b0 = g; b0 < nseg; b0 += 8 * G) {
                int4 h[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int b = b0 + u * G;
                    h[u] = b < nseg ? h4[(size_t)b * Q] : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    tot.x += h[u].x; tot.y += h[u].y; tot.z += h[u].z; tot.w += h[u].w;
                    if (b0 + u * G < seg0) {
                        before.x += h[u].x; before.y += h[u].y;
                        before.z += h[u].z; before.w += h[u].w;
                    }
                }
            }
            atomicAdd(&tot_s[4 * q], tot.x);
            atomicAdd(&tot_s[4 * q + 1], tot.y);
            atomicAdd(&tot_s[4 * q + 2], tot.z);
            atomicAdd(&tot_s[4 * q + 3], tot.w);
            atomicAdd(&before_s[4 * q], before.x);
            atomicAdd(&before_s[4 * q + 1], before.y);
            atomicAdd(&before_s[4 * q + 2], before.z);
            atomicAdd(&before_s[4 * q + 3], before.w);
        }
    } else {
        const int G = 256 / E > 0 ? 256 / E : 1;   // threads per expert
        const int e = tid % E, g = tid / E;
        if (g < G && tid < G * E) {
            int tot = 0, before = 0;
            for (int b = g; b < nseg; b += G) {
                const int h = seg_hist[(size_t)b * E + e];
                tot += h;
                if (b < seg0) before += h;
            }
            atomicAdd(&tot_s[e], tot);
            atomicAdd(&before_s[e], before);
        }
    }
    __syncthreads();
    // exclusive scan of the kept counts over experts (one warp, E/32 experts per lane)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int e0 = lane * per, e1 = min(e0 + per, E);
        int local = 0;
        for (int e = e0; e < e1; ++e) local += min(tot_s[e], capacity);
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int e = e0; e < e1; ++e) {
            off_s[e] = run;
            run += min(tot_s[e], capacity);
        }
        if (lane == 31) off_s[E] = incl;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = tid; e < E; e += 256) {
            routed_counts[e] = tot_s[e];
            counts[e] = min(tot_s[e], capacity);
            expert_offsets[e] = off_s[e];
        }
        if (tid == 0) expert_offsets[E] = off_s[E];
        if (tid <= P) part_offsets[tid] = off_s[tid * (E / P)];
    }
    // this warp's segment: rank base = pairs of earlier segments per expert
    const int seg = seg0 + warp;
    if (seg >= nseg) return;   // warp-uniform; no block-wide barrier follows
    int *base = base_s[warp];
    for (int e = lane; e < E; e += 32) {
        int b = before_s[e];
        for (int s2 = seg0; s2 < seg; ++s2) b += seg_hist[(size_t)s2 * E + e];
        base[e] = b;
    }
    __syncwarp();
    const SegWalk<SLOT> walk(seg, N, k);
    const unsigned lt_mask = (1u << lane) - 1u;
    // the expert ids of 8 rounds of 32 pairs are loaded first, so the loads' latencies
    // overlap instead of adding up round after round
    constexpr int PF = 8;
    for (int ic0 = 0; ic0 < walk.count; ic0 += 32 * PF) {
        int ev[PF];
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            const int ic = ic0 + 32 * u;
            ev[u] = ic + lane < walk.count ? idx[walk.pair(ic + lane)] : -1;
        }
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            const int ic = ic0 + 32 * u;
            if (ic >= walk.count) break;   // warp-uniform
            const bool live = ic + lane < walk.count;
            const int64_t p = live ? walk.pair(ic + lane) : 0;
            int e = ev[u];
            const bool valid = live && e >= 0 && e < E;
            if (live && !valid) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
            if (!valid) e = -1 - lane;   // unique key: never matches another lane
            const unsigned same = __match_any_sync(0xffffffffu, e);
            int rank = 0;
            if (valid) rank = base[e] + __popc(same & lt_mask);
            __syncwarp();
            // the lowest lane of each group advances that expert's running base
            if (valid && (same & lt_mask) == 0) base[e] += __popc(same);
            __syncwarp();
            if (live) {
                int slot = -1;
                if (valid && rank < capacity) {
                    slot = off_s[e] + rank;
                    perm[slot] = (int32_t)p;
                }
                slot_pos[p] = slot;
            }
        }
    }
}

// One warp per token: read the token's row once (16-byte vectors), write it to every
// kept slot. Stores of one instruction cover 512 contiguous bytes of one send row.
template <typename T>
__global__ void __launch_bounds__(256)
permute_kernel(const T *__restrict__ x, int N, int H, int k, const int32_t *__restrict__ slot_pos,
               T *__restrict__ send) {
    grid_dep_wait();
    grid_dep_trigger();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * 8 + warp;
    if (t >= N) return;
    const int my_slot = (lane < k) ? slot_pos[(size_t)t * k + lane] : -1;
    const int nvec = H / Vec16<T>::N;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    for (int v0 = 0; v0 < nvec; v0 += 32 * 4) {
        uint4 r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < nvec) r[u] = __ldg(src + v);
        }
        for (int j = 0; j < k; ++j) {
            const int slot = __shfl_sync(0xffffffffu, my_slot, j);
            if (slot < 0) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(send + (size_t)slot * H);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) dst[v] = r[u];
            }
        }
    }
}

// After-step update of the selection-only bias (Ultralytics glossary, "Load balancing
// and capacity"): an expert above the equal share N*k/E of the step's routed pairs is
// lowered by gamma, one below it raised, compared exactly as count*E against N*k.
__global__ void __launch_bounds__(256)
update_selection_bias_kernel(int E, long long share_num, const int32_t *__restrict__ counts,
                             float *__restrict__ bias, float gamma) {
    grid_dep_wait();
    grid_dep_trigger();
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
        const long long diff = (long long)counts[e] * E - share_num;
        const float b = bias[e];
        bias[e] = diff > 0 ? __fsub_rn(b, gamma) : diff < 0 ? __fadd_rn(b, gamma) : b;
    }
}

}  // namespace

cudaError_t launch_update_selection_bias(const LayerDims &d, const int32_t *routed_counts,
                                        float *selection_bias, float gamma, cudaStream_t s) {
    return launch_pdl(update_selection_bias_kernel, dim3(1), dim3(256), 0, s, d.E,
                      (long long)d.N * d.k, routed_counts, selection_bias, gamma);
}

int num_segments(const LayerDims &d) {
    if (d.slot_priority) return d.k * ceil_div(d.N, kSegTokens * d.k);
    return ceil_div(d.N, kSegTokens);
}

cudaError_t launch_histogram(const LayerDims &d, const int32_t *topk_idx, int32_t *seg_hist,
                             int32_t *status, cudaStream_t s) {
    const int nseg = num_segments(d);
    if (nseg == 0) return cudaSuccess;
    auto kern = d.slot_priority ? histogram_kernel<true> : histogram_kernel<false>;
    return launch_pdl(kern, dim3(nseg), dim3(256), 0, s, topk_idx, d.N, d.k, d.E, seg_hist, status);
}

cudaError_t launch_scan_assign(const LayerDims &d, const int32_t *topk_idx, const int32_t *seg_hist,
                               int32_t *routed_counts, int32_t *counts, int32_t *expert_offsets,
                               int32_t *part_offsets, int32_t *slot_pos, int32_t *perm,
                               int32_t *status, cudaStream_t s) {
    const int nseg = num_segments(d);
    auto kern = d.slot_priority ? scan_assign_kernel<true> : scan_assign_kernel<false>;
    return launch_pdl(kern, dim3(std::max(1, ceil_div(nseg, 8))), dim3(256), 0, s, topk_idx,
                      seg_hist, d.N, nseg, d.k, d.E, d.P, d.capacity, routed_counts, counts,
                      expert_offsets, part_offsets, slot_pos, perm, status);
}

cudaError_t launch_permute(const LayerDims &d, const void *x, const int32_t *slot_pos,
                           void *send, cudaStream_t s) {
    const int grid = ceil_div(d.N, 8);
    if (d.dtype == MOE_DTYPE_BF16)
        return launch_pdl(permute_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s,
                          (const __nv_bfloat16 *)x, d.N, d.H, d.k, slot_pos, (__nv_bfloat16 *)send);
    return launch_pdl(permute_kernel<float>, dim3(grid), dim3(256), 0, s, (const float *)x, d.N, d.H,
                      d.k, slot_pos, (float *)send);
}

}  // namespace moe
