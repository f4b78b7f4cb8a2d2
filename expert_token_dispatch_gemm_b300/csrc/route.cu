// Step 1 -- routing: logits = x W_r^T (+ b), top-k with ties to the lower expert id,
// softmax over the k chosen logits, and the per-segment expert histogram that the
// dispatch scan consumes. (Ultralytics glossary "Expert Parallelism", section "How tokens
// move between GPUs", step 1 and its routing example.)
//
// One CTA of 256 threads routes kSegTokens = 64 tokens. The 64 x E logit tile is an
// FFMA register-blocked product over H in chunks staged through shared memory (each
// thread owns RT tokens x RE experts); logits stay on chip. One warp then selects each
// token's top-k by k rounds of a warp arg-max on (value desc, id asc).
// Exactness: products of the stored values are exact in fp32 and, for inputs on the
// dyadic grids of the exact test variant, every partial sum is too, so the chosen ids
// do not depend on the summation order.
#include <float.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;
// Hidden columns staged per step: wide for few experts (fewer load/barrier round trips),
// narrow for many (the expert tile grows with E).
__host__ __device__ constexpr int route_k_chunk(int ep) { return ep <= 16 ? 128 : 32; }

template <typename T, int RE, int EG>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const T *__restrict__ x, const T *__restrict__ wr, const float *__restrict__ bias,
             const float *__restrict__ sel_bias, int group_limit, int P, int N, int H, int E,
             int k, int32_t *__restrict__ topk_idx, float *__restrict__ topk_w,
             int32_t *__restrict__ seg_hist, float *__restrict__ logits_out) {
    grid_dep_wait();
    grid_dep_trigger();
    constexpr int TB = kSegTokens;
    constexpr int KC = route_k_chunk(RE * EG);
    constexpr int EP = RE * EG;               // experts padded to the thread layout
    constexpr int TGN = kRouteThreads / EG;   // token groups
    constexpr int RT = TB / TGN;              // tokens per thread
    static_assert(RT >= 1 && TB % TGN == 0, "thread layout");
    extern __shared__ float smem[];
    float *xs = smem;                    // [TB][KC+1]
    float *ws = xs + TB * (KC + 1);      // [EP][KC+1]
    __shared__ int hist_s[kMaxExperts];

    const int tid = threadIdx.x;
    const int eg = tid % EG, tg = tid / EG;
    const int t0 = blockIdx.x * TB;
    for (int e = tid; e < E; e += kRouteThreads) hist_s[e] = 0;

    float acc[RT][RE];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int q = 0; q < RE; ++q) acc[r][q] = 0.f;

    // Staging: every thread first issues all of its 16-byte loads of the chunk (x rows and
    // router rows; H is a multiple of 8, so a vector lies wholly inside or outside H),
    // then widens them into shared memory, so the loads' latencies overlap.
    using V = Vec16<T>;
    constexpr int XV = V::N;                               // elements per vector
    constexpr int CV = KC / XV;                            // vectors per staged row
    constexpr int XIT = TB * CV / kRouteThreads;           // x vectors per thread
    constexpr int WIT = (EP * CV + kRouteThreads - 1) / kRouteThreads;
    static_assert(TB * CV % kRouteThreads == 0, "x staging layout");
    for (int h0 = 0; h0 < H; h0 += KC) {
        uint4 xr[XIT], wv[WIT];
#pragma unroll
        for (int u = 0; u < XIT; ++u) {
            const int i = tid + u * kRouteThreads;
            const int r = i / CV, c = (i % CV) * XV, t = t0 + r, h = h0 + c;
            xr[u] = (t < N && h < H) ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * H + h))
                                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < WIT; ++u) {
            const int i = tid + u * kRouteThreads;
            const int r = i / CV, c = (i % CV) * XV, h = h0 + c;
            wv[u] = (i < EP * CV && r < E && h < H)
                        ? __ldg(reinterpret_cast<const uint4 *>(wr + (size_t)r * H + h))
                        : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < XIT; ++u) {
            const int i = tid + u * kRouteThreads;
            const int r = i / CV, c = (i % CV) * XV;
            float f[XV];
            V::to_float(xr[u], f);
#pragma unroll
            for (int q = 0; q < XV; ++q) xs[r * (KC + 1) + c + q] = f[q];
        }
#pragma unroll
        for (int u = 0; u < WIT; ++u) {
            const int i = tid + u * kRouteThreads;
            if (i < EP * CV) {
                const int r = i / CV, c = (i % CV) * XV;
                float f[XV];
                V::to_float(wv[u], f);
#pragma unroll
                for (int q = 0; q < XV; ++q) ws[r * (KC + 1) + c + q] = f[q];
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < KC; ++c) {
            float a[RT], b[RE];
#pragma unroll
            for (int r = 0; r < RT; ++r) a[r] = xs[(tg + r * TGN) * (KC + 1) + c];
#pragma unroll
            for (int q = 0; q < RE; ++q) b[q] = ws[(eg + q * EG) * (KC + 1) + c];
#pragma unroll
            for (int r = 0; r < RT; ++r)
#pragma unroll
                for (int q = 0; q < RE; ++q) acc[r][q] = fmaf(a[r], b[q], acc[r][q]);
        }
        __syncthreads();
    }

    // logits tile to shared memory (reuses the staging buffers)
    float *lg = smem;   // [TB][EP+1]
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int q = 0; q < RE; ++q) {
            const int e = eg + q * EG;
            float v = acc[r][q];
            if (bias != nullptr && e < E) v += bias[e];
            lg[(tg + r * TGN) * (EP + 1) + e] = v;
        }
    __syncthreads();
    if (logits_out != nullptr)   // optional copy for load statistics, coalesced
        for (int i = tid; i < TB * E; i += kRouteThreads) {
            const int r = i / E, e = i - r * E;
            if (t0 + r < N) logits_out[(size_t)(t0 + r) * E + e] = lg[r * (EP + 1) + e];
        }

    // top-k: one warp per token. Selection on logit + selection bias (a NaN ranks
    // last), optionally among the experts of the group_limit best partitions; the
    // weights are the softmax of the chosen experts' logits.
    constexpr int EPL = (EP + 31) / 32;
    const int warp = tid / 32, lane = tid % 32;
    const int per_part = E / P;
    for (int tl = warp; tl < TB; tl += kRouteThreads / 32) {
        const int t = t0 + tl;
        if (t >= N) break;
        float v[EPL], sv[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            const float l = (e < E) ? lg[tl * (EP + 1) + e] : -INFINITY;
            const float sc = (e < E && sel_bias != nullptr) ? l + sel_bias[e] : l;
            v[i] = isnan(l) ? -INFINITY : l;
            sv[i] = isnan(sc) ? -INFINITY : sc;
        }
        unsigned taken = 0;
        if (group_limit > 0) {
            // best selection score of partitions lane and lane + 32
            float pb[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pp = lane + 32 * h;
                if (pp < P)
                    for (int e = pp * per_part; e < (pp + 1) * per_part; ++e) {
                        const float l = lg[tl * (EP + 1) + e];
                        const float sc = sel_bias != nullptr ? l + sel_bias[e] : l;
                        if (!isnan(sc)) pb[h] = fmaxf(pb[h], sc);
                    }
            }
            // the group_limit best partitions (ties: lower id)
            unsigned long long kept = 0;
            for (int m = 0; m < group_limit; ++m) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int pp = lane + 32 * h;
                    if (pp < P && !((kept >> pp) & 1ull) && (pb[h] > bv || (pb[h] == bv && pp < bi))) {
                        bv = pb[h];
                        bi = pp;
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (ov > bv || (ov == bv && oi < bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                kept |= 1ull << bi;
            }
            // experts outside the kept partitions are never chosen
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((kept >> (e / per_part)) & 1ull)) taken |= 1u << i;
            }
        }
        float my_v = 0.f;
        int my_i = 0;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && (sv[i] > bv || (sv[i] == bv && e < bi))) {
                    bv = sv[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            // the chosen expert's logit, from the lane that holds it
            float bl = -INFINITY;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == bi) bl = v[i];
            bl = __shfl_sync(0xffffffffu, bl, bi & 31);
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) {
                my_v = bl;
                my_i = bi;
            }
        }
        // softmax over the chosen experts' logits
        float m = lane < k ? my_v : -INFINITY;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float ex = (lane < k) ? expf(my_v - m) : 0.f;
        float sum = ex;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane < k) {
            topk_idx[(size_t)t * k + lane] = my_i;
            topk_w[(size_t)t * k + lane] = ex / sum;
            atomicAdd(&hist_s[my_i], 1);
        }
    }
    if (seg_hist != nullptr) {
        __syncthreads();
        for (int e = tid; e < E; e += kRouteThreads) seg_hist[(size_t)blockIdx.x * E + e] = hist_s[e];
    }
}

template <typename T, int RE, int EG>
cudaError_t launch_route_t(const LayerDims &d, const T *x, const T *wr, const float *b,
                           int32_t *idx, float *w, int32_t *hist, float *lgo, cudaStream_t s) {
    constexpr int EP = RE * EG;
    const size_t stage = (size_t)(kSegTokens + EP) * (route_k_chunk(EP) + 1) * sizeof(float);
    const size_t logits = (size_t)kSegTokens * (EP + 1) * sizeof(float);
    const size_t smem = stage > logits ? stage : logits;
    auto kern = route_kernel<T, RE, EG>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    const int grid = ceil_div(d.N, kSegTokens);
    return launch_pdl(kern, dim3(grid), dim3(kRouteThreads), smem, s, x, wr, b, d.sel_bias,
                      d.group_limit, d.P, d.N, d.H, d.E, d.k, idx, w, hist, lgo);
}

template <typename T>
cudaError_t launch_route_dt(const LayerDims &d, const T *x, const T *wr, const float *b,
                            int32_t *idx, float *w, int32_t *hist, float *lgo, cudaStream_t s) {
    // experts per thread RE and expert groups EG, EP = RE*EG >= E
    if (d.E <= 4) return launch_route_t<T, 1, 4>(d, x, wr, b, idx, w, hist, lgo, s);
    if (d.E <= 8) return launch_route_t<T, 1, 8>(d, x, wr, b, idx, w, hist, lgo, s);
    if (d.E <= 16) return launch_route_t<T, 1, 16>(d, x, wr, b, idx, w, hist, lgo, s);
    if (d.E <= 32) return launch_route_t<T, 2, 16>(d, x, wr, b, idx, w, hist, lgo, s);
    if (d.E <= 64) return launch_route_t<T, 4, 16>(d, x, wr, b, idx, w, hist, lgo, s);
    if (d.E <= 128) return launch_route_t<T, 8, 16>(d, x, wr, b, idx, w, hist, lgo, s);
    return launch_route_t<T, 16, 16>(d, x, wr, b, idx, w, hist, lgo, s);
}

}  // namespace

cudaError_t launch_route(const LayerDims &d, const void *x, const void *w_router,
                         const float *b_router, int32_t *topk_idx, float *topk_w,
                         float *logits, int32_t *seg_hist, cudaStream_t s) {
    if (d.dtype == MOE_DTYPE_BF16)
        return launch_route_dt<__nv_bfloat16>(d, (const __nv_bfloat16 *)x,
                                              (const __nv_bfloat16 *)w_router, b_router,
                                              topk_idx, topk_w, seg_hist, logits, s);
    return launch_route_dt<float>(d, (const float *)x, (const float *)w_router, b_router,
                                  topk_idx, topk_w, seg_hist, logits, s);
}

}  // namespace moe
