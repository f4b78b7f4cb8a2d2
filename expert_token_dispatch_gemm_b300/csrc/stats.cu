// Router load statistics and the TP row split's output reduction.
//
// Load statistics (Ultralytics glossary "Expert Parallelism", section "Load balancing and
// capacity": an auxiliary loss term pushes the router towards an even spread of tokens;
// the page names no formula, so the library returns the two per-expert quantities such a
// term is built from, not a loss):
//   load_frac[e] = routed_counts[e] / (N k)
//   prob_mean[e] = (1/N) sum_t softmax(logits[t])[e]   (softmax over all E experts)
// The token sum is deterministic: block b adds its contiguous token range in a fixed
// order (warp w takes every 8th token, the warps' sums are then added in warp order),
// and one block adds the blocks' partial sums in block order.
//
// TP row split (Hugging Face docs "Expert parallelism", section "With tensor
// parallelism"): each TP rank dispatches a disjoint slice of the shared batch and an
// all-reduce over the group of the zero-padded slice outputs restores the whole output.
// On one device the all-reduce is the ordered sum out = padded[0] + ... + padded[tp-1],
// accumulated in fp32.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxExpertsPerLane = (kMaxExperts + 31) / 32;

__global__ void __launch_bounds__(256)
balance_partials_kernel(const float *__restrict__ logits, int N, int E, int chunk,
                        float *__restrict__ partials) {
    grid_dep_wait();
    grid_dep_trigger();
    __shared__ float warp_sum[8][kMaxExperts];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t0 = blockIdx.x * chunk, t1 = min(N, t0 + chunk);
    float acc[kMaxExpertsPerLane];
#pragma unroll
    for (int i = 0; i < kMaxExpertsPerLane; ++i) acc[i] = 0.f;
    for (int t = t0 + warp; t < t1; t += 8) {
        const float *row = logits + (size_t)t * E;
        float v[kMaxExpertsPerLane];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMaxExpertsPerLane; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? row[e] : -INFINITY;
            m = fmaxf(m, v[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxExpertsPerLane; ++i) {
            v[i] = lane + 32 * i < E ? expf(v[i] - m) : 0.f;
            z += v[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        const float inv = 1.0f / z;
#pragma unroll
        for (int i = 0; i < kMaxExpertsPerLane; ++i) acc[i] += v[i] * inv;
    }
#pragma unroll
    for (int i = 0; i < kMaxExpertsPerLane; ++i)
        if (lane + 32 * i < E) warp_sum[warp][lane + 32 * i] = acc[i];
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += 256) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += warp_sum[w][e];
        partials[(size_t)blockIdx.x * E + e] = s;
    }
}

__global__ void __launch_bounds__(256)
balance_final_kernel(const float *__restrict__ partials, int nblocks, int N, int k, int E,
                     const int32_t *__restrict__ routed, float *__restrict__ load_frac,
                     float *__restrict__ prob_mean) {
    grid_dep_wait();
    grid_dep_trigger();
    for (int e = threadIdx.x; e < E; e += 256) {
        float s = 0.f;
        for (int b = 0; b < nblocks; ++b) s += partials[(size_t)b * E + e];
        prob_mean[e] = s / (float)N;
        load_frac[e] = (float)((double)routed[e] / ((double)N * k));
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
tp_reduce_kernel(const T *__restrict__ padded, size_t n_vec, size_t stride_vec, int tp,
                 T *__restrict__ out) {
    grid_dep_wait();
    grid_dep_trigger();
    constexpr int V = Vec16<T>::N;
    const uint4 *src = reinterpret_cast<const uint4 *>(padded);
    uint4 *dst = reinterpret_cast<uint4 *>(out);
    for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n_vec; i += (size_t)gridDim.x * 256) {
        float acc[V];
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] = 0.f;
        for (int s = 0; s < tp; ++s) {
            float f[V];
            Vec16<T>::to_float(__ldg(src + (size_t)s * stride_vec + i), f);
#pragma unroll
            for (int c = 0; c < V; ++c) acc[c] += f[c];
        }
        dst[i] = Vec16<T>::from_float(acc);
    }
}

}  // namespace

cudaError_t launch_balance_stats(const LayerDims &d, const float *logits,
                                 const int32_t *routed_counts, float *partials, float *load_frac,
                                 float *prob_mean, cudaStream_t s) {
    const int nblocks = std::max(1, std::min(kStatsBlocks, ceil_div(d.N, 32)));
    const int chunk = ceil_div(d.N, nblocks);
    cudaError_t e = launch_pdl(balance_partials_kernel, dim3(nblocks), dim3(256), 0, s, logits, d.N,
                               d.E, chunk, partials);
    if (e != cudaSuccess) return e;
    return launch_pdl(balance_final_kernel, dim3(1), dim3(256), 0, s, (const float *)partials,
                      nblocks, d.N, d.k, d.E, routed_counts, load_frac, prob_mean);
}

cudaError_t launch_tp_reduce(const LayerDims &d, int tp_size, const void *padded, void *out,
                             cudaStream_t s) {
    const size_t elems = (size_t)d.N * d.H;
    if (d.dtype == MOE_DTYPE_BF16) {
        const size_t nv = elems / 8;
        const int grid = (int)std::min<size_t>(std::max<size_t>(1, (nv + 255) / 256), 148 * 16);
        return launch_pdl(tp_reduce_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s,
                          (const __nv_bfloat16 *)padded, nv, nv, tp_size, (__nv_bfloat16 *)out);
    }
    const size_t nv = elems / 4;
    const int grid = (int)std::min<size_t>(std::max<size_t>(1, (nv + 255) / 256), 148 * 16);
    return launch_pdl(tp_reduce_kernel<float>, dim3(grid), dim3(256), 0, s, (const float *)padded, nv,
                      nv, tp_size, (float *)out);
}

}  // namespace moe
