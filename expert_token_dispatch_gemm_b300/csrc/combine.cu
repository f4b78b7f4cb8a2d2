// Step 4 -- combine, both forward rules, and the one-time gate/up weight packing.
//
// Dispatch rule (Ultralytics glossary "Expert Parallelism", step 4; Hugging Face
// "Expert parallelism" docs, "Token dispatch"): the expert outputs come back to their
// token already weighted (the down-projection epilogue wrote w * y into the pair's slot)
// and are summed in slot order.
// Mask-and-sum rule (Hugging Face docs, "DistributedConfig": "ep_router" masks the
// experts of other ranks, "moe_tp_experts" computes the local ones, an all-reduce sums
// the rank outputs): every partition forms its partial output from the slots whose
// expert it owns; the partials are then summed in partition order. An expert's slots
// are the same whichever launch computed them, so the experts run once for all
// partitions and the masking and the ordered sum happen here.
// Both kernels are one warp per token with 16-byte vector accesses: HBM-bound.
#include "common.cuh"

namespace moe {
namespace {

// Each lane sums two 16-byte vectors of the token's row per step and issues the loads
// of up to four slots for both before adding, so eight loads are in flight per lane;
// the adds still run in slot order.
template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const T *__restrict__ slots, const int32_t *__restrict__ slot_pos, int N, int k,
               int H, T *__restrict__ out) {
    grid_dep_wait();
    grid_dep_trigger();
    using V = Vec16<T>;
    constexpr int KU = 4, VU = 2;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * 8 + warp;
    if (t >= N) return;
    const unsigned kept = __ballot_sync(0xffffffffu, lane < k && slot_pos[(size_t)t * k + lane] >= 0);
    const int nvec = H / V::N;
    const uint4 *src = reinterpret_cast<const uint4 *>(slots + (size_t)t * k * H);
    uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)t * H);
    for (int v0 = lane; v0 < nvec; v0 += 32 * VU) {
        float acc[VU][V::N];
#pragma unroll
        for (int w = 0; w < VU; ++w)
#pragma unroll
            for (int i = 0; i < V::N; ++i) acc[w][i] = 0.f;
        for (int j0 = 0; j0 < k; j0 += KU) {
            uint4 r[KU][VU];
#pragma unroll
            for (int u = 0; u < KU; ++u)
#pragma unroll
                for (int w = 0; w < VU; ++w) {
                    const int j = j0 + u, v = v0 + 32 * w;
                    r[u][w] = (j < k && ((kept >> j) & 1u) && v < nvec)
                                  ? __ldg(src + (size_t)j * nvec + v)
                                  : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int u = 0; u < KU; ++u) {
                const int j = j0 + u;
                if (j < k && ((kept >> j) & 1u))
#pragma unroll
                    for (int w = 0; w < VU; ++w) {
                        float f[V::N];
                        V::to_float(r[u][w], f);
#pragma unroll
                        for (int i = 0; i < V::N; ++i) acc[w][i] += f[i];
                    }
            }
        }
#pragma unroll
        for (int w = 0; w < VU; ++w)
            if (v0 + 32 * w < nvec) dst[v0 + 32 * w] = V::from_float(acc[w]);
    }
}

// Mask-and-sum: partition p's partial output of token t is the fp32 sum, in slot order,
// of the slots whose expert partition p owns (the other partitions' experts are masked
// out); the partials are then added in partition order. Partials stay in registers.
//
// k <= KS (4 or 8): once per token, the kept slots in (partition, slot) order, packed four
// bits per entry, and a bit at every position that ends a partition's run. Each vector
// then runs one fixed sequence of adds: the slots in that order into the partition's
// partial, which is added to the sum where its run ends -- the same additions, in the
// same order, as summing each partition and then the partials. KS * VU loads are in
// flight per lane; four blocks of 256 threads fit on an SM.
template <typename T, int KS>
__global__ void __launch_bounds__(256, 4)
mask_sum_small_kernel(const T *__restrict__ slots, const int32_t *__restrict__ idx,
                      const int32_t *__restrict__ slot_pos, int N, int k, int H, int E, int P,
                      T *__restrict__ out) {
    grid_dep_wait();
    grid_dep_trigger();
    using V = Vec16<T>;
    constexpr int VU = KS == 4 ? 2 : 1;   // vectors per lane per step
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * 8 + warp;
    if (t >= N) return;
    const int per_part = E / P;
    int owner = -1;
    if (lane < k && slot_pos[(size_t)t * k + lane] >= 0) owner = idx[(size_t)t * k + lane] / per_part;
    const int nvec = H / V::N;
    const uint4 *src = reinterpret_cast<const uint4 *>(slots + (size_t)t * k * H);
    uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)t * H);
    // partitions that own at least one kept slot of this token, in increasing order; an
    // empty partition's partial is 0 and adding it leaves the sum unchanged
    unsigned todo = __ballot_sync(0xffffffffu, owner >= 0) & ((1u << k) - 1u);
    uint32_t order = 0, ends = 0;
    int nk = 0;
    while (todo) {
        int pmin = 0x7fffffff;
        for (unsigned m = todo; m; m &= m - 1) {
            const int o = __shfl_sync(0xffffffffu, owner, __ffs(m) - 1);
            pmin = o < pmin ? o : pmin;
        }
        const unsigned mine = __ballot_sync(0xffffffffu, owner == pmin) & todo;
        for (unsigned m = mine; m; m &= m - 1) {
            order |= (uint32_t)(__ffs(m) - 1) << (4 * nk);
            ++nk;
        }
        ends |= 1u << (nk - 1);
        todo &= ~mine;
    }
    for (int v0 = lane; v0 < nvec; v0 += 32 * VU) {
        uint4 r[KS][VU];
#pragma unroll
        for (int s = 0; s < KS; ++s)
#pragma unroll
            for (int w = 0; w < VU; ++w) {
                const int v = v0 + 32 * w;
                const int j = (int)((order >> (4 * s)) & 15u);
                r[s][w] = (s < nk && v < nvec) ? __ldg(src + (size_t)j * nvec + v)
                                                : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
        for (int w = 0; w < VU; ++w) {
            float acc[V::N], part[V::N];
#pragma unroll
            for (int i = 0; i < V::N; ++i) acc[i] = part[i] = 0.f;
#pragma unroll
            for (int s = 0; s < KS; ++s)
                if (s < nk) {
                    float f[V::N];
                    V::to_float(r[s][w], f);
#pragma unroll
                    for (int i = 0; i < V::N; ++i) part[i] += f[i];
                    if ((ends >> s) & 1u) {
#pragma unroll
                        for (int i = 0; i < V::N; ++i) {
                            acc[i] += part[i];
                            part[i] = 0.f;
                        }
                    }
                }
            if (v0 + 32 * w < nvec) dst[v0 + 32 * w] = V::from_float(acc);
        }
    }
}

// k > 8: the same sums. The (partition, slot) order is found once per token, with every
// lane of the warp in the ballots and shuffles, and kept in shared memory (up to 32
// entries); then each vector runs the same fixed sequence of adds as the small kernels.
template <typename T>
__global__ void __launch_bounds__(256)
mask_sum_kernel(const T *__restrict__ slots, const int32_t *__restrict__ idx,
                const int32_t *__restrict__ slot_pos, int N, int k, int H, int E, int P,
                T *__restrict__ out) {
    __shared__ int order_s[8][32];
    grid_dep_wait();
    grid_dep_trigger();
    using V = Vec16<T>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * 8 + warp;
    if (t >= N) return;
    const int per_part = E / P;
    int owner = -1;
    if (lane < k && slot_pos[(size_t)t * k + lane] >= 0) owner = idx[(size_t)t * k + lane] / per_part;
    const int nvec = H / V::N;
    const uint4 *src = reinterpret_cast<const uint4 *>(slots + (size_t)t * k * H);
    uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)t * H);
    unsigned todo = __ballot_sync(0xffffffffu, owner >= 0) & ((k < 32) ? ((1u << k) - 1u) : ~0u);
    uint32_t ends = 0;
    int nk = 0;
    while (todo) {
        // lowest partition among the remaining slots, its slots in slot order
        int pmin = 0x7fffffff;
        for (unsigned m = todo; m; m &= m - 1) {
            const int o = __shfl_sync(0xffffffffu, owner, __ffs(m) - 1);
            pmin = o < pmin ? o : pmin;
        }
        const unsigned mine = __ballot_sync(0xffffffffu, owner == pmin) & todo;
        for (unsigned m = mine; m; m &= m - 1) {
            if (lane == 0) order_s[warp][nk] = __ffs(m) - 1;
            ++nk;
        }
        ends |= 1u << (nk - 1);
        todo &= ~mine;
    }
    __syncwarp();
    for (int v = lane; v < nvec; v += 32) {
        float acc[V::N], part[V::N];
#pragma unroll
        for (int i = 0; i < V::N; ++i) acc[i] = part[i] = 0.f;
        for (int s = 0; s < nk; ++s) {
            float f[V::N];
            V::to_float(__ldg(src + (size_t)order_s[warp][s] * nvec + v), f);
#pragma unroll
            for (int i = 0; i < V::N; ++i) part[i] += f[i];
            if ((ends >> s) & 1u) {
#pragma unroll
                for (int i = 0; i < V::N; ++i) {
                    acc[i] += part[i];
                    part[i] = 0.f;
                }
            }
        }
        dst[v] = V::from_float(acc);
    }
}

// packed[e][r][:] for r in [0, 2*Ipad): block b = r / 256 holds gate rows 128b..128b+127
// then up rows 128b..128b+127; rows at or beyond I are zero.
template <typename T>
__global__ void pack_gate_up_kernel(const T *__restrict__ wg, const T *__restrict__ wu, int E,
                                    int I, int Ipad, int H, T *__restrict__ packed) {
    using V = Vec16<T>;
    const int nvec = H / V::N;
    const int64_t total = (int64_t)E * 2 * Ipad * nvec;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int v = (int)(i % nvec);
        const int64_t row = i / nvec;            // e * 2 * Ipad + r
        const int r = (int)(row % (2 * Ipad));
        const int e = (int)(row / (2 * Ipad));
        const int blk = r / (2 * kGateUpBlock), within = r % (2 * kGateUpBlock);
        const int src_row = blk * kGateUpBlock + within % kGateUpBlock;
        const T *src = within < kGateUpBlock ? wg : wu;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (src_row < I)
            val = reinterpret_cast<const uint4 *>(src + ((size_t)e * I + src_row) * H)[v];
        reinterpret_cast<uint4 *>(packed)[i] = val;
    }
}

}  // namespace

cudaError_t launch_combine(const LayerDims &d, const void *out_slots, const int32_t *slot_pos,
                           void *out, cudaStream_t s) {
    const int grid = ceil_div(d.N, 8);
    if (d.dtype == MOE_DTYPE_BF16)
        return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s,
                          (const __nv_bfloat16 *)out_slots, slot_pos, d.N, d.k, d.H,
                          (__nv_bfloat16 *)out);
    return launch_pdl(combine_kernel<float>, dim3(grid), dim3(256), 0, s, (const float *)out_slots,
                      slot_pos, d.N, d.k, d.H, (float *)out);
}

template <typename T>
cudaError_t launch_mask_sum_t(const LayerDims &d, const T *out_slots, const int32_t *topk_idx,
                              const int32_t *slot_pos, T *out, cudaStream_t s) {
    const int grid = ceil_div(d.N, 8);
    if (d.k <= 4)
        return launch_pdl(mask_sum_small_kernel<T, 4>, dim3(grid), dim3(256), 0, s, out_slots,
                          topk_idx, slot_pos, d.N, d.k, d.H, d.E, d.P, out);
    if (d.k <= 8)
        return launch_pdl(mask_sum_small_kernel<T, 8>, dim3(grid), dim3(256), 0, s, out_slots,
                          topk_idx, slot_pos, d.N, d.k, d.H, d.E, d.P, out);
    return launch_pdl(mask_sum_kernel<T>, dim3(grid), dim3(256), 0, s, out_slots, topk_idx,
                      slot_pos, d.N, d.k, d.H, d.E, d.P, out);
}

cudaError_t launch_mask_sum(const LayerDims &d, const void *out_slots, const int32_t *topk_idx,
                            const int32_t *slot_pos, void *out, cudaStream_t s) {
    if (d.dtype == MOE_DTYPE_BF16)
        return launch_mask_sum_t(d, (const __nv_bfloat16 *)out_slots, topk_idx, slot_pos,
                                 (__nv_bfloat16 *)out, s);
    return launch_mask_sum_t(d, (const float *)out_slots, topk_idx, slot_pos, (float *)out, s);
}

cudaError_t launch_pack_gate_up(const LayerDims &d, const void *w_gate, const void *w_up,
                                void *packed, cudaStream_t s) {
    const int64_t nvec = (int64_t)d.E * 2 * d.Ipad * d.H / (d.dtype == MOE_DTYPE_BF16 ? 8 : 4);
    const int grid = (int)std::min<int64_t>(ceil_div64(nvec, 256), 148 * 32);
    if (d.dtype == MOE_DTYPE_BF16)
        pack_gate_up_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            (const __nv_bfloat16 *)w_gate, (const __nv_bfloat16 *)w_up, d.E, d.I, d.Ipad, d.H,
            (__nv_bfloat16 *)packed);
    else
        pack_gate_up_kernel<float><<<grid, 256, 0, s>>>((const float *)w_gate, (const float *)w_up,
                                                        d.E, d.I, d.Ipad, d.H, (float *)packed);
    return cudaGetLastError();
}

}  // namespace moe
