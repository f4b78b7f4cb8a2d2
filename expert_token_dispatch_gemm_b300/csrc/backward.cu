// Backward of the router and of the combine step (the chain rule through step 1 and
// step 4 of the Ultralytics glossary "Expert Parallelism": the output is the routing-
// weighted sum of the experts' outputs, the weights a softmax over the chosen logits).
//
//   dweight[t, j] = <dout_t, y_tj> for a kept pair (summed from the per-M-tile partials
//                   of the dgrad-down epilogue, in tile order), 0 for a dropped one;
//   dl[t, j]      = w_tj (dweight_tj - sum_j' w_tj' dweight_tj')   (softmax Jacobian;
//                   a dropped pair's weight still enters the softmax, so it still gets
//                   a logit gradient);
//   dx[t]         = sum_j over kept pairs of dx_slots[t k + j] + sum_j dl_tj W_r[e_tj]
//                   (fp32, in slot order, then the router rows in slot order);
//   dW_r[e]       = sum over the pairs routed to e, in token order, of dl x_t;
//   db_r[e]       = sum of the same dl.
// The selection is piecewise constant, so the selection bias gets no gradient.
#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256)
router_dl_kernel(int N, int k, int m_tiles, int rows, const float *__restrict__ dweight_part,
                 const int32_t *__restrict__ slot_pos, const float *__restrict__ topk_w,
                 float *__restrict__ dl) {
    grid_dep_wait();
    grid_dep_trigger();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N) return;
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
        const size_t pr = (size_t)t * k + j;
        const int slot = slot_pos[pr];
        float dw = 0.f;
        if (slot >= 0)
            for (int f = 0; f < m_tiles; ++f) dw += dweight_part[(size_t)f * rows + slot];
        dl[pr] = dw;
        s = fmaf(topk_w[pr], dw, s);
    }
    for (int j = 0; j < k; ++j) {
        const size_t pr = (size_t)t * k + j;
        dl[pr] = topk_w[pr] * (dl[pr] - s);
    }
}

// One warp per token, 16-byte vectors (8 bf16 or 4 fp32).
template <typename T>
__global__ void __launch_bounds__(256)
dx_combine_kernel(const T *__restrict__ dx_slots, const int32_t *__restrict__ slot_pos,
                  const int32_t *__restrict__ topk_idx, const float *__restrict__ dl,
                  const T *__restrict__ w_router, int N, int H, int k, T *__restrict__ dx) {
    constexpr int V = Vec16<T>::N;
    // the token's slots, experts and logit gradients, shared by the warp's lanes (a lane
    // past the last vector of a row takes no part in the loop below)
    __shared__ int slot_s[8][32], e_s[8][32];
    __shared__ float dl_s[8][32];
    grid_dep_wait();
    grid_dep_trigger();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = blockIdx.x * 8 + warp;
    if (t >= N) return;
    if (lane < k) {
        slot_s[warp][lane] = slot_pos[(size_t)t * k + lane];
        e_s[warp][lane] = topk_idx[(size_t)t * k + lane];
        dl_s[warp][lane] = dl[(size_t)t * k + lane];
    }
    __syncwarp();
    const int nvec = H / V;
    // the vectors of four slots (then four router rows) are loaded before any is added,
    // so that their latencies overlap; the sums keep the slot order
    for (int v = lane; v < nvec; v += 32) {
        float acc[V] = {};
        for (int j0 = 0; j0 < k; j0 += 4) {
            uint4 r[4];
            bool live[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int slot = j0 + u < k ? slot_s[warp][j0 + u] : -1;
                live[u] = slot >= 0;
                r[u] = live[u] ? __ldg(reinterpret_cast<const uint4 *>(
                                           dx_slots + ((size_t)t * k + j0 + u) * H) + v)
                               : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (live[u]) {
                    float f[V];
                    Vec16<T>::to_float(r[u], f);
#pragma unroll
                    for (int c = 0; c < V; ++c) acc[c] += f[c];
                }
        }
        for (int j0 = 0; j0 < k; j0 += 4) {
            uint4 r[4];
            float c0[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool in = j0 + u < k;
                c0[u] = in ? dl_s[warp][j0 + u] : 0.f;
                r[u] = in ? __ldg(reinterpret_cast<const uint4 *>(w_router + (size_t)e_s[warp][j0 + u] * H) + v)
                          : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (j0 + u < k) {
                    float f[V];
                    Vec16<T>::to_float(r[u], f);
#pragma unroll
                    for (int c = 0; c < V; ++c) acc[c] = fmaf(c0[u], f[c], acc[c]);
                }
        }
        reinterpret_cast<uint4 *>(dx + (size_t)t * H)[v] = Vec16<T>::from_float(acc);
    }
}

// Block (expert e, column chunk of 2048, split z): the z-th contiguous part of e's
// routed pairs, in order; partial [Z, E, H] fp32, and the part's sum of dl. Each thread
// owns 8 columns.
template <typename T>
__global__ void __launch_bounds__(256)
router_wgrad_partial_kernel(const int32_t *__restrict__ eoff_all, const int32_t *__restrict__ perm_all,
                            const float *__restrict__ dl, const T *__restrict__ x, int H, int E,
                            int k, float *__restrict__ partial, float *__restrict__ partial_db) {
    grid_dep_wait();
    grid_dep_trigger();
    const int e = blockIdx.x, z = blockIdx.z, Z = gridDim.z;
    const int r0 = eoff_all[e], n = eoff_all[e + 1] - r0;
    const int a = r0 + (int)((int64_t)n * z / Z), b = r0 + (int)((int64_t)n * (z + 1) / Z);
    const int col = (blockIdx.y * 256 + threadIdx.x) * 8;
    float acc[8] = {};
    float db = 0.f;
    if (col < H) {
        for (int r = a; r < b; ++r) {
            const int pr = perm_all[r];
            const float c0 = dl[pr];
            float f[8];
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(pr / k) * H + col);
            Vec16<T>::to_float(__ldg(src), f);
            if (Vec16<T>::N == 4) Vec16<T>::to_float(__ldg(src + 1), f + 4);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = fmaf(c0, f[c], acc[c]);
            db += c0;
        }
        float *dst = partial + ((size_t)z * E + e) * H + col;
        *reinterpret_cast<float4 *>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4 *>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) partial_db[(size_t)z * E + e] = db;
}

__global__ void __launch_bounds__(256)
router_wgrad_reduce_kernel(const float *__restrict__ partial, const float *__restrict__ partial_db,
                           int Z, int E, int H, float *__restrict__ dw_router,
                           float *__restrict__ db_router) {
    grid_dep_wait();
    grid_dep_trigger();
    const size_t n = (size_t)E * H;
    for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (size_t)gridDim.x * 256) {
        float s = 0.f;
        for (int z = 0; z < Z; ++z) s += partial[(size_t)z * n + i];
        dw_router[i] = s;
    }
    if (db_router != nullptr && blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += 256) {
            float s = 0.f;
            for (int z = 0; z < Z; ++z) s += partial_db[(size_t)z * E + e];
            db_router[e] = s;
        }
}

// The expert-grouped rows of a token matrix, transposed into the K-major operand of the
// weight-gradient GEMMs: dstT[h][64 pk_e + j] = src[perm[eo_e + j] / k][h] for the j-th
// row of expert e's segment (pk_e = the 64-row blocks of the experts before e), zero for
// j in [seg_e, 64 ceil(seg_e / 64)), so that every K block of an expert is whole. One
// block per 64 columns of dstT (64 rows of one expert) and 512 of the hidden dimension,
// 128 at a time through a shared-memory tile. The blocks also zero rows
// [A, A + 64) (A = the kept rows) of two [rows, cols] buffers, which the same GEMMs read
// as their other operand in an expert's last K block.
__global__ void __launch_bounds__(256)
transpose_rows_kernel(const __nv_bfloat16 *__restrict__ src, int H, int k,
                      const int32_t *__restrict__ eoff, int E, const int32_t *__restrict__ perm,
                      __nv_bfloat16 *__restrict__ dstT, int64_t ldt, __nv_bfloat16 *z0, int z0_cols,
                      __nv_bfloat16 *z1, int z1_cols, int rows) {
    __shared__ int eo[kMaxExperts + 1], pk[kMaxExperts + 1];
    __shared__ int tok_s[64];
    // [row j][column h]; the 16-byte chunk of columns 8c .. 8c + 7 of row j is stored at
    // chunk c ^ (j / 8 % 8), so that the column reads below spread over the banks
    __shared__ __align__(16) __nv_bfloat16 tile[64][128];
    grid_dep_wait();
    grid_dep_trigger();
    const int tid = threadIdx.x;
    if (tid < 32) build_tile_tables(eoff, 0, E, 64, eo, pk);
    __syncthreads();
    // zero the rows past the kept rows (16-byte chunks spread over the whole grid)
    {
        const int64_t nthreads = (int64_t)gridDim.x * gridDim.y * blockDim.x;
        const int A = eo[E];
        const int64_t n0 = 64LL * (z0_cols / 8), n1 = 64LL * (z1_cols / 8);
        for (int64_t g = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + tid;
             g < n0 + n1; g += nthreads) {
            __nv_bfloat16 *z = g < n0 ? z0 : z1;
            const int cols = g < n0 ? z0_cols : z1_cols;
            const int64_t c = g < n0 ? g : g - n0;
            const int r = A + (int)(c / (cols / 8));
            if (z != nullptr && r < rows)
                *reinterpret_cast<uint4 *>(z + (size_t)r * cols + (c % (cols / 8)) * 8) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
    }
    const int cb = blockIdx.x;
    if (cb >= pk[E]) return;   // past the last expert's blocks
    int e, blk, unused;
    decode_tile(cb, pk, E, 1, e, blk, unused);
    const int seg = eo[e + 1] - eo[e];
    if (tid < 64) tok_s[tid] = blk * 64 + tid < seg ? perm[eo[e] + blk * 64 + tid] / k : -1;
    __syncthreads();
    for (int h0 = blockIdx.y * 512; h0 < min(H, (int)blockIdx.y * 512 + 512); h0 += 128) {
        // 64 rows x 128 columns of the source in 16-byte chunks; rows past the segment
        // are zero
        uint4 v[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = tid + 256 * it;
            const int j = c >> 4, hc = (c & 15) * 8;
            const int tok = tok_s[j];
            v[it] = make_uint4(0u, 0u, 0u, 0u);
            if (tok >= 0 && h0 + hc < H)
                v[it] = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)tok * H + h0 + hc));
        }
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = tid + 256 * it;
            const int j = c >> 4;
            *reinterpret_cast<uint4 *>(&tile[j][((c & 15) ^ ((j >> 3) & 7)) * 8]) = v[it];
        }
        __syncthreads();
        // 128 rows of dstT (columns h0 ..), each 64 columns = eight 16-byte chunks
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = tid + 256 * it;
            const int hh = c >> 3, jc = (c & 7) * 8;
            if (h0 + hh < H) {
                __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    o[q] = tile[jc + q][(((hh >> 3) ^ ((jc >> 3) & 7)) << 3) | (hh & 7)];
                *reinterpret_cast<uint4 *>(dstT + (size_t)(h0 + hh) * ldt + (size_t)cb * 64 + jc) =
                    *reinterpret_cast<const uint4 *>(o);
            }
        }
        __syncthreads();
    }
}

}  // namespace

int router_wgrad_splits(const LayerDims &d) {
    const int chunks = ceil_div(d.H, 2048);
    const int z = (148 * 4) / std::max(1, d.E * chunks);
    return std::max(1, std::min(z, 64));
}

cudaError_t launch_router_dl(const LayerDims &d, const float *dweight_part, int m_tiles,
                             const int32_t *slot_pos, const float *topk_w, float *dl,
                             cudaStream_t s) {
    return launch_pdl(router_dl_kernel, dim3(ceil_div(d.N, 256)), dim3(256), 0, s, d.N, d.k, m_tiles,
                      d.N * d.k, dweight_part, slot_pos, topk_w, dl);
}

cudaError_t launch_transpose_rows(const LayerDims &d, const void *src, const int32_t *eoff,
                                  const int32_t *perm, void *dstT, int64_t ldt, void *z0, int z0_cols,
                                  void *z1, int z1_cols, cudaStream_t s) {
    return launch_pdl(transpose_rows_kernel, dim3((unsigned)(ldt / 64), (unsigned)ceil_div(d.H, 512)),
                      dim3(256), 0, s, (const __nv_bfloat16 *)src,
                      d.H, d.k, eoff, d.E, perm, (__nv_bfloat16 *)dstT, ldt,
                      (__nv_bfloat16 *)z0, z0_cols, (__nv_bfloat16 *)z1, z1_cols, d.N * d.k);
}

cudaError_t launch_dx_combine(const LayerDims &d, const void *dx_slots, const int32_t *slot_pos,
                              const int32_t *topk_idx, const float *dl, const void *w_router,
                              void *dx, cudaStream_t s) {
    if (d.dtype == MOE_DTYPE_BF16)
        return launch_pdl(dx_combine_kernel<__nv_bfloat16>, dim3(ceil_div(d.N, 8)), dim3(256), 0, s,
                          (const __nv_bfloat16 *)dx_slots, slot_pos, topk_idx, dl,
                          (const __nv_bfloat16 *)w_router, d.N, d.H, d.k, (__nv_bfloat16 *)dx);
    return launch_pdl(dx_combine_kernel<float>, dim3(ceil_div(d.N, 8)), dim3(256), 0, s,
                      (const float *)dx_slots, slot_pos, topk_idx, dl, (const float *)w_router, d.N,
                      d.H, d.k, (float *)dx);
}

cudaError_t launch_router_wgrad(const LayerDims &d, const int32_t *eoff_all, const int32_t *perm_all,
                                const float *dl, const void *x, float *partial, float *partial_db,
                                float *dw_router, float *db_router, cudaStream_t s) {
    const int Z = router_wgrad_splits(d);
    const dim3 grid(d.E, ceil_div(d.H, 2048), Z);
    cudaError_t e = d.dtype == MOE_DTYPE_BF16
        ? launch_pdl(router_wgrad_partial_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, eoff_all,
                     perm_all, dl, (const __nv_bfloat16 *)x, d.H, d.E, d.k, partial, partial_db)
        : launch_pdl(router_wgrad_partial_kernel<float>, grid, dim3(256), 0, s, eoff_all, perm_all,
                     dl, (const float *)x, d.H, d.E, d.k, partial, partial_db);
    if (e != cudaSuccess) return e;
    const int rgrid = (int)std::min<int64_t>(ceil_div64((int64_t)d.E * d.H, 256), 148 * 4);
    return launch_pdl(router_wgrad_reduce_kernel, dim3(rgrid), dim3(256), 0, s,
                      (const float *)partial, (const float *)partial_db, Z, d.E, d.H, dw_router,
                      db_router);
}

}  // namespace moe
