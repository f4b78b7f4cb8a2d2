// Step 3 for fp32 layers -- the same grouped SwiGLU FFN as the tensor-core path, in fp32
// FFMA (single-pass TF32 tensor cores carry 10 mantissa bits, too few for a 1e-4
// relative bound). 128x64 output tiles over (expert, n tile, m tile), 256 threads, each
// owning 8 rows x 4 columns (of gate and of up in the first kernel: 16 FFMA per 16-byte
// shared-memory load). K advances 16 at a time through two shared-memory buffers: the
// next slice is loaded into registers while the current one is multiplied, so one
// barrier per slice suffices. The first kernel fuses SwiGLU, the second the weighted
// un-permute into the pair's slot.
#include "common.cuh"

namespace moe {
namespace {

constexpr int SBM = kSimtBlockM;   // 128
constexpr int SBN = 64;
constexpr int SBK = 16;
static_assert(SBM == 128 && SBN == kGateUpBlock, "tile shape of the thread layout");

__device__ __forceinline__ float4 ld4_or_zero(const float *p, bool ok) {
    return ok ? __ldg(reinterpret_cast<const float4 *>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
}
// 4 consecutive k of one row into the k-major tile s[k][row]
template <int W>
__device__ __forceinline__ void st_col(float (*s)[W], int k, int r, float4 v) {
    s[k + 0][r] = v.x;
    s[k + 1][r] = v.y;
    s[k + 2][r] = v.z;
    s[k + 3][r] = v.w;
}

__global__ void __launch_bounds__(256, 2)
simt_gate_up_kernel(const float *__restrict__ send, const int32_t *__restrict__ eoff, int e_begin,
                    int ne, const float *__restrict__ packed, int H, int Ipad,
                    float *__restrict__ hbuf, float *__restrict__ gu) {
    grid_dep_wait();
    grid_dep_trigger();
    __shared__ int eo[kMaxExperts + 1], mtp[kMaxExperts + 1];
    __shared__ __align__(16) float As[2][SBK][SBM + 4];
    __shared__ __align__(16) float Gs[2][SBK][SBN + 4];
    __shared__ __align__(16) float Us[2][SBK][SBN + 4];
    if (threadIdx.x < 32) build_tile_tables(eoff, e_begin, ne, SBM, eo, mtp);
    __syncthreads();
    const int n_tiles = Ipad / SBN;
    const int total = mtp[ne] * n_tiles;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int lr = tid / 4, lk = (tid % 4) * 4;   // loader: row (and row + 64), k offset
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int i, m, n;
        decode_tile(tile, mtp, ne, n_tiles, i, m, n);
        const int e = e_begin + i;
        const int row0 = eo[i] + m * SBM;
        const int rows = min(SBM, eo[i + 1] - row0);
        const int col0 = n * SBN;   // output column = intermediate feature
        // packed block col0 / 64: its 64 gate rows, then the 64 matching up rows
        const size_t g_row0 = (size_t)e * 2 * Ipad + (size_t)(col0 / kGateUpBlock) * 2 * kGateUpBlock;
        const size_t u_row0 = g_row0 + kGateUpBlock;
        float4 ra0, ra1, rg, ru;
        auto load = [&](int k0) {
            const bool kin = k0 + lk < H;
            ra0 = ld4_or_zero(send + (size_t)(row0 + lr) * H + k0 + lk, kin && lr < rows);
            ra1 = ld4_or_zero(send + (size_t)(row0 + lr + 64) * H + k0 + lk, kin && lr + 64 < rows);
            rg = ld4_or_zero(packed + (g_row0 + lr) * H + k0 + lk, kin);
            ru = ld4_or_zero(packed + (u_row0 + lr) * H + k0 + lk, kin);
        };
        auto store = [&](int b) {
            st_col(As[b], lk, lr, ra0);
            st_col(As[b], lk, lr + 64, ra1);
            st_col(Gs[b], lk, lr, rg);
            st_col(Us[b], lk, lr, ru);
        };
        float ag[8][4] = {}, au[8][4] = {};
        load(0);
        store(0);
        __syncthreads();
        for (int k0 = 0, b = 0; k0 < H; k0 += SBK, b ^= 1) {
            const bool more = k0 + SBK < H;
            if (more) load(k0 + SBK);
#pragma unroll
            for (int kk = 0; kk < SBK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8 + 4]);
                const float4 g = *reinterpret_cast<const float4 *>(&Gs[b][kk][tx * 4]);
                const float4 u = *reinterpret_cast<const float4 *>(&Us[b][kk][tx * 4]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float gv[4] = {g.x, g.y, g.z, g.w};
                const float uv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        ag[r][c] = fmaf(av[r], gv[c], ag[r][c]);
                        au[r][c] = fmaf(av[r], uv[c], au[r][c]);
                    }
            }
            if (more) store(b ^ 1);   // the other buffer: its readers passed the barrier
            __syncthreads();
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int rr = ty * 8 + r;
            if (rr < rows) {
                float o[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float g = ag[r][c];
                    o[c] = g / (1.0f + expf(-g)) * au[r][c];
                }
                *reinterpret_cast<float4 *>(hbuf + (size_t)(row0 + rr) * Ipad + col0 + tx * 4) =
                    make_float4(o[0], o[1], o[2], o[3]);
                if (gu != nullptr) {   // training: the pre-activations, packed column order
                    float *gd = gu + (size_t)(row0 + rr) * 2 * Ipad + (col0 / kGateUpBlock) * 2 * kGateUpBlock + tx * 4;
                    *reinterpret_cast<float4 *>(gd) = make_float4(ag[r][0], ag[r][1], ag[r][2], ag[r][3]);
                    *reinterpret_cast<float4 *>(gd + kGateUpBlock) =
                        make_float4(au[r][0], au[r][1], au[r][2], au[r][3]);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(256)
simt_down_kernel(const float *__restrict__ hbuf, int Ipad, int I, const int32_t *__restrict__ eoff,
                 int e_begin, int ne, const float *__restrict__ wd, int H,
                 const int32_t *__restrict__ perm, const float *__restrict__ topk_w,
                 float *__restrict__ slots) {
    grid_dep_wait();
    grid_dep_trigger();
    __shared__ int eo[kMaxExperts + 1], mtp[kMaxExperts + 1];
    __shared__ __align__(16) float As[2][SBK][SBM + 4];
    __shared__ __align__(16) float Bs[2][SBK][SBN + 4];
    if (threadIdx.x < 32) build_tile_tables(eoff, e_begin, ne, SBM, eo, mtp);
    __syncthreads();
    const int n_tiles = (H + SBN - 1) / SBN;
    const int total = mtp[ne] * n_tiles;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int lr = tid / 4, lk = (tid % 4) * 4;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int i, m, n;
        decode_tile(tile, mtp, ne, n_tiles, i, m, n);
        const int e = e_begin + i;
        const int row0 = eo[i] + m * SBM;
        const int rows = min(SBM, eo[i + 1] - row0);
        const int col0 = n * SBN;
        float4 ra0, ra1, rb;
        auto load = [&](int k0) {
            const bool kin = k0 + lk < I;
            ra0 = ld4_or_zero(hbuf + (size_t)(row0 + lr) * Ipad + k0 + lk, kin && lr < rows);
            ra1 = ld4_or_zero(hbuf + (size_t)(row0 + lr + 64) * Ipad + k0 + lk, kin && lr + 64 < rows);
            rb = ld4_or_zero(wd + ((size_t)e * H + col0 + lr) * I + k0 + lk, kin && col0 + lr < H);
        };
        auto store = [&](int b) {
            st_col(As[b], lk, lr, ra0);
            st_col(As[b], lk, lr + 64, ra1);
            st_col(Bs[b], lk, lr, rb);
        };
        float acc[8][4] = {};
        load(0);
        store(0);
        __syncthreads();
        for (int k0 = 0, b = 0; k0 < I; k0 += SBK, b ^= 1) {
            const bool more = k0 + SBK < I;
            if (more) load(k0 + SBK);
#pragma unroll
            for (int kk = 0; kk < SBK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8 + 4]);
                const float4 w = *reinterpret_cast<const float4 *>(&Bs[b][kk][tx * 4]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
            }
            if (more) store(b ^ 1);
            __syncthreads();
        }
        const int col = col0 + tx * 4;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int rr = ty * 8 + r;
            if (rr < rows && col < H) {
                const int pair = perm[row0 + rr];
                const float w = topk_w[pair];
                *reinterpret_cast<float4 *>(slots + (size_t)pair * H + col) =
                    make_float4(w * acc[r][0], w * acc[r][1], w * acc[r][2], w * acc[r][3]);
            }
        }
    }
}

int simt_grid(const LayerDims &d, int ne, int n_tiles) {
    const int64_t max_tiles = (ceil_div64((int64_t)d.N * d.k, SBM) + ne) * n_tiles;
    return (int)std::min<int64_t>(max_tiles, 148 * 8);
}

}  // namespace

cudaError_t launch_simt_gate_up(const LayerDims &d, const float *send,
                                const int32_t *expert_offsets, int e_begin, int e_end,
                                const float *packed, float *h, float *gu, cudaStream_t s) {
    const int ne = e_end - e_begin;
    const int grid = simt_grid(d, ne, d.Ipad / SBN);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(simt_gate_up_kernel, dim3(grid), dim3(256), 0, s, send, expert_offsets, e_begin,
                      ne, packed, d.H, d.Ipad, h, gu);
}

cudaError_t launch_simt_down(const LayerDims &d, const float *h, const int32_t *expert_offsets,
                             int e_begin, int e_end, const float *w_down, const int32_t *perm,
                             const float *topk_w, float *out_slots, cudaStream_t s) {
    const int ne = e_end - e_begin;
    const int grid = simt_grid(d, ne, ceil_div(d.H, SBN));
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(simt_down_kernel, dim3(grid), dim3(256), 0, s, h, d.Ipad, d.I, expert_offsets,
                      e_begin, ne, w_down, d.H, perm, topk_w, out_slots);
}

}  // namespace moe
