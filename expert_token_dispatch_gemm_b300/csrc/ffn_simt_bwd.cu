// Backward of the local experts for fp32 layers, in fp32 FFMA (the counterpart of
// ffn_simt.cu; the chain rule and the readings are those of grouped_gemm_bwd.cu):
//   dgrad_down : da_u[r, i] = sum_h dout_r[h] W_d[h, i]; epilogue: dweight partials,
//                dg, du (packed order), w * silu(g) * u
//   dgrad_gu   : dx_r[h] = sum_f dgu_r[f] W_gu[f, h]  -> the pair's dx slot
//   wgrad      : dW_gu[f, h] = sum_r dgu_r[f] x_r[h],  dW_d[h, i] = sum_r dout_r[h] wa_r[i]
// 128 x 64 output tiles, 256 threads owning 8 rows x 4 columns, K in steps of 16 through
// two shared-memory buffers with register prefetch. The dgrad kernels read token rows
// along K and the weights as [K rows][N columns]; the weight-gradient kernel reads both
// operands as [K = the expert's rows][columns], zero past the segment.
#include "common.cuh"

namespace moe {
namespace {

constexpr int TBM = kSimtBlockM;   // 128
constexpr int TBN = 64;
constexpr int TBK = 16;

__device__ __forceinline__ float4 ld4z(const float *p, bool ok) {
    return ok ? __ldg(reinterpret_cast<const float4 *>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ float sigm(float g) { return 1.0f / (1.0f + expf(-g)); }

enum { SB_DGRAD_DOWN = 0, SB_DGRAD_GU = 1 };

// Token rows [row0, row0 + rows) of one expert x a 64-column slice of a [K, ncols]
// row-major weight block (K rows from w_row0).
template <int EPI>
__global__ void __launch_bounds__(256, 2)
simt_dgrad_kernel(const float *__restrict__ a_rows, int lda, const int32_t *__restrict__ eoff,
                  int ne, const float *__restrict__ w, size_t w_expert_stride, int K, int ldw,
                  int ncols, int n_tiles, const int32_t *__restrict__ perm,
                  const float *__restrict__ topk_w, const float *__restrict__ gu, int I, int Ipad,
                  float *__restrict__ dgu, float *__restrict__ wa, float *__restrict__ dweight_part,
                  int rows_total, float *__restrict__ dx_slots, int H) {
    grid_dep_wait();
    grid_dep_trigger();
    __shared__ int eo[kMaxExperts + 1], mtp[kMaxExperts + 1];
    __shared__ __align__(16) float As[2][TBK][TBM + 4];
    __shared__ __align__(16) float Bs[2][TBK][TBN + 4];
    if (threadIdx.x < 32) build_tile_tables(eoff, 0, ne, TBM, eo, mtp);
    __syncthreads();
    const int total = mtp[ne] * n_tiles;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int lr = tid / 4, lk = (tid % 4) * 4;   // A loader: row (and row + 64), k offset
    const int bk = tid / 16, bn = (tid % 16) * 4; // B loader: k row, 4 columns
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int i, m, n;
        decode_tile(tile, mtp, ne, n_tiles, i, m, n);
        const int row0 = eo[i] + m * TBM;
        const int rows = min(TBM, eo[i + 1] - row0);
        const int col0 = n * TBN;
        const float *wb = w + (size_t)i * w_expert_stride;
        float4 ra0, ra1, rb;
        auto load = [&](int k0) {
            const bool kin = k0 + lk < K;
            ra0 = ld4z(a_rows + (size_t)(row0 + lr) * lda + k0 + lk, kin && lr < rows);
            ra1 = ld4z(a_rows + (size_t)(row0 + lr + 64) * lda + k0 + lk, kin && lr + 64 < rows);
            rb = ld4z(wb + (size_t)(k0 + bk) * ldw + col0 + bn, k0 + bk < K && col0 + bn < ncols);
        };
        auto store = [&](int b) {
            As[b][lk + 0][lr] = ra0.x; As[b][lk + 1][lr] = ra0.y;
            As[b][lk + 2][lr] = ra0.z; As[b][lk + 3][lr] = ra0.w;
            As[b][lk + 0][lr + 64] = ra1.x; As[b][lk + 1][lr + 64] = ra1.y;
            As[b][lk + 2][lr + 64] = ra1.z; As[b][lk + 3][lr + 64] = ra1.w;
            *reinterpret_cast<float4 *>(&Bs[b][bk][bn]) = rb;
        };
        float acc[8][4] = {};
        load(0);
        store(0);
        __syncthreads();
        for (int k0 = 0, b = 0; k0 < K; k0 += TBK, b ^= 1) {
            const bool more = k0 + TBK < K;
            if (more) load(k0 + TBK);
#pragma unroll
            for (int kk = 0; kk < TBK; ++kk) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8 + 4]);
                const float4 bv = *reinterpret_cast<const float4 *>(&Bs[b][kk][tx * 4]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bb[c], acc[r][c]);
            }
            if (more) store(b ^ 1);
            __syncthreads();
        }
        const int col = col0 + tx * 4;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int rr = ty * 8 + r;
            const bool rv = rr < rows;
            const size_t row = (size_t)row0 + rr;
            if (EPI == SB_DGRAD_DOWN) {
                // col = intermediate feature i (4 of them); packed column of its gate
                float part = 0.f;
                if (rv) {
                    const int gcol = (col / 64) * 128 + (col % 64);
                    float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
                    float wv[4] = {0.f, 0.f, 0.f, 0.f};
                    if (col < I) {
                        const float wt = topk_w[perm[row]];
                        const float4 g4 = *reinterpret_cast<const float4 *>(gu + row * 2 * Ipad + gcol);
                        const float4 u4 = *reinterpret_cast<const float4 *>(gu + row * 2 * Ipad + gcol + 64);
                        const float g[4] = {g4.x, g4.y, g4.z, g4.w}, u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float sg = sigm(g[c]);
                            const float sl = g[c] * sg;
                            const float a = sl * u[c];
                            part = fmaf(acc[r][c], a, part);
                            const float dw = wt * acc[r][c];
                            dg[c] = dw * u[c] * (sg * (1.0f + g[c] * (1.0f - sg)));
                            du[c] = dw * sl;
                            wv[c] = wt * a;
                        }
                    }
                    *reinterpret_cast<float4 *>(dgu + row * 2 * Ipad + gcol) = make_float4(dg[0], dg[1], dg[2], dg[3]);
                    *reinterpret_cast<float4 *>(dgu + row * 2 * Ipad + gcol + 64) = make_float4(du[0], du[1], du[2], du[3]);
                    *reinterpret_cast<float4 *>(wa + row * Ipad + col) = make_float4(wv[0], wv[1], wv[2], wv[3]);
                }
                // the 16 threads of a row (tx) hold its 64 features: add in fixed order
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (rv && tx == 0) dweight_part[(size_t)n * rows_total + row] = part;
            } else {
                if (rv && col < H) {
                    const int pr = perm[row];
                    *reinterpret_cast<float4 *>(dx_slots + (size_t)pr * H + col) =
                        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
                }
            }
        }
    }
}

// dW[e][m][n] = sum over the expert's rows r of A[r][m] * B[r][n] (A, B row-major with
// leading dimensions lda, ldb); tiles (expert, m tile of 128, n tile of 64).
__global__ void __launch_bounds__(256, 2)
simt_wgrad_kernel(const float *__restrict__ A, int lda, int mdim, const float *__restrict__ B,
                  int ldb, int ndim, const int32_t *__restrict__ eoff, int ne, int m_tiles,
                  int n_tiles, int gu_rows, int I, float *__restrict__ out0,
                  float *__restrict__ out1) {
    grid_dep_wait();
    grid_dep_trigger();
    __shared__ __align__(16) float As[2][TBK][TBM + 4];
    __shared__ __align__(16) float Bs[2][TBK][TBN + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int ak = tid / 32, am = (tid % 32) * 4;   // A loader: k rows ak, ak + 8; 4 columns
    const int bk = tid / 16, bn = (tid % 16) * 4;
    const int total = ne * m_tiles * n_tiles;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const int e = tile / (m_tiles * n_tiles);
        const int l = tile - e * m_tiles * n_tiles;
        const int mt = l / n_tiles, nt = l - mt * n_tiles;
        const int r0 = eoff[e], nr = eoff[e + 1] - r0;
        const int m0 = mt * TBM, n0 = nt * TBN;
        float4 ra0, ra1, rb;
        auto load = [&](int k0) {
            ra0 = ld4z(A + (size_t)(r0 + k0 + ak) * lda + m0 + am, k0 + ak < nr && m0 + am < mdim);
            ra1 = ld4z(A + (size_t)(r0 + k0 + ak + 8) * lda + m0 + am, k0 + ak + 8 < nr && m0 + am < mdim);
            rb = ld4z(B + (size_t)(r0 + k0 + bk) * ldb + n0 + bn, k0 + bk < nr && n0 + bn < ndim);
        };
        auto store = [&](int b) {
            *reinterpret_cast<float4 *>(&As[b][ak][am]) = ra0;
            *reinterpret_cast<float4 *>(&As[b][ak + 8][am]) = ra1;
            *reinterpret_cast<float4 *>(&Bs[b][bk][bn]) = rb;
        };
        float acc[8][4] = {};
        if (nr > 0) {
            load(0);
            store(0);
            __syncthreads();
            for (int k0 = 0, b = 0; k0 < nr; k0 += TBK, b ^= 1) {
                const bool more = k0 + TBK < nr;
                if (more) load(k0 + TBK);
#pragma unroll
                for (int kk = 0; kk < TBK; ++kk) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8]);
                    const float4 a1 = *reinterpret_cast<const float4 *>(&As[b][kk][ty * 8 + 4]);
                    const float4 bv = *reinterpret_cast<const float4 *>(&Bs[b][kk][tx * 4]);
                    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                    for (int r = 0; r < 8; ++r)
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bb[c], acc[r][c]);
                }
                if (more) store(b ^ 1);
                __syncthreads();
            }
        }
        const int col = n0 + tx * 4;
        if (col >= ndim) continue;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int m = m0 + ty * 8 + r;
            float *dst = nullptr;
            if (gu_rows) {   // packed gate/up row -> dW_gate / dW_up row
                const int i = (m / 128) * 64 + (m % 64);
                if (m < mdim && i < I) dst = ((m % 128) < 64 ? out0 : out1) + ((size_t)e * I + i) * ndim;
            } else if (m < mdim) {
                dst = out0 + ((size_t)e * mdim + m) * ndim;
            }
            if (dst != nullptr)
                *reinterpret_cast<float4 *>(dst + col) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        }
    }
}

int simt_bwd_grid(int64_t max_tiles) { return (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, 148 * 8)); }

}  // namespace

cudaError_t launch_simt_dgrad_down(const LayerDims &d, const float *dout_send, const int32_t *eoff,
                                   const float *w_down, const float *gu, const int32_t *perm,
                                   const float *topk_w, float *dgu, float *wa, float *dweight_part,
                                   cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    const int n_tiles = d.Ipad / TBN;
    const int64_t max_tiles = (ceil_div64(rows, TBM) + d.E) * n_tiles;
    return launch_pdl(simt_dgrad_kernel<SB_DGRAD_DOWN>, dim3(simt_bwd_grid(max_tiles)), dim3(256), 0, s,
                      dout_send, d.H, eoff, d.E, w_down, (size_t)d.H * d.I, d.H, d.I, d.I, n_tiles,
                      perm, topk_w, gu, d.I, d.Ipad, dgu, wa, dweight_part, (int)rows,
                      (float *)nullptr, d.H);
}

cudaError_t launch_simt_dgrad_gate_up(const LayerDims &d, const float *dgu, const int32_t *eoff,
                                      const float *packed, const int32_t *perm, float *dx_slots,
                                      cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    const int n_tiles = ceil_div(d.H, TBN);
    const int64_t max_tiles = (ceil_div64(rows, TBM) + d.E) * n_tiles;
    return launch_pdl(simt_dgrad_kernel<SB_DGRAD_GU>, dim3(simt_bwd_grid(max_tiles)), dim3(256), 0, s,
                      dgu, 2 * d.Ipad, eoff, d.E, packed, (size_t)2 * d.Ipad * d.H, 2 * d.Ipad, d.H,
                      d.H, n_tiles, perm, (const float *)nullptr, (const float *)nullptr, d.I,
                      d.Ipad, (float *)nullptr, (float *)nullptr, (float *)nullptr, (int)rows,
                      dx_slots, d.H);
}

cudaError_t launch_simt_wgrad_gate_up(const LayerDims &d, const float *dgu, const float *send,
                                      const int32_t *eoff, float *dw_gate, float *dw_up,
                                      cudaStream_t s) {
    const int m_tiles = 2 * d.Ipad / TBM, n_tiles = ceil_div(d.H, TBN);
    return launch_pdl(simt_wgrad_kernel, dim3(simt_bwd_grid((int64_t)d.E * m_tiles * n_tiles)),
                      dim3(256), 0, s, dgu, 2 * d.Ipad, 2 * d.Ipad, send, d.H, d.H, eoff, d.E,
                      m_tiles, n_tiles, 1, d.I, dw_gate, dw_up);
}

cudaError_t launch_simt_wgrad_down(const LayerDims &d, const float *dout_send, const float *wa,
                                   const int32_t *eoff, float *dw_down, cudaStream_t s) {
    const int m_tiles = ceil_div(d.H, TBM), n_tiles = ceil_div(d.I, TBN);
    return launch_pdl(simt_wgrad_kernel, dim3(simt_bwd_grid((int64_t)d.E * m_tiles * n_tiles)),
                      dim3(256), 0, s, dout_send, d.H, d.H, wa, d.Ipad, d.I, eoff, d.E, m_tiles,
                      n_tiles, 0, d.I, dw_down, (float *)nullptr);
}

}  // namespace moe
