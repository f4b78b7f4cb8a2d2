// Step 1 on the tensor cores -- routing for bf16 layers (Ultralytics glossary "Expert
// Parallelism", section "How tokens move between GPUs", step 1 and its routing example):
// logits = x W_r^T (+ b) accumulate in TMEM, M = 128 tokens by N = E rounded up to 16;
// each epilogue thread owns one token's logits, keeps its top-k in registers (ties to
// the lower expert id), applies the softmax over the k chosen logits and adds the
// token's experts to the per-segment histogram that the dispatch scan consumes.
//
// One CTA per 128-token tile. The top-k runs over column slices: with SLICES groups of
// four epilogue warps, group g selects each token's top-k among its slice of the experts
// and group 0 merges the other groups' lists in expert order, which keeps the ordering
// (value descending, ties to the lower id).
//
// Per CTA (64 + 128 * SLICES threads, one tile):
//   warp 0      TMA producer: 128x64 x tile + round16(E) x 64 router tile per stage,
//               128-byte swizzle, 3-stage ring guarded by full/empty mbarriers;
//   warp 1      allocates TMEM (round16(E) columns, at least 32) and one thread issues
//               tcgen05.mma (M=128, N=round16(E), K=16, bf16 in, fp32 acc);
//   warps 2..   epilogue: tcgen05.ld of the logits of their TMEM lane quarter and
//               column slice, top-k, merge, softmax and histogram.
// Exactness: bf16 products are exact in fp32 and, for inputs on the dyadic grids of the
// exact test variant, every partial sum is too, so the chosen ids do not depend on the
// order in which the tensor cores accumulate.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records
// MOE_DEV_TIMEOUT in the status word, skips the remaining work, waits (bounded) for its
// own copies, frees TMEM and returns.
#include <mutex>

#include "sm100.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = kTcBlockM;   // 128 tokens per tile
constexpr int STAGES = 3;
constexpr uint32_t A_BYTES = BM * BK * 2;
static_assert(BM == 2 * kSegTokens, "a route tile covers two histogram segments");

// Routing variants (template MODE): 0 plain top-k of the logits; 1 selection on
// logits + selection bias, weights from the logits; 2 as 1 within the group_limit best
// partitions (one column slice, two passes over the accumulator).
enum { ROUTE_PLAIN = 0, ROUTE_SELBIAS = 1, ROUTE_GROUP = 2 };

struct RouteParams {
    int rows;                // tokens
    int bn;                  // MMA N (E rounded up to 16)
    uint32_t idesc;
    int num_kb;              // K blocks of BK
    uint32_t tmem_cols;
    int E, k, nseg;
    const float *bias;       // [E] or nullptr
    const float *sel_bias;   // [E] or nullptr (selection only)
    int group_limit, per_part;   // ROUTE_GROUP: partitions kept, experts per partition
    int32_t *route_idx;      // [N, k] out
    float *route_w;          // [N, k] out
    int32_t *seg_hist;       // [nseg, E] or nullptr
    float *logits;           // [N, E] out (logit + router bias) or nullptr
    int32_t *status;         // or nullptr
};

// Shared-memory layout for a given MMA N.
struct RouteSmem {
    uint32_t b_off, bar_off, misc_off, bias_off, sbias_off, hist_off, alloc;
};
__host__ __device__ inline RouteSmem route_smem(int bn, int E) {
    RouteSmem m;
    m.b_off = STAGES * A_BYTES;
    m.bar_off = m.b_off + STAGES * (uint32_t)bn * BK * 2;
    m.misc_off = m.bar_off + 16 * 8;
    m.bias_off = m.misc_off + 16;
    m.sbias_off = m.bias_off + (uint32_t)(E + 3) / 4 * 16;
    m.hist_off = m.sbias_off + (uint32_t)(E + 3) / 4 * 16;
    m.alloc = m.hist_off + 2 * (uint32_t)E * 4 + 1024;   // + slack to align the base
    return m;
}

template <int KMAX>
__device__ __forceinline__ void topk_push(float (&val)[KMAX], int (&idx)[KMAX], float v, int e) {
    if (!(v > val[KMAX - 1] || idx[KMAX - 1] < 0)) return;
    val[KMAX - 1] = v;
    idx[KMAX - 1] = e;
#pragma unroll
    for (int j = KMAX - 1; j > 0; --j) {
        const bool up = val[j] > val[j - 1] || idx[j - 1] < 0;
        const float hv = up ? val[j] : val[j - 1], lv = up ? val[j - 1] : val[j];
        const int hi = up ? idx[j] : idx[j - 1], li = up ? idx[j - 1] : idx[j];
        val[j - 1] = hv;
        val[j] = lv;
        idx[j - 1] = hi;
        idx[j] = li;
    }
}

// As topk_push, carrying each entry's raw logit along (the routing variants select on
// logit + selection bias but weight by the logit).
template <int KMAX>
__device__ __forceinline__ void topk_push_raw(float (&val)[KMAX], float (&raw)[KMAX],
                                              int (&idx)[KMAX], float v, float l, int e) {
    if (!(v > val[KMAX - 1] || idx[KMAX - 1] < 0)) return;
    val[KMAX - 1] = v;
    raw[KMAX - 1] = l;
    idx[KMAX - 1] = e;
#pragma unroll
    for (int j = KMAX - 1; j > 0; --j) {
        const bool up = val[j] > val[j - 1] || idx[j - 1] < 0;
        const float hv = up ? val[j] : val[j - 1], lv = up ? val[j - 1] : val[j];
        const float hr = up ? raw[j] : raw[j - 1], lr = up ? raw[j - 1] : raw[j];
        const int hi = up ? idx[j] : idx[j - 1], li = up ? idx[j - 1] : idx[j];
        val[j - 1] = hv;
        val[j] = lv;
        raw[j - 1] = hr;
        raw[j] = lr;
        idx[j - 1] = hi;
        idx[j] = li;
    }
}

template <int KMAX, int SLICES, int MODE>
__global__ void __launch_bounds__(64 + 128 * SLICES, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w, const RouteParams p) {
    constexpr int NT = 128 * SLICES;   // epilogue threads
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const RouteSmem L = route_smem(p.bn, p.E);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *full = bars;                  // [STAGES]
    uint64_t *empty = bars + STAGES;        // [STAGES]
    uint64_t *tfull = bars + 2 * STAGES;    // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + L.misc_off + 4);
    float *bias_s = reinterpret_cast<float *>(smem + L.bias_off);
    float *sbias_s = reinterpret_cast<float *>(smem + L.sbias_off);
    int *hist_s = reinterpret_cast<int *>(smem + L.hist_off);   // [2][E]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tile = blockIdx.x;
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tmap_x);
            tma_prefetch_desc(&tmap_w);
        }
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else if (warp == 2 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dep_wait();   // the previous kernel's writes are visible from here on
    grid_dep_trigger();
    if (warp == 3) {
        for (int e = lane; e < p.E; e += 32) {
            bias_s[e] = p.bias != nullptr ? p.bias[e] : 0.f;
            sbias_s[e] = p.sel_bias != nullptr ? p.sel_bias[e] : 0.f;
        }
        for (int e = lane; e < 2 * p.E; e += 32) hist_s[e] = 0;
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            const uint32_t tx = A_BYTES + (uint32_t)p.bn * BK * 2;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_s, p.status)) break;
                mbar_arrive_expect_tx(&full[stage], tx);
                const uint32_t fb = smem_u32(&full[stage]);
                tma_load_2d(smem_u32(smem + stage * A_BYTES), &tmap_x, fb, kb * BK, tile * BM);
                tma_load_2d(smem_u32(smem + L.b_off + stage * (uint32_t)p.bn * BK * 2), &tmap_w,
                            fb, kb * BK, 0);
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // no copy may still be landing when the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) {
                    volatile int no_abort = 0;
                    mbar_wait(&full[s], (armed_parity >> s) & 1u, &no_abort, p.status);
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                if (!mbar_wait(&full[stage], phase, abort_s, p.status)) break;
                fence_after();
                const uint32_t a_addr = smem_u32(smem + stage * A_BYTES);
                const uint32_t b_addr = smem_u32(smem + L.b_off + stage * (uint32_t)p.bn * BK * 2);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16(tmem_base, smem_desc_sw128(a_addr + kk * 32),
                             smem_desc_sw128(b_addr + kk * 32), p.idesc, (kb | kk) != 0);
                commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // the accumulator is final (after a timeout: every issued MMA is done, and
            // the epilogue sees the abort flag)
            commit(tfull);
        }
    } else {   // ------------------------------------------------------ epilogue
        const int q = warp & 3;                // TMEM lane quarter
        const int slice = (warp - 2) >> 2;     // column slice of the experts
        const int r = q * 32 + lane;           // accumulator row = token of the tile
        const int tok = tile * BM + r;
        const int etid = threadIdx.x - 64;     // 0 .. NT-1
        // tcgen05.ld is warp-collective and the epilogue warps share named barriers:
        // all of them decide together
        const bool ok = epilogue_all<NT>(mbar_wait(tfull, 0, abort_s, p.status) && *abort_s == 0);
        fence_after();
        float val[KMAX], raw[KMAX];   // raw: the entry's logit (MODE > ROUTE_PLAIN)
        int idx[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            val[j] = -INFINITY;
            raw[j] = -INFINITY;
            idx[j] = -1;
        }
        // a candidate: logit l = acc + bias, selection score l (+ selection bias); a NaN
        // ranks last
        auto push = [&](float acc, int e) {
            const float l = acc + bias_s[e];
            if (MODE == ROUTE_PLAIN) {
                topk_push<KMAX>(val, idx, isnan(l) ? -INFINITY : l, e);
            } else {
                const float sc = l + sbias_s[e];
                topk_push_raw<KMAX>(val, raw, idx, isnan(sc) ? -INFINITY : sc,
                                    isnan(l) ? -INFINITY : l, e);
            }
        };
        // optional copy of the token's logits (with the router bias) for load statistics
        auto store_logits = [&](const float (&v)[32], int c) {
            if (p.logits == nullptr || tok >= p.rows) return;
            float *dst = p.logits + (size_t)tok * p.E + c;
            if (c + 32 <= p.E && (p.E & 3) == 0) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) =
                        make_float4(v[j] + bias_s[c + j], v[j + 1] + bias_s[c + j + 1],
                                    v[j + 2] + bias_s[c + j + 2], v[j + 3] + bias_s[c + j + 3]);
            } else {
                for (int j = 0; j < 32 && c + j < p.E; ++j) dst[j] = v[j] + bias_s[c + j];
            }
        };
        if (ok) {
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
            if (MODE == ROUTE_GROUP) {
                // pass 1: every partition's best selection score, the best partitions
                // in a list (pushed in increasing partition id: ties keep the lower)
                float pv[kMaxGroupLimit];
                int pi[kMaxGroupLimit];
#pragma unroll
                for (int j = 0; j < kMaxGroupLimit; ++j) {
                    pv[j] = -INFINITY;
                    pi[j] = -1;
                }
                float cur = -INFINITY;
                int cur_p = 0;
                for (int c = 0; c < p.bn; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = c + j;
                        if (e < p.E) {
                            const int pp = e / p.per_part;
                            if (pp != cur_p) {
                                topk_push<kMaxGroupLimit>(pv, pi, cur, cur_p);
                                cur = -INFINITY;
                                cur_p = pp;
                            }
                            const float sc = v[j] + bias_s[e] + sbias_s[e];
                            cur = isnan(sc) ? cur : fmaxf(cur, sc);
                        }
                    }
                }
                topk_push<kMaxGroupLimit>(pv, pi, cur, cur_p);
                uint64_t allowed = 0;
#pragma unroll
                for (int j = 0; j < kMaxGroupLimit; ++j)
                    if (j < p.group_limit && pi[j] >= 0) allowed |= 1ull << pi[j];
                // pass 2: the top-k among the experts of the kept partitions
                for (int c = 0; c < p.bn; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = c + j;
                        if (e < p.E && ((allowed >> (e / p.per_part)) & 1ull)) push(v[j], e);
                    }
                    store_logits(v, c);
                }
            } else {
                const int cps = (p.bn + 32 * SLICES - 1) / (32 * SLICES) * 32;   // columns per slice
                const int c1 = min(p.bn, (slice + 1) * cps);
                for (int c = slice * cps; c < c1; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = c + j;
                        if (e < p.E) push(v[j], e);
                    }
                    store_logits(v, c);
                }
            }
            if (SLICES > 1) {
                // lists of slices 1.. into the stage ring (every MMA has read it), then
                // group 0 pushes them in slice order, i.e. in increasing expert id
                float *lv = reinterpret_cast<float *>(smem);   // [SLICES-1][BM][KMAX]
                float *lr = lv + (SLICES - 1) * BM * KMAX;
                int *li = reinterpret_cast<int *>(lr + (SLICES - 1) * BM * KMAX);
                if (slice > 0)
#pragma unroll
                    for (int j = 0; j < KMAX; ++j) {
                        lv[((slice - 1) * BM + r) * KMAX + j] = val[j];
                        lr[((slice - 1) * BM + r) * KMAX + j] = raw[j];
                        li[((slice - 1) * BM + r) * KMAX + j] = idx[j];
                    }
                epilogue_sync<NT>();
                if (slice == 0)
                    for (int g = 0; g < SLICES - 1; ++g)
#pragma unroll
                        for (int j = 0; j < KMAX; ++j) {
                            const int o = (g * BM + r) * KMAX + j;
                            const int e = li[o];
                            if (e < 0) continue;
                            if (MODE == ROUTE_PLAIN)
                                topk_push<KMAX>(val, idx, lv[o], e);
                            else
                                topk_push_raw<KMAX>(val, raw, idx, lv[o], lr[o], e);
                        }
            }
            if (slice == 0 && tok < p.rows) {
                // softmax over the chosen experts' logits
                const float *lg = MODE == ROUTE_PLAIN ? val : raw;
                float m = lg[0];
#pragma unroll
                for (int j = 1; j < KMAX; ++j)
                    if (j < p.k) m = fmaxf(m, lg[j]);
                float ex[KMAX], sum = 0.f;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    ex[j] = j < p.k ? expf(lg[j] - m) : 0.f;
                    sum += ex[j];
                }
                const float inv = 1.0f / sum;
#pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (j < p.k) {
                        p.route_idx[(size_t)tok * p.k + j] = idx[j];
                        p.route_w[(size_t)tok * p.k + j] = ex[j] * inv;
                        if (p.seg_hist != nullptr) atomicAdd(&hist_s[(r >> 6) * p.E + idx[j]], 1);
                    }
            }
            if (p.seg_hist != nullptr) {
                epilogue_sync<NT>();
                for (int j = etid; j < 2 * p.E; j += NT) {
                    const int seg = 2 * tile + j / p.E;
                    if (seg < p.nseg) p.seg_hist[(size_t)seg * p.E + j % p.E] = hist_s[j];
                }
            }
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(p.tmem_cols)
                     : "memory");
    }
}

template <int KMAX, int SLICES, int MODE>
cudaError_t launch_route_tc(const CUtensorMap &mx, const CUtensorMap &mw, const RouteParams &prm,
                            int tiles, cudaStream_t s) {
    auto kern = route_tc_kernel<KMAX, SLICES, MODE>;
    const RouteSmem L = route_smem(prm.bn, prm.E);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        // the dynamic shared-memory limit, per device, only ever grows
        static std::mutex mu;
        static uint32_t attr_max[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (L.alloc > attr_max[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)L.alloc);
            if (e != cudaSuccess) return e;
            attr_max[dev] = L.alloc;
        }
    }
    return launch_pdl(kern, dim3(tiles), dim3(64 + 128 * SLICES), L.alloc, s, mx, mw, prm);
}

// Four column slices while one CTA per SM covers every tile, two otherwise (two CTAs of
// 320 threads fit on an SM); lists longer than 8 are not sliced.
template <int KMAX>
cudaError_t launch_route_k(const CUtensorMap &mx, const CUtensorMap &mw, const RouteParams &prm,
                           int tiles, int num_sms, cudaStream_t s) {
    if (tiles <= 0) return cudaSuccess;
    if (prm.group_limit > 0) return launch_route_tc<KMAX, 1, ROUTE_GROUP>(mx, mw, prm, tiles, s);
    if constexpr (KMAX > 8) {
        (void)num_sms;
        if (prm.sel_bias != nullptr)
            return launch_route_tc<KMAX, 1, ROUTE_SELBIAS>(mx, mw, prm, tiles, s);
        return launch_route_tc<KMAX, 1, ROUTE_PLAIN>(mx, mw, prm, tiles, s);
    } else {
        const bool wide = tiles <= num_sms;
        if (prm.sel_bias != nullptr)
            return wide ? launch_route_tc<KMAX, 4, ROUTE_SELBIAS>(mx, mw, prm, tiles, s)
                        : launch_route_tc<KMAX, 2, ROUTE_SELBIAS>(mx, mw, prm, tiles, s);
        return wide ? launch_route_tc<KMAX, 4, ROUTE_PLAIN>(mx, mw, prm, tiles, s)
                    : launch_route_tc<KMAX, 2, ROUTE_PLAIN>(mx, mw, prm, tiles, s);
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t get_encoder(EncodeTiledFn *fn) {
    static EncodeTiledFn cached = nullptr;
    if (cached == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || ptr == nullptr) return cudaErrorNotSupported;
        cached = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    *fn = cached;
    return cudaSuccess;
}

}  // namespace

cudaError_t tc::make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                         uint64_t ld, uint32_t box_rows) {
    EncodeTiledFn enc;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc::make_store_map_3d(CUtensorMap *map, void *base, uint64_t d0, uint64_t d1,
                                 uint64_t d2, uint32_t box0, uint32_t box1) {
    EncodeTiledFn enc;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_tc_route(const LayerDims &d, const void *x, const void *w_router,
                            const float *bias, int32_t *topk_idx, float *topk_w,
                            float *logits, int32_t *seg_hist, int32_t *status, int num_sms,
                            cudaStream_t s) {
    const int bn = (d.E + 15) / 16 * 16;
    CUtensorMap mx, mw;
    cudaError_t e = tc::make_map(&mx, x, d.N, d.H, d.H, BM);
    if (e != cudaSuccess) return e;
    e = tc::make_map(&mw, w_router, d.E, d.H, d.H, (uint32_t)bn);
    if (e != cudaSuccess) return e;
    RouteParams prm = {};
    prm.rows = d.N;
    prm.bn = bn;
    prm.idesc = make_idesc(BM, bn);
    prm.num_kb = ceil_div(d.H, BK);
    prm.tmem_cols = 32;
    while ((int)prm.tmem_cols < bn) prm.tmem_cols <<= 1;
    prm.E = d.E;
    prm.k = d.k;
    prm.nseg = ceil_div(d.N, kSegTokens);
    prm.bias = bias;
    prm.sel_bias = d.sel_bias;
    prm.group_limit = d.group_limit;
    prm.per_part = d.E / d.P;
    prm.route_idx = topk_idx;
    prm.route_w = topk_w;
    prm.seg_hist = seg_hist;
    prm.logits = logits;
    prm.status = status;
    const int tiles = ceil_div(d.N, BM);
    // the register list holds k rounded up to a power of two
    if (d.k <= 1) return launch_route_k<1>(mx, mw, prm, tiles, num_sms, s);
    if (d.k <= 2) return launch_route_k<2>(mx, mw, prm, tiles, num_sms, s);
    if (d.k <= 4) return launch_route_k<4>(mx, mw, prm, tiles, num_sms, s);
    if (d.k <= 8) return launch_route_k<8>(mx, mw, prm, tiles, num_sms, s);
    if (d.k <= 16) return launch_route_k<16>(mx, mw, prm, tiles, num_sms, s);
    return launch_route_k<32>(mx, mw, prm, tiles, num_sms, s);
}

}  // namespace moe
