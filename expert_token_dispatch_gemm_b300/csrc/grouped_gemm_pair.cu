// Step 3 -- the local experts as grouped GEMMs on pairs of SMs (Ultralytics glossary
// "Expert Parallelism", step 3: each partition runs its local experts on the rows it
// received; Hugging Face "Expert parallelism" docs: the "grouped_gemm" rule splits expert
// weights along the expert dimension).
//
// Expert weights are the MMA's M side and the expert's tokens its N side ("swap AB"):
//   gate_up : D[f, t] = W_gu[f, :] . send[t, :]   -> h[t, f] = silu(gate) * up
//   down    : D[f, t] = W_d[f, :]  . h[t, :]      -> out_slots[perm[t], f] = w_t * D[f, t]
// so a ragged expert segment costs at most 31 padded token columns, not a padded
// 128-row tile. One tile = 256 weight rows x up to 256 tokens of one expert, computed by
// a cluster of two CTAs on two SMs with tcgen05.mma.cta_group::2 (M = 256, N = tokens
// rounded up to 32, K = 16): each CTA stages its 128 weight rows and half of the token
// rows, and holds its 128 rows of the fp32 accumulator in its own TMEM.
//
// The packed gate/up weights interleave 64 gate rows and the 64 matching up rows, so
// each CTA's 128 accumulator lanes hold the gate (lanes 0-63) and up (64-127) rows of
// the same 64 intermediate features; the epilogue pairs them through shared memory.
//
// Per CTA (192 threads, one CTA per SM, persistent over the tile list):
//   warp 0      TMA producer: 128 x 64 weight tile + (N/2, rounded up to 16, 32, 64 or
//               128) x 64 token tile per stage, 128-byte swizzle, 6-stage ring. Both CTAs' copies complete on the even
//               CTA's full barrier, which the even CTA arms with the pair's bytes.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) in both
//               CTAs; in the even CTA one thread issues the pair MMAs and commits them
//               to the empty / accumulator-full barriers of both CTAs.
//   warps 2..5  epilogue: tcgen05.ld of the CTA's accumulator lanes, 32 token columns at
//               a time, through shared memory into row-major bf16 stores; then one
//               arrival per warp on the even CTA's accumulator-empty barrier.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records
// MOE_DEV_TIMEOUT in the status word, stops issuing work, waits (bounded) for its own
// copies and MMAs, frees TMEM and returns.
#include "sm100.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int PM = 256;                 // weight rows per tile (the pair's M)
constexpr int CM = PM / 2;              // weight rows per CTA
constexpr int PN = 256;                 // max tokens per tile (the MMA's N)
constexpr int CN = PN / 2;              // token rows staged per CTA (TMA box height)
constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = CM * BK * 2;
constexpr uint32_t B_BYTES = CN * BK * 2;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * PN;
constexpr int CHUNK = 32;               // token columns per epilogue step
constexpr int GU_FEATS = kGateUpBlock;  // intermediate features per CTA in gate_up (64)
static_assert(2 * GU_FEATS == CM, "a CTA's weight rows are one gate/up block");

enum { EPI_SWIGLU = 0, EPI_DOWN = 1 };

// Weight map (box 128 rows) and token maps with box heights 16, 32, 64 and 128 rows:
// a tile stages only the token rows its MMA reads (N/2 per CTA).
struct PairMaps {
    CUtensorMap w;
    CUtensorMap t[4];
};
__host__ __device__ constexpr int token_box_index(int half_rows) {
    return half_rows <= 16 ? 0 : half_rows <= 32 ? 1 : half_rows <= 64 ? 2 : 3;
}

struct PairParams {
    const int32_t *expert_offsets;
    int e_begin, ne;
    int num_kb;              // K blocks of BK
    int f_tiles;             // PM-row weight tiles per expert
    int a_rows_per_expert;   // rows between experts in A's tensor map
    int live_halves;         // CM-row halves of A per expert holding real weight rows;
                             // a tile's half 2f + c at or past it is skipped (rows
                             // past I / H: its loads, and gate_up's stores)
    __nv_bfloat16 *h;        // EPI_SWIGLU output [pairs, h_ld]
    int h_ld;
    __nv_bfloat16 *gu;       // EPI_SWIGLU, training: gate / up pre-activations
                             // [pairs, 2 h_ld] in packed column order, or nullptr
    __nv_bfloat16 *out_slots;   // EPI_DOWN output [pairs, H]
    const int32_t *perm;
    const float *topk_w;
    int H;
    int32_t *status;
};

struct Smem {
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = STAGES * A_BYTES;
    static constexpr uint32_t epi_off = b_off + STAGES * B_BYTES;      // 16 KB staging
    static constexpr uint32_t epi_bytes = 2 * CHUNK * GU_FEATS * 4;
    static constexpr uint32_t pairs_off = epi_off + epi_bytes;        // [PN] int + [PN] float
    static constexpr uint32_t bar_off = pairs_off + 2 * PN * 4;
    static constexpr uint32_t misc_off = bar_off + 24 * 8;
    static constexpr uint32_t tables_off = misc_off + 16;
    static constexpr uint32_t end = tables_off + 2 * (kMaxExperts + 1) * 4;
    static constexpr uint32_t alloc = end + 1024;   // slack to align the base to 1024
};
static_assert(CHUNK * CM * 2 <= Smem::epi_bytes, "down staging fits");
static_assert(Smem::alloc <= 227 * 1024, "shared memory per CTA");

// Tile -> expert i, weight tile f, token tile m (tokens fastest, so the pairs that run
// at the same time share the weight tile in L2) and its token count. gate_up cuts an
// expert's rows into 256-row tiles and a remainder; down (EVEN) splits them evenly over
// the same ceil(rows / 256) tiles (each a multiple of 32 but the last), so no tile is a
// short remainder that re-streams its weight tile for a fraction of the MMAs -- measured
// faster for down (gpt-oss 0.539 -> 0.519 ms) and slightly slower for gate_up.
struct Tile {
    int i, f, m, tok0, ntok, nmma;
};
template <bool EVEN>
__device__ __forceinline__ Tile tile_at(int t, const int *mtp, const int *eo, int ne, int f_tiles) {
    Tile r;
    decode_tile(t, mtp, ne, f_tiles, r.i, r.m, r.f);
    const int seg = eo[r.i + 1] - eo[r.i];
    const int ntiles = mtp[r.i + 1] - mtp[r.i];                    // ceil(seg / PN)
    const int base = EVEN ? ((seg + ntiles - 1) / ntiles + 31) & ~31 : PN;   // <= PN
    r.tok0 = eo[r.i] + r.m * base;
    r.ntok = min(base, seg - r.m * base);
    r.nmma = (r.ntok + 31) & ~31;   // pair MMA N: a multiple of 32, 32..256
    return r;
}

template <int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ PairMaps maps, const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    // The dynamic shared-memory base is the same in both CTAs, so is every offset below:
    // the pair MMA addresses both CTAs' tiles with the even CTA's descriptors.
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Smem::bar_off);
    uint64_t *full = bars;                  // [STAGES], used in the even CTA
    uint64_t *empty = bars + STAGES;        // [STAGES], both CTAs
    uint64_t *tfull = bars + 2 * STAGES;    // [2], both CTAs
    uint64_t *tempty = tfull + 2;           // [2], used in the even CTA (8 arrivals)
    uint64_t *mma_done = tempty + 2;        // [1], both CTAs
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::misc_off);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + Smem::misc_off + 4);
    int *eo = reinterpret_cast<int *>(smem + Smem::tables_off);
    int *mtp = eo + (kMaxExperts + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t cta = cluster_ctarank();   // 0 = even CTA (issues the MMAs)
    const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

    if (warp == 0) {
        if (lane < 5) tma_prefetch_desc(lane == 0 ? &maps.w : &maps.t[lane - 1]);
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else if (warp == 2 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);
        }
        mbar_init(mma_done, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dep_wait();   // the previous kernel's writes are visible from here on
    grid_dep_trigger();
    if (warp == 0) build_tile_tables(p.expert_offsets, p.e_begin, p.ne, PN, eo, mtp);
    fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers exist before any cross-CTA signal
    fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = mtp[p.ne] * p.f_tiles;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------ TMA producer
            const uint32_t full_even0 = mapa_shared(smem_u32(&full[0]), 0);
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int t = pair; ok && t < total; t += num_pairs) {
                const Tile tl = tile_at<EPI == EPI_DOWN>(t, mtp, eo, p.ne, p.f_tiles);
                const int w_row = (p.e_begin + tl.i) * p.a_rows_per_expert + tl.f * PM + cta * CM;
                const int t_row = tl.tok0 + (int)cta * (tl.nmma >> 1);
                const int bsel = token_box_index(tl.nmma >> 1);
                const CUtensorMap *tmap_t = &maps.t[bsel];
                // a weight half past the expert's real rows is not loaded: its MMA rows
                // are never stored
                const bool live0 = 2 * tl.f < p.live_halves, live1 = 2 * tl.f + 1 < p.live_halves;
                const bool a_live = cta == 0 ? live0 : live1;
                const uint32_t tx = (live0 ? A_BYTES : 0u) + (live1 ? A_BYTES : 0u) +
                                    2u * (uint32_t)(16 << bsel) * BK * 2;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    if (cta == 0) mbar_arrive_expect_tx(&full[stage], tx);
                    const uint32_t fb = full_even0 + stage * 8;
                    if (a_live)
                        tma_load_2d_pair(smem_u32(smem + Smem::a_off + stage * A_BYTES), &maps.w,
                                         fb, kb * BK, w_row);
                    tma_load_2d_pair(smem_u32(smem + Smem::b_off + stage * B_BYTES), tmap_t, fb,
                                     kb * BK, t_row);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // no copy may still be landing when the CTA exits: the even CTA's full
            // barriers count both CTAs' bytes
            if (cta == 0)
                for (int s = 0; s < STAGES; ++s)
                    if ((armed >> s) & 1u) {
                        volatile int no_abort = 0;
                        mbar_wait<true>(&full[s], (armed_parity >> s) & 1u, &no_abort, p.status);
                    }
        }
    } else if (warp == 1) {
        if (lane == 0 && cta == 0) {   // ---------------------------- MMA issuer (even CTA)
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, issued = false;
            for (int t = pair; ok && t < total; t += num_pairs) {
                const Tile tl = tile_at<EPI == EPI_DOWN>(t, mtp, eo, p.ne, p.f_tiles);
                const uint32_t idesc = make_idesc(PM, tl.nmma);
                if (!mbar_wait<true>(&tempty[acc], acc_phase ^ 1u, abort_s, p.status)) break;
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * PN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait<true>(&full[stage], phase, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t a_addr = smem_u32(smem + Smem::a_off + stage * A_BYTES);
                    const uint32_t b_addr = smem_u32(smem + Smem::b_off + stage * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16_pair(d_tmem, smem_desc_sw128(a_addr + kk * 32),
                                      smem_desc_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0);
                    issued = true;
                    commit_pair(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                commit_pair(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (issued) commit_pair(mma_done);   // every MMA done before TMEM is freed
        }
        if (lane == 0 && pair < total) {   // the pair had tiles, so MMAs were issued
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, p.status);
        }
    } else {   // ------------------------------------------------------ epilogue
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int etid = threadIdx.x - 64;   // 0..127 across the epilogue warps
        const uint32_t tempty_even0 = mapa_shared(smem_u32(&tempty[0]), 0);
        float *stage_f = reinterpret_cast<float *>(smem + Smem::epi_off);
        __nv_bfloat16 *stage_h = reinterpret_cast<__nv_bfloat16 *>(smem + Smem::epi_off);
        int *pair_s = reinterpret_cast<int *>(smem + Smem::pairs_off);      // [PN]
        float *wgt_s = reinterpret_cast<float *>(pair_s + PN);              // [PN]
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = pair; t < total; t += num_pairs) {
            const Tile tl = tile_at<EPI == EPI_DOWN>(t, mtp, eo, p.ne, p.f_tiles);
            if (EPI == EPI_DOWN) {
                // pair id and routing weight of every token of the tile, loaded while
                // the tile's MMAs run (the previous tile's readers passed a barrier)
#pragma unroll 2
                for (int j = etid; j < tl.nmma; j += 128) {
                    const bool tv = j < tl.ntok;
                    const int pr = tv ? p.perm[tl.tok0 + j] : -1;
                    pair_s[j] = pr;
                    wgt_s[j] = tv ? p.topk_w[pr] : 0.f;
                }
            }
            // tcgen05.ld is warp-collective and the epilogue warps share named
            // barriers: all four leave together on abort (the vote is also the barrier
            // after which the tile's pair ids are visible)
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_s, p.status);
            if (!epilogue_all(ok)) break;
            fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * PN);
            for (int c = 0; c < tl.nmma; c += CHUNK) {
                float v[32];
                tmem_ld32(taddr + c, v);
                if (c + CHUNK >= tl.nmma) {   // accumulator fully read: hand it back
                    fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_even0 + acc * 8);
                }
                if (EPI == EPI_SWIGLU) {
                    // lanes 0-63: gate rows, 64-127: up rows of the same 64 features.
                    // G[j][f] = gate, U[j][f] = up, j = token column in the chunk; the
                    // SwiGLU itself is spread over all 128 threads below.
                    float *dst = stage_f + (q >= 2 ? CHUNK * GU_FEATS : 0);
                    const int f = (q & 1) * 32 + lane;
#pragma unroll
                    for (int j = 0; j < CHUNK; ++j) dst[j * GU_FEATS + f] = v[j];
                    epilogue_sync();
                    // 32 tokens x 64 features: each thread writes two 8-feature vectors
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int item = etid + 128 * s;
                        const int j = item >> 3, f8 = (item & 7) * 8;
                        if (c + j < tl.ntok && 2 * tl.f + (int)cta < p.live_halves) {
                            const float4 *g4 = reinterpret_cast<const float4 *>(stage_f + j * GU_FEATS + f8);
                            const float4 *u4 = reinterpret_cast<const float4 *>(
                                stage_f + CHUNK * GU_FEATS + j * GU_FEATS + f8);
                            const float4 g0 = g4[0], g1 = g4[1], u0 = u4[0], u1 = u4[1];
                            const float hv[8] = {silu_fast(g0.x) * u0.x, silu_fast(g0.y) * u0.y,
                                                 silu_fast(g0.z) * u0.z, silu_fast(g0.w) * u0.w,
                                                 silu_fast(g1.x) * u1.x, silu_fast(g1.y) * u1.y,
                                                 silu_fast(g1.z) * u1.z, silu_fast(g1.w) * u1.w};
                            __nv_bfloat16 *out = p.h + (size_t)(tl.tok0 + c + j) * p.h_ld +
                                                 tl.f * (2 * GU_FEATS) + cta * GU_FEATS + f8;
                            *reinterpret_cast<uint4 *>(out) = pack8_bf16(hv);
                            if (p.gu != nullptr) {
                                const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                                const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                                __nv_bfloat16 *gd = p.gu + (size_t)(tl.tok0 + c + j) * 2 * p.h_ld +
                                                    (2 * tl.f + cta) * CM + f8;
                                *reinterpret_cast<uint4 *>(gd) = pack8_bf16(gv);
                                *reinterpret_cast<uint4 *>(gd + GU_FEATS) = pack8_bf16(uv);
                            }
                        }
                    }
                    epilogue_sync();
                } else {
                    const float w = wgt_s[c + lane];   // routing weight of token c + lane
                    const int f = q * 32 + lane;       // weight row of this CTA
#pragma unroll
                    for (int j = 0; j < CHUNK; ++j)
                        stage_h[j * CM + f] = __float2bfloat16_rn(__shfl_sync(0xffffffffu, w, j) * v[j]);
                    epilogue_sync();
                    // 32 tokens x 128 features: 16 vectors per token row
                    const int col0 = tl.f * PM + cta * CM;
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const int item = etid + 128 * s;
                        const int j = item >> 4, f8 = (item & 15) * 8;
                        const int prj = pair_s[c + j];
                        if (prj >= 0 && col0 + f8 < p.H)
                            *reinterpret_cast<uint4 *>(p.out_slots + (size_t)prj * p.H + col0 + f8) =
                                *reinterpret_cast<const uint4 *>(stage_h + j * CM + f8);
                    }
                    epilogue_sync();
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    fence_before();
    __syncthreads();
    cluster_sync_all();   // no CTA leaves while its peer may still signal its barriers
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

cudaError_t make_maps(PairMaps *m, const void *w, uint64_t w_rows, uint64_t w_cols, uint64_t w_ld,
                      const void *t, uint64_t t_rows, uint64_t t_cols, uint64_t t_ld) {
    cudaError_t e = make_map(&m->w, w, w_rows, w_cols, w_ld, CM);
    for (int b = 0; b < 4 && e == cudaSuccess; ++b)
        e = make_map(&m->t[b], t, t_rows, t_cols, t_ld, 16u << b);
    return e;
}

// Clusters of two that fit on the device at once (one CTA per SM), cached per kernel.
template <int EPI>
cudaError_t launch_pair(const PairMaps &maps, const PairParams &prm, int64_t max_tiles,
                        cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    auto kern = grouped_gemm_pair_kernel<EPI>;
    static int max_clusters_dev[64] = {};   // per device
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int &max_clusters = max_clusters_dev[dev];
    if (max_clusters == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Smem::alloc);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = Smem::alloc;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_clusters = n;
    }
    const int clusters = (int)std::min<int64_t>(max_tiles, max_clusters);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Smem::alloc;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps, prm);
}

}  // namespace

cudaError_t launch_tc_gate_up(const LayerDims &d, const void *send, const int32_t *expert_offsets,
                              int e_begin, int e_end, const void *packed, void *h, void *gu,
                              int32_t *status, int /*num_sms*/, cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    PairMaps maps;
    cudaError_t e = make_maps(&maps, packed, (uint64_t)d.E * 2 * d.Ipad, d.H, d.H, send, rows,
                              d.H, d.H);
    if (e != cudaSuccess) return e;
    PairParams prm = {};
    prm.expert_offsets = expert_offsets;
    prm.e_begin = e_begin;
    prm.ne = e_end - e_begin;
    prm.num_kb = ceil_div(d.H, BK);
    prm.f_tiles = 2 * d.Ipad / PM;
    prm.a_rows_per_expert = 2 * d.Ipad;
    prm.live_halves = ceil_div(d.I, GU_FEATS);
    prm.h = (__nv_bfloat16 *)h;
    prm.h_ld = d.Ipad;
    prm.gu = (__nv_bfloat16 *)gu;
    prm.H = d.H;
    prm.status = status;
    const int64_t max_tiles = (ceil_div64(rows, PN) + prm.ne) * prm.f_tiles;
    return launch_pair<EPI_SWIGLU>(maps, prm, max_tiles, s);
}

cudaError_t launch_tc_down(const LayerDims &d, const void *h, const int32_t *expert_offsets,
                           int e_begin, int e_end, const void *w_down, const int32_t *perm,
                           const float *topk_w, void *out_slots, int32_t *status, int /*num_sms*/,
                           cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    PairMaps maps;
    cudaError_t e = make_maps(&maps, w_down, (uint64_t)d.E * d.H, d.I, d.I, h, rows, d.I, d.Ipad);
    if (e != cudaSuccess) return e;
    PairParams prm = {};
    prm.expert_offsets = expert_offsets;
    prm.e_begin = e_begin;
    prm.ne = e_end - e_begin;
    prm.num_kb = ceil_div(d.I, BK);
    prm.f_tiles = ceil_div(d.H, PM);
    prm.a_rows_per_expert = d.H;
    prm.live_halves = ceil_div(d.H, CM);
    prm.out_slots = (__nv_bfloat16 *)out_slots;
    prm.perm = perm;
    prm.topk_w = topk_w;
    prm.H = d.H;
    prm.status = status;
    const int64_t max_tiles = (ceil_div64(rows, PN) + prm.ne) * prm.f_tiles;
    return launch_pair<EPI_DOWN>(maps, prm, max_tiles, s);
}

}  // namespace moe
