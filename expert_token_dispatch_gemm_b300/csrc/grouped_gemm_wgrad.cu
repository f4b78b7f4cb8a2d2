// Weight gradients of the local experts as grouped GEMMs on pairs of SMs. An expert's
// weight gradient sums over every row it received (Hugging Face "Expert parallelism"
// docs, "How the sizes combine"); the products are those of the chain rule through the
// experts of step 3 (Ultralytics glossary "Expert Parallelism"):
//   wgrad gate/up : dW_gu[f, h] = sum_r dgu_r[f] x_r[h]        (M = packed f, N = h)
//   wgrad down    : dW_d[h, i]  = sum_r dout_r[h] (w a)_r[i]    (M = h, N = i)
// with K = the rows r of the expert's segment. A (dgu or dout, token-major rows of the
// send layout) is read as an MN-major operand. B is a transposed copy of the other
// operand, [N][the 64-row blocks of every expert in turn], zero past each segment: it is
// K-major, and every K block of an expert is whole, so a row past a segment is only
// ever multiplied by zero (the A rows past the last segment are zeroed by the kernel
// that writes the transposed copy of x, so they are finite).
//
// One tile = 256 rows of M x 256 columns of N of one expert, computed by a cluster of
// two CTAs on two SMs with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): each CTA
// stages its 128 M rows of A (two 64-column MN-major boxes) and 128 of the B rows per
// 64-row K block (32 KB per stage) and holds its 128 accumulator rows in its own TMEM.
// (Pair MMAs whose B operand is MN-major and split over the two CTAs kept the tensor
// pipe under 30% busy; one-CTA tiles stage 48 KB per K block.)
// Per CTA (320 threads, one CTA per SM, persistent over the tile list):
//   warp 0      TMA producer, 4-stage ring; both CTAs' copies complete on the even CTA's
//               full barrier, which the even CTA arms with the pair's bytes;
//   warp 1      TMEM (two 128 x 256 fp32 accumulators in each CTA); in the even CTA one
//               thread issues the pair MMAs and commits them to both CTAs' barriers;
//   warps 2..9  epilogue, two warps per TMEM lane quarter: each takes 128 of the tile's
//               256 columns in one TMEM load; after all eight have loaded, one arrival
//               per CTA on the even CTA's accumulator-empty barrier hands the accumulator
//               back (per-warp cluster-scope arrivals stalled the warps on memory
//               barriers); then each warp stores its columns as two 64-column
//               chunks, each through its own 128-byte-swizzled 4 KB staging block into a
//               3-D TMA store (rows past I / H and columns past the output's width are
//               clipped by the map), so a warp's two stores are in flight together.
// An expert without rows gets zero gradients. Every mbarrier wait is bounded (about
// 2 s); on expiry the kernel records MOE_DEV_TIMEOUT in the status word, stops issuing
// work, waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include <mutex>

#include "tc_bwd.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int PM = 256;                 // M rows per tile (the pair MMA's M)
constexpr int CM = PM / 2;              // M rows per CTA (its TMEM lanes)
constexpr int BN = 256;                 // N columns per tile
constexpr int CN = BN / 2;              // B rows staged per CTA
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = CM * BK * 2;   // 16 KB: two 64-column MN-major boxes
constexpr uint32_t B_BYTES = CN * BK * 2;   // 16 KB
constexpr uint32_t MN_BOX = 64 * BK * 2;    // 8 KB
constexpr int NUM_THREADS = 320;
constexpr uint32_t TMEM_COLS = 2 * BN;

struct WgradMaps {
    CUtensorMap a;       // token-major rows [rows, M cols], box 64 x 64 (MN-major A)
    CUtensorMap b;       // transposed [N rows, padded K cols], box 64 x 128 (K-major B)
    CUtensorMap out[2];  // [E][rows][cols] outputs, box 64 x 32 (TMA stores)
};

struct WgradParams {
    const int32_t *expert_offsets;
    int ne;
    int m_tiles, n_tiles;    // pair M tiles of PM, N tiles of BN
    int I, H;
    int wgrad_gu;            // 1: M = packed gate/up rows (outputs dW_gate, dW_up);
                             // 0: M = hidden rows (output dW_down)
    uint32_t lbo, sbo;       // MN-major descriptor strides
    int32_t *status;
};

struct Smem {
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = STAGES * A_BYTES;
    static constexpr uint32_t epi_off = b_off + STAGES * B_BYTES;   // 8 warps x 2 x 4 KB
    static constexpr uint32_t bar_off = epi_off + 8 * 8192;
    static constexpr uint32_t misc_off = bar_off + 24 * 8;
    static constexpr uint32_t tables_off = misc_off + 16;
    static constexpr uint32_t end = tables_off + 2 * (kMaxExperts + 1) * 4;
    static constexpr uint32_t alloc = end + 1024;   // slack to align the base to 1024
};
static_assert(2 * STAGES + 5 <= 24, "barriers");
static_assert(Smem::alloc <= 227 * 1024, "shared memory per CTA");

// Tile t -> expert e, M tile mt, N tile nt (N fastest: the tiles running at the same
// time share their A rows in L2), the expert's rows and its first 64-row block of B.
struct Tile {
    int e, mt, nt, row0, nkb, kb0;
};
__device__ __forceinline__ Tile tile_at(int t, const int *eo, const int *pk, int m_tiles, int n_tiles) {
    Tile r;
    const int per = m_tiles * n_tiles;
    r.e = t / per;
    const int l = t - r.e * per;
    r.mt = l / n_tiles;
    r.nt = l - r.mt * n_tiles;
    r.row0 = eo[r.e];
    r.kb0 = pk[r.e];
    r.nkb = pk[r.e + 1] - r.kb0;
    return r;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_wgrad_kernel(const __grid_constant__ WgradMaps maps, const WgradParams p) {
    extern __shared__ uint8_t smem_raw[];
    // The dynamic shared-memory base is the same in both CTAs, so is every offset below:
    // the pair MMA addresses both CTAs' tiles with the even CTA's descriptors.
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Smem::bar_off);
    uint64_t *full = bars;                  // [STAGES], used in the even CTA
    uint64_t *empty = bars + STAGES;        // [STAGES], both CTAs
    uint64_t *tfull = bars + 2 * STAGES;    // [2], both CTAs
    uint64_t *tempty = tfull + 2;           // [2], used in the even CTA (one arrival per CTA)
    uint64_t *mma_done = tempty + 2;        // [1], both CTAs
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::misc_off);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + Smem::misc_off + 4);
    int *eo = reinterpret_cast<int *>(smem + Smem::tables_off);
    int *pk = eo + (kMaxExperts + 1);   // 64-row blocks of the experts before e

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t cta = cluster_ctarank();   // 0 = even CTA (issues the MMAs)
    const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

    if (warp == 0) {
        if (lane < 4) tma_prefetch_desc(lane == 0 ? &maps.a : lane == 1 ? &maps.b : &maps.out[lane - 2]);
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
            mbar_init(&tempty[a], 2);   // the epilogue of each CTA
        }
        mbar_init(mma_done, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dep_wait();   // the previous kernels' writes are visible from here on
    grid_dep_trigger();
    if (warp == 0) build_tile_tables(p.expert_offsets, 0, p.ne, 64, eo, pk);
    fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers exist before any cross-CTA signal
    fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = p.ne * p.m_tiles * p.n_tiles;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------ TMA producer
            const uint32_t full_even0 = mapa_shared(smem_u32(&full[0]), 0);
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int t = pair; ok && t < total; t += num_pairs) {
                const Tile tl = tile_at(t, eo, pk, p.m_tiles, p.n_tiles);
                const int a_x = (2 * tl.mt + (int)cta) * CM;
                const int b_y = tl.nt * BN + (int)cta * CN;
                for (int kb = 0; kb < tl.nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    if (cta == 0) mbar_arrive_expect_tx(&full[stage], 2u * (A_BYTES + B_BYTES));
                    const uint32_t fb = full_even0 + stage * 8;
                    const uint32_t a_dst = smem_u32(smem + Smem::a_off + stage * A_BYTES);
                    const int y = tl.row0 + kb * BK;
                    tma_load_2d_pair(a_dst, &maps.a, fb, a_x, y);
                    tma_load_2d_pair(a_dst + MN_BOX, &maps.a, fb, a_x + 64, y);
                    tma_load_2d_pair(smem_u32(smem + Smem::b_off + stage * B_BYTES), &maps.b, fb,
                                     (tl.kb0 + kb) * BK, b_y);
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
            bool ok = true;
            const uint32_t idesc = make_idesc(PM, BN) | (1u << 15);   // A MN-major, B K-major
            for (int t = pair; ok && t < total; t += num_pairs) {
                const Tile tl = tile_at(t, eo, pk, p.m_tiles, p.n_tiles);
                if (!mbar_wait<true>(&tempty[acc], acc_phase ^ 1u, abort_s, p.status)) break;
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < tl.nkb; ++kb) {
                    if (!mbar_wait<true>(&full[stage], phase, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t a_addr = smem_u32(smem + Smem::a_off + stage * A_BYTES);
                    const uint32_t b_addr = smem_u32(smem + Smem::b_off + stage * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_bf16_pair(d_tmem, smem_desc_mn_sw128(a_addr + kk * 2048, p.lbo, p.sbo),
                                      smem_desc_sw128(b_addr + kk * 32), idesc, (kb | kk) != 0);
                    commit_pair(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                commit_pair(&tfull[acc]);   // after no K block: arrives at once
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA done before TMEM is freed (a pair with tiles commits, MMAs or not)
            if (pair < total) commit_pair(mma_done);
        }
        if (lane == 0 && pair < total) {
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, p.status);
        }
    } else {   // ------------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;        // accumulator columns 128 half ..
        const uint32_t tempty_even0 = mapa_shared(smem_u32(&tempty[0]), 0);
        uint8_t *bufs = smem + Smem::epi_off + (warp - 2) * 8192;
        int last = -1;   // staging block read by the warp's most recent store
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = pair; t < total; t += num_pairs) {
            const Tile tl = tile_at(t, eo, pk, p.m_tiles, p.n_tiles);
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_s, p.status);
            // tcgen05.ld is warp-collective: the epilogue warps leave together on abort
            if (!epi8_all(ok)) break;
            fence_after();
            // This CTA's accumulator rows are M block 2 mt + cta; the warp's 32 rows are
            // 32 consecutive rows of one output.
            const int blk = 2 * tl.mt + (int)cta;
            int sel = 0, r0 = blk * CM + q * 32, ncols = p.I;
            if (p.wgrad_gu) {
                sel = q >= 2 ? 1 : 0;                  // gate rows, then up rows
                r0 = blk * 64 + (q & 1) * 32;
                ncols = p.H;
            }
            const bool live = r0 < (p.wgrad_gu ? p.I : p.H);
            const int c2 = 128 * half;
            const bool cols_live = tl.nt * BN + c2 < ncols;   // uniform over the warp
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            float v[128];
            if (cols_live) {
                if (tl.nkb > 0) {
                    tmem_ld128(taddr + c2, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 128; ++j) v[j] = 0.f;   // an expert with no rows
                }
            }
            // the CTA's accumulator is read: hand it back (one cluster-scope arrival per
            // CTA after the epilogue warps' barrier)
            fence_before();
            epi8_sync();
            if (warp == 2 && lane == 0) mbar_arrive_cluster(tempty_even0 + acc * 8);
            if (live && cols_live) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int col0 = tl.nt * BN + c2 + 64 * h;
                    if (col0 >= ncols) break;
                    // the store that last read this staging block is done: it is the
                    // warp's most recent store, or the one before it
                    uint8_t *buf = bufs + h * 4096;
                    if (lane == 0) {
                        if (last == h)
                            tma_store_wait_read();
                        else
                            tma_store_wait_read1();
                    }
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4 *>(buf + lane * 128 + ((j ^ (lane & 7)) * 16)) =
                            pack8_bf16(v + 64 * h + 8 * j);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) tma_store_3d(&maps.out[sel], smem_u32(buf), col0, r0, tl.e);
                    last = h;
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) tma_store_wait_all();   // stores done, staging free
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

// Clusters of two that fit on the device at once (one CTA per SM), cached per device.
cudaError_t launch_wgrad(const WgradMaps &maps, WgradParams prm, int64_t max_tiles, cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    // MN-major descriptor strides: 64-element groups one 8 KB box apart, 8-row K groups
    // one 1024-byte swizzle atom apart
    prm.lbo = MN_BOX;
    prm.sbo = 1024;
    auto kern = grouped_gemm_wgrad_kernel;
    static std::mutex mu;
    static int clusters_dev[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int max_clusters;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (clusters_dev[dev] == 0) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
            clusters_dev[dev] = n;
        }
        max_clusters = clusters_dev[dev];
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

int64_t wgrad_t_cols(const LayerDims &d) {
    return ((int64_t)d.N * d.k + 63) / 64 * 64 + 64LL * d.E;
}

cudaError_t launch_tc_wgrad_gate_up(const LayerDims &d, const void *dgu, const void *xT,
                                    const int32_t *eoff, void *dw_gate, void *dw_up,
                                    int32_t *status, cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    WgradMaps maps = {};
    // A = dgu [rows, 2 Ipad] (M = packed gate/up feature); B = x^T [H, t_cols]
    cudaError_t e = make_map(&maps.a, dgu, rows, 2 * d.Ipad, 2 * d.Ipad, 64);
    if (e == cudaSuccess) e = make_map(&maps.b, xT, d.H, wgrad_t_cols(d), wgrad_t_cols(d), CN);
    if (e == cudaSuccess) e = make_store_map_3d(&maps.out[0], dw_gate, d.H, d.I, d.E, 64, 32);
    if (e == cudaSuccess) e = make_store_map_3d(&maps.out[1], dw_up, d.H, d.I, d.E, 64, 32);
    if (e != cudaSuccess) return e;
    WgradParams prm = {};
    prm.expert_offsets = eoff;
    prm.ne = d.E;
    prm.m_tiles = 2 * d.Ipad / PM;
    prm.n_tiles = ceil_div(d.H, BN);
    prm.I = d.I;
    prm.H = d.H;
    prm.wgrad_gu = 1;
    prm.status = status;
    return launch_wgrad(maps, prm, (int64_t)d.E * prm.m_tiles * prm.n_tiles, s);
}

cudaError_t launch_tc_wgrad_down(const LayerDims &d, const void *dout_send, const void *waT,
                                 const int32_t *eoff, void *dw_down, int32_t *status,
                                 cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    WgradMaps maps = {};
    // A = dout in the send layout [rows, H] (M = h); B = (w a)^T [Ipad, t_cols]
    cudaError_t e = make_map(&maps.a, dout_send, rows, d.H, d.H, 64);
    if (e == cudaSuccess) e = make_map(&maps.b, waT, d.Ipad, wgrad_t_cols(d), wgrad_t_cols(d), CN);
    if (e == cudaSuccess) e = make_store_map_3d(&maps.out[0], dw_down, d.I, d.H, d.E, 64, 32);
    if (e == cudaSuccess) maps.out[1] = maps.out[0];
    if (e != cudaSuccess) return e;
    WgradParams prm = {};
    prm.expert_offsets = eoff;
    prm.ne = d.E;
    prm.m_tiles = ceil_div(d.H, PM);
    prm.n_tiles = ceil_div(d.I, BN);
    prm.I = d.I;
    prm.H = d.H;
    prm.wgrad_gu = 0;
    prm.status = status;
    return launch_wgrad(maps, prm, (int64_t)d.E * prm.m_tiles * prm.n_tiles, s);
}

}  // namespace moe
