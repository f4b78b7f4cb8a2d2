// Step 3 -- the local experts as grouped GEMMs on the 5th-generation tensor cores
// (Ultralytics glossary "Expert Parallelism", step 3: each partition runs its local
// experts on the rows it received; Hugging Face "Expert parallelism" docs: the
// "grouped_gemm" rule splits expert weights along the expert dimension).
//
// Three instantiations of one persistent, warp-specialised kernel:
//   gate_up : h = silu(x W_g^T) * (x W_u^T)      A = send [rows, H], B = packed gate/up
//   down    : out_slots[perm[r]] = w * (h W_d^T)  A = h [rows, I],    B = W_d [E*H, I]
//   route   : logits = x W_r^T (+ b), then top-k / softmax / segment histogram in the
//             epilogue (Ultralytics glossary, step 1): A = x [N, H], B = W_r [E, H],
//             MMA N = E rounded up to 16; each epilogue thread owns one token's logits.
// The tile space is (expert, n tile, m tile) over variable-length expert segments; a
// 128-row M tile may run past its segment, those rows are computed on neighbouring
// data and never stored.
//
// Per CTA (one per SM, 192 threads):
//   warp 0      TMA producer: 128x64 A tile + 256x64 B tile per stage, 128-byte swizzle,
//               4-stage ring guarded by full/empty mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators) and one
//               thread issues tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 acc);
//               tcgen05.commit frees smem stages and publishes finished accumulators;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows of their TMEM lane quarter,
//               SwiGLU or weighting, bf16 stores; the accumulator is released for the
//               next-but-one tile so MMA and epilogue overlap.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records
// MOE_DEV_TIMEOUT in the status word, stops issuing work, waits (bounded) for its own
// copies and MMAs in flight, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = kTcBlockM;   // 128
constexpr int BN = 256;
constexpr int BK = 64;          // 64 bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bit 17,
// M >> 4 at bit 24.
constexpr uint32_t make_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

enum { EPI_SWIGLU = 0, EPI_DOWN = 1, EPI_ROUTE = 2 };
static_assert(BM == 2 * kSegTokens, "a route tile covers two histogram segments");

struct TcParams {
    const int32_t *expert_offsets;   // nullptr: one segment of `rows` rows (routing)
    int rows;
    int e_begin, ne;
    int bn;                  // MMA N of every tile (multiple of 16, <= BN)
    uint32_t idesc;
    int num_kb;              // K blocks of BK
    int n_tiles;             // N tiles per expert
    int b_rows_per_expert;   // rows between experts in B's tensor map
    __nv_bfloat16 *h;        // EPI_SWIGLU output, row stride h_ld
    int h_ld;
    __nv_bfloat16 *out_slots;   // EPI_DOWN output [pairs, H]
    const int32_t *perm;
    const float *topk_w;
    int H;
    // EPI_ROUTE
    int E, k, nseg;
    const float *bias;       // [E] or nullptr
    int32_t *route_idx;      // [N, k] out
    float *route_w;          // [N, k] out
    int32_t *seg_hist;       // [nseg, E] or nullptr
    int32_t *status;         // or nullptr
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Waits for the phase of `parity` to complete. Gives up (returns false) after
// kWaitLimitNs or once another role of the CTA has given up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_s,
                                          int32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*abort_s) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort_s = 1;
                if (status != nullptr) atomicOr(status, MOE_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor for a K-major tile written by TMA with 128-byte
// swizzle: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart (stride byte
// offset), leading byte offset unused for this layout, descriptor version 1 at bit 46,
// swizzle mode 2 (128B) at bits 61-63. Advancing K by 16 elements inside the 128-byte
// row adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
// 32 consecutive fp32 accumulator columns of this thread's TMEM lane; the wait is in the
// same statement so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__device__ __forceinline__ uint4 pack8_bf16(const float *f) {
    uint4 v;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

// Sorted (descending) top-KMAX list in registers; empty slots have idx < 0. A new value
// enters behind equal ones, so scanning experts in increasing id keeps ties ordered by
// the lower id.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&val)[KMAX], int (&idx)[KMAX], float v, int e) {
    if (!(v > val[KMAX - 1] || idx[KMAX - 1] < 0)) return;
#pragma unroll
    for (int j = KMAX - 1; j > 0; --j) {
        const bool beat_prev = v > val[j - 1] || idx[j - 1] < 0;
        const bool beat_cur = v > val[j] || idx[j] < 0;
        if (beat_prev) {
            val[j] = val[j - 1];
            idx[j] = idx[j - 1];
        } else if (beat_cur) {
            val[j] = v;
            idx[j] = e;
        }
    }
    if (v > val[0] || idx[0] < 0) {
        val[0] = v;
        idx[0] = e;
    }
}

// Barrier among the four epilogue warps only.
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct SmemLayout {
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = STAGES * A_BYTES;
    static constexpr uint32_t bar_off = STAGES * STAGE_BYTES;
    static constexpr uint32_t misc_off = bar_off + 16 * 8;
    static constexpr uint32_t tables_off = misc_off + 16;
    static constexpr uint32_t bias_off = tables_off + 2 * (kMaxExperts + 1) * 4;
    static constexpr uint32_t hist_off = bias_off + kMaxExperts * 4;
    static constexpr uint32_t end = hist_off + 2 * kMaxExperts * 4;
    static constexpr uint32_t alloc = end + 1024;   // slack to align the base to 1024
};

template <int EPI, int KMAX>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_b, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SmemLayout::bar_off);
    uint64_t *full = bars;                  // [STAGES]
    uint64_t *empty = bars + STAGES;        // [STAGES]
    uint64_t *tfull = bars + 2 * STAGES;    // [2]
    uint64_t *tempty = tfull + 2;           // [2]
    uint64_t *mma_done = tempty + 2;        // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + SmemLayout::misc_off);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + SmemLayout::misc_off + 4);
    int *eo = reinterpret_cast<int *>(smem + SmemLayout::tables_off);
    int *mtp = eo + (kMaxExperts + 1);
    float *bias_s = reinterpret_cast<float *>(smem + SmemLayout::bias_off);
    int *hist_s = reinterpret_cast<int *>(smem + SmemLayout::hist_off);   // [2][E]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0) {
        if (p.expert_offsets != nullptr) {
            build_tile_tables(p.expert_offsets, p.e_begin, p.ne, BM, eo, mtp);
        } else if (lane == 0) {
            eo[0] = 0;
            eo[1] = p.rows;
            mtp[0] = 0;
            mtp[1] = (p.rows + BM - 1) / BM;
        }
        if (lane == 0) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_b);
        }
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else if (warp == 3) {
        if (EPI == EPI_ROUTE)
            for (int e = lane; e < p.E; e += 32) bias_s[e] = p.bias != nullptr ? p.bias[e] : 0.f;
    } else if (warp == 2 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(mma_done, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = mtp[p.ne] * p.n_tiles;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                int i, m, n;
                decode_tile(tile, mtp, p.ne, p.n_tiles, i, m, n);
                const int a_row = eo[i] + m * BM;
                const int b_row = (p.e_begin + i) * p.b_rows_per_expert + n * BN;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], A_BYTES + (uint32_t)p.bn * BK * 2);
                    const uint32_t fb = smem_u32(&full[stage]);
                    tma_load_2d(smem_u32(smem + SmemLayout::a_off + stage * A_BYTES), &tmap_a, fb,
                                kb * BK, a_row);
                    tma_load_2d(smem_u32(smem + SmemLayout::b_off + stage * B_BYTES), &tmap_b, fb,
                                kb * BK, b_row);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
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
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued = false, ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_s, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + SmemLayout::a_off + stage * A_BYTES);
                    const uint32_t b_addr = smem_u32(smem + SmemLayout::b_off + stage * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(d_tmem, smem_desc_sw128(a_addr + kk * 32),
                                  smem_desc_sw128(b_addr + kk * 32), p.idesc, (kb | kk) != 0);
                    issued = true;
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (issued) {   // every MMA done before TMEM is freed
                umma_commit(mma_done);
                volatile int no_abort = 0;
                mbar_wait(mma_done, 0, &no_abort, p.status);
            }
        }
    } else {   // ------------------------------------------------------ epilogue
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int r = q * 32 + lane;      // accumulator row = tile row
        int acc = 0;
        uint32_t acc_phase = 0;
        const int etid = threadIdx.x - 64;   // 0..127 across the epilogue warps
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int i, m, n;
            decode_tile(tile, mtp, p.ne, p.n_tiles, i, m, n);
            if (EPI == EPI_ROUTE) {   // previous tile's histogram is flushed; clear it
                epilogue_sync();
                for (int j = etid; j < 2 * p.E; j += 128) hist_s[j] = 0;
                epilogue_sync();
            }
            // tcgen05.ld is warp-collective: the whole warp leaves together on abort
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_s, p.status);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int seg_row = m * BM + r;
            const bool valid = seg_row < eo[i + 1] - eo[i];
            const int grow = eo[i] + seg_row;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (EPI == EPI_ROUTE) {
                float val[KMAX];
                int idx[KMAX];
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    val[j] = -INFINITY;
                    idx[j] = -1;
                }
                for (int c = 0; c < p.bn; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = c + j;
                        if (e < p.E) {
                            const float l = v[j] + bias_s[e];
                            topk_insert<KMAX>(val, idx, isnan(l) ? -INFINITY : l, e);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);   // logits are in registers: free the accumulator
                if (valid) {
                    float ex[KMAX], sum = 0.f;
#pragma unroll
                    for (int j = 0; j < KMAX; ++j) {
                        ex[j] = j < p.k ? expf(val[j] - val[0]) : 0.f;
                        sum += ex[j];
                    }
                    const float inv = 1.0f / sum;
#pragma unroll
                    for (int j = 0; j < KMAX; ++j)
                        if (j < p.k) {
                            p.route_idx[(size_t)grow * p.k + j] = idx[j];
                            p.route_w[(size_t)grow * p.k + j] = ex[j] * inv;
                            if (p.seg_hist != nullptr)
                                atomicAdd(&hist_s[(r >> 6) * p.E + idx[j]], 1);
                        }
                }
                if (p.seg_hist != nullptr) {
                    epilogue_sync();
                    for (int j = etid; j < 2 * p.E; j += 128) {
                        const int seg = 2 * m + j / p.E;
                        if (seg < p.nseg) p.seg_hist[(size_t)seg * p.E + j % p.E] = hist_s[j];
                    }
                }
            } else if (EPI == EPI_SWIGLU) {
                __nv_bfloat16 *dst = p.h + (size_t)grow * p.h_ld + n * (BN / 2);
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    float g[32], u[32];
                    tmem_ld32(taddr + c, g);
                    tmem_ld32(taddr + BN / 2 + c, u);
                    if (valid) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            float hv[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) hv[e] = silu_f(g[v * 8 + e]) * u[v * 8 + e];
                            *reinterpret_cast<uint4 *>(dst + c + v * 8) = pack8_bf16(hv);
                        }
                    }
                }
            } else {
                int pair = 0;
                float w = 0.f;
                if (valid) {
                    pair = p.perm[grow];
                    w = p.topk_w[pair];
                }
                __nv_bfloat16 *dst = p.out_slots + (size_t)pair * p.H;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float y[32];
                    tmem_ld32(taddr + c, y);
                    const int col = n * BN + c;
                    if (valid) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            if (col + v * 8 < p.H) {
                                float o[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) o[e] = w * y[v * 8 + e];
                                *reinterpret_cast<uint4 *>(dst + col + v * 8) = pack8_bf16(o);
                            }
                        }
                    }
                }
            }
            if (EPI != EPI_ROUTE) {
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
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

// 2-D bf16 tensor map of a row-major [rows, cols] matrix with row stride `ld` elements,
// box of box_rows x 64 columns, 128-byte swizzle, out-of-range elements read as zero.
cudaError_t make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint64_t ld,
                     uint32_t box_rows) {
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

template <int EPI, int KMAX>
cudaError_t launch_tc(const CUtensorMap &ma, const CUtensorMap &mb, const TcParams &prm,
                      int max_tiles, int num_sms, cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    auto kern = grouped_gemm_tc_kernel<EPI, KMAX>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SmemLayout::alloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int grid = max_tiles < num_sms ? max_tiles : num_sms;
    kern<<<grid, NUM_THREADS, SmemLayout::alloc, s>>>(ma, mb, prm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gate_up(const LayerDims &d, const void *send, const int32_t *expert_offsets,
                              int e_begin, int e_end, const void *packed, void *h,
                              int32_t *status, int num_sms, cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    CUtensorMap ma, mb;
    cudaError_t e = make_map(&ma, send, rows, d.H, d.H, BM);
    if (e != cudaSuccess) return e;
    e = make_map(&mb, packed, (uint64_t)d.E * 2 * d.Ipad, d.H, d.H, BN);
    if (e != cudaSuccess) return e;
    TcParams prm = {};
    prm.expert_offsets = expert_offsets;
    prm.e_begin = e_begin;
    prm.ne = e_end - e_begin;
    prm.bn = BN;
    prm.idesc = make_idesc(BM, BN);
    prm.num_kb = ceil_div(d.H, BK);
    prm.n_tiles = 2 * d.Ipad / BN;
    prm.b_rows_per_expert = 2 * d.Ipad;
    prm.h = (__nv_bfloat16 *)h;
    prm.h_ld = d.Ipad;
    prm.H = d.H;
    prm.status = status;
    const int64_t max_tiles = (ceil_div64(rows, BM) + prm.ne) * prm.n_tiles;
    return launch_tc<EPI_SWIGLU, 1>(ma, mb, prm, (int)std::min<int64_t>(max_tiles, 1 << 30),
                                    num_sms, s);
}

cudaError_t launch_tc_down(const LayerDims &d, const void *h, const int32_t *expert_offsets,
                           int e_begin, int e_end, const void *w_down, const int32_t *perm,
                           const float *topk_w, void *out_slots, int32_t *status, int num_sms,
                           cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    CUtensorMap ma, mb;
    cudaError_t e = make_map(&ma, h, rows, d.I, d.Ipad, BM);
    if (e != cudaSuccess) return e;
    e = make_map(&mb, w_down, (uint64_t)d.E * d.H, d.I, d.I, BN);
    if (e != cudaSuccess) return e;
    TcParams prm = {};
    prm.expert_offsets = expert_offsets;
    prm.e_begin = e_begin;
    prm.ne = e_end - e_begin;
    prm.bn = BN;
    prm.idesc = make_idesc(BM, BN);
    prm.num_kb = ceil_div(d.I, BK);
    prm.n_tiles = ceil_div(d.H, BN);
    prm.b_rows_per_expert = d.H;
    prm.out_slots = (__nv_bfloat16 *)out_slots;
    prm.perm = perm;
    prm.topk_w = topk_w;
    prm.H = d.H;
    prm.status = status;
    const int64_t max_tiles = (ceil_div64(rows, BM) + prm.ne) * prm.n_tiles;
    return launch_tc<EPI_DOWN, 1>(ma, mb, prm, (int)std::min<int64_t>(max_tiles, 1 << 30),
                                  num_sms, s);
}

cudaError_t launch_tc_route(const LayerDims &d, const void *x, const void *w_router,
                            const float *bias, int32_t *topk_idx, float *topk_w,
                            int32_t *seg_hist, int32_t *status, int num_sms, cudaStream_t s) {
    const int bn = (d.E + 15) / 16 * 16;
    CUtensorMap ma, mb;
    cudaError_t e = make_map(&ma, x, d.N, d.H, d.H, BM);
    if (e != cudaSuccess) return e;
    e = make_map(&mb, w_router, d.E, d.H, d.H, (uint32_t)bn);
    if (e != cudaSuccess) return e;
    TcParams prm = {};
    prm.expert_offsets = nullptr;
    prm.rows = d.N;
    prm.e_begin = 0;
    prm.ne = 1;
    prm.bn = bn;
    prm.idesc = make_idesc(BM, bn);
    prm.num_kb = ceil_div(d.H, BK);
    prm.n_tiles = 1;
    prm.b_rows_per_expert = 0;
    prm.H = d.H;
    prm.E = d.E;
    prm.k = d.k;
    prm.nseg = ceil_div(d.N, kSegTokens);
    prm.bias = bias;
    prm.route_idx = topk_idx;
    prm.route_w = topk_w;
    prm.seg_hist = seg_hist;
    prm.status = status;
    const int tiles = ceil_div(d.N, BM);
    if (d.k <= 8) return launch_tc<EPI_ROUTE, 8>(ma, mb, prm, tiles, num_sms, s);
    return launch_tc<EPI_ROUTE, 32>(ma, mb, prm, tiles, num_sms, s);
}

}  // namespace moe
