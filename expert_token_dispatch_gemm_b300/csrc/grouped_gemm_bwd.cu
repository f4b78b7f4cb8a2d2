// Backward of the local experts, the dgrad GEMMs on the tensor cores. The chain rule
// through y = W_d (silu(g) * u), g = W_g x, u = W_u x of every kept (token, expert) pair
// (Ultralytics glossary "Expert Parallelism", step 3). Per send row r (pair of token t,
// weight w) with upstream gradient dout_t:
//   dgrad_down : da_u[i, r] = sum_h W_d[h, i] dout_t[h]       (tokens on N, K = H)
//                epilogue: a = silu(g) u, dweight_r += da_u . a (the routing weight's
//                gradient), dg = w da_u u silu'(g), du = w da_u silu(g) into the dgu
//                rows, and (w a)^T in the transposed layout of the weight-gradient GEMMs
//                (grouped_gemm_wgrad.cu)
//   dgrad_gu   : dx_r[h] = sum_f W_gu[f, h] dgu_r[f]           (tokens on N, K = 2 Ipad)
// The weights stay in their forward layouts: the GEMMs read them as MN-major A operands
// (M = the weight's column index), so nothing is transposed in memory.
//
// dgrad-gate/up: one tile = 256 weight columns (M) x up to 256 tokens (N) of one expert,
// computed by a cluster of two CTAs on two SMs with tcgen05.mma.cta_group::2 (M = 256,
// K = 16): each CTA stages its 128 M columns of A and half of the tokens (K-major B, the
// case in which the pair MMA runs at full rate), 32 KB per K block, and holds its 128
// accumulator rows in its own TMEM. dgrad-down: one CTA per tile of 128 weight columns x
// up to 256 tokens (cta_group::1), 48 KB per K block. Per CTA (320 threads, one CTA per
// SM, persistent over its tiles):
//   warp 0      TMA producer, ring of 6 (pairs) or 4 stages (A: 128 x 64, B: up to 128 or
//               256 x 64; 128-byte swizzle). MN-major tiles are 64-element boxes: one
//               128-byte row per K. A pair's copies complete on the even CTA's barrier.
//   warp 1      TMEM (two 128 x 256 fp32 accumulators in each CTA); lane 0 (of the even
//               CTA in a pair) issues the MMAs and commits them.
//   warps 2..9  epilogue, two warps per TMEM lane quarter taking alternate 16-token
//               chunks, each half with its own named barrier; each warp arrives on the
//               (even CTA's) accumulator-empty barrier after its last TMEM read; in a pair
//               without release semantics, so that the arrival does not wait for the
//               warp's earlier global stores.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records
// MOE_DEV_TIMEOUT in the status word, stops issuing work, waits (bounded) for its own
// copies and MMAs, frees TMEM and returns.
#include <mutex>

#include "tc_bwd.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;                 // M rows per tile (TMEM lanes)
constexpr int PM = 2 * BM;              // M rows per pair tile (the pair MMA's M)
constexpr int BN = 256;                 // max N per tile
constexpr int CN = BN / 2;              // token rows staged per CTA
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t MN_BOX = 64 * BK * 2;    // one 64-element x 64-row MN-major box: 8 KB
// Threads: producer warp, MMA warp and 8 epilogue warps (two per TMEM lane quarter).
template <int KIND> constexpr int num_threads() { return 320; }
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int CHUNK = 32;

enum { BWD_DGRAD_DOWN = 0, BWD_DGRAD_GU = 1 };

// Token maps with box heights 16, 32, 64, 128 and 256 rows (K-major B: a CTA stages a
// tile's tokens, or half of them in a pair).
struct BwdMaps {
    CUtensorMap a;       // MN-major A: box 64 x 64
    CUtensorMap b[5];    // token rows (K-major)
};
__host__ __device__ constexpr int token_box_index(int rows) {
    return rows <= 16 ? 0 : rows <= 32 ? 1 : rows <= 64 ? 2 : rows <= 128 ? 3 : 4;
}

struct BwdParams {
    const int32_t *expert_offsets;
    int ne;                  // experts (all of the layer)
    int num_kb;              // dgrad: K blocks of BK
    int m_tiles;             // pair M tiles of PM
    int m_blocks;            // M blocks of BM that hold output columns (a last pair tile
                             // may have one past them, whose results are not stored)
    int a_rows_per_expert;   // dgrad: rows between experts in A's map (K rows)
    uint32_t lbo, sbo;       // MN-major descriptor strides
    int I, Ipad, H;
    // dgrad_down
    const __nv_bfloat16 *gu;      // [rows, 2 Ipad] saved gate / up pre-activations
    __nv_bfloat16 *dgu;           // [rows, 2 Ipad] out
    __nv_bfloat16 *waT;           // [Ipad, ldt] out: (w * silu(g) * u)^T, the 64-row
    int64_t ldt;                  // blocks of every expert in turn, zero past each segment
    float *dweight_part;          // [m_tiles, rows] out
    int rows;                     // send rows of the buffers (N * k)
    // dgrad_down / dgrad_gu
    const int32_t *perm;
    const float *topk_w;
    __nv_bfloat16 *dx_slots;      // dgrad_gu: [N*k, H] out (row = pair id)
    int32_t *status;
};

// Ring (pairs: 6 stages of 32 KB per CTA; one CTA per tile: 4 of 48 KB), a 16 KB staging
// block, the token tile's pair ids and weights and the tile tables (dgrad-down also the
// 64-row block prefix of (w a)^T's columns).
template <int KIND>
struct Smem {
    // dgrad-gate/up runs on SM pairs; dgrad-down, whose epilogue is the heavier, one CTA
    // per tile (on pairs the two CTAs' epilogues gate each other's accumulators: measured
    // 0.73 -> 0.85 ms at gpt-oss, against 1.08 -> 1.01 ms for dgrad-gate/up)
    static constexpr bool PAIR = KIND == BWD_DGRAD_GU;
    static constexpr uint32_t B_BYTES = (PAIR ? CN : BN) * BK * 2;
    static constexpr int STAGES = PAIR ? 6 : 4;
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = STAGES * A_BYTES;
    static constexpr uint32_t epi_off = b_off + STAGES * B_BYTES;
    static constexpr uint32_t epi_bytes = CHUNK * BM * 4;
    static constexpr uint32_t pairs_off = epi_off + epi_bytes;       // [BN] int + [BN] float
    static constexpr uint32_t bar_off = pairs_off + 2 * BN * 4;
    static constexpr uint32_t misc_off = bar_off + 24 * 8;
    static constexpr uint32_t tables_off = misc_off + 16;
    static constexpr uint32_t end = tables_off + 4 * (kMaxExperts + 1) * 4;
    static constexpr uint32_t alloc = end + 1024;
};
static_assert(Smem<BWD_DGRAD_DOWN>::alloc <= 227 * 1024 && Smem<BWD_DGRAD_GU>::alloc <= 227 * 1024,
              "shared memory per CTA");

// Tile of a dgrad GEMM: expert i, M tile f, token tile m; tokens fastest. The MMA's N is
// the tile's tokens rounded up to 32, to 64 in dgrad-down, whose epilogue then writes
// every column of the expert's last 64-row block of (w a)^T (zeros past the segment).
struct DTile {
    int i, f, m, tok0, ntok, nmma;
};
template <int KIND>
__device__ __forceinline__ DTile dtile_at(int t, const int *mtp, const int *eo, int ne, int m_tiles) {
    DTile r;
    decode_tile(t, mtp, ne, m_tiles, r.i, r.m, r.f);
    const int seg = eo[r.i + 1] - eo[r.i];
    // dgrad-down splits an expert's rows evenly over its ceil(rows / 256) token tiles (a
    // multiple of 64 each but the last), so that no tile is a short remainder: the tiles
    // of an expert then take about as long, and the adjacent CTAs running them stay
    // together and share the weight strip in L2
    const int ntiles = mtp[r.i + 1] - mtp[r.i];
    const int base = KIND == BWD_DGRAD_DOWN ? ((seg + ntiles - 1) / ntiles + 63) & ~63 : BN;
    r.tok0 = eo[r.i] + r.m * base;
    r.ntok = min(base, seg - r.m * base);
    r.nmma = KIND == BWD_DGRAD_DOWN ? (r.ntok + 63) & ~63 : (r.ntok + 31) & ~31;
    return r;
}
template <int KIND>
__global__ void __launch_bounds__(num_threads<KIND>(), 1)
grouped_gemm_bwd_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p) {
    using L = Smem<KIND>;
    constexpr int STAGES = L::STAGES;
    constexpr bool PAIR = L::PAIR;
    constexpr uint32_t B_BYTES = L::B_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *full = bars;                  // [STAGES]
    uint64_t *empty = bars + STAGES;        // [STAGES]
    uint64_t *tfull = bars + 2 * STAGES;    // [2]
    uint64_t *tempty = tfull + 2;           // [2] even CTA (every epilogue warp of both)
    uint64_t *mma_done = tempty + 2;        // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);
    int *eo = reinterpret_cast<int *>(smem + L::tables_off);
    int *mtp = eo + (kMaxExperts + 1);
    int *eo2 = mtp + (kMaxExperts + 1);
    int *pk = eo2 + (kMaxExperts + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // pairs: the CTA's rank in its cluster (0 = even CTA, issues the MMAs) and the pair's
    // index; one CTA per tile: rank 0 and the CTA's index
    const uint32_t cta = PAIR ? cluster_ctarank() : 0u;
    const int pair = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int num_pairs = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    if (warp == 0) {
        if (lane < 6) tma_prefetch_desc(lane == 0 ? &maps.a : &maps.b[lane - 1]);
    } else if (warp == 1) {
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    } else if (warp == 2 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], PAIR ? 16 : 8);   // one arrival per epilogue warp
        }
        mbar_init(mma_done, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dep_wait();
    grid_dep_trigger();
    if (warp == 0) {
        build_tile_tables(p.expert_offsets, 0, p.ne, BN, eo, mtp);
        // dgrad-down: the 64-row blocks of the experts before e, the column of expert e's
        // first row in (w a)^T (eo2 is the same expert-offset table again)
        if (KIND == BWD_DGRAD_DOWN) build_tile_tables(p.expert_offsets, 0, p.ne, 64, eo2, pk);
    }
    fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();   // both CTAs' barriers exist before any cross-CTA signal
    fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // One cluster (or CTA) per tile, persistent over the tiles t = pair + j * num_pairs.
    const int total = mtp[p.ne] * p.m_tiles;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------ TMA producer
            // both CTAs' copies complete on the even CTA's full barrier, which the even
            // CTA arms with the pair's bytes
            const uint32_t full_even0 = PAIR ? mapa_shared(smem_u32(&full[0]), 0) : smem_u32(&full[0]);
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int t = pair; ok && t < total; t += num_pairs) {
                const DTile tl = dtile_at<KIND>(t, mtp, eo, p.ne, p.m_tiles);
                const int a_x = ((PAIR ? 2 : 1) * tl.f + (int)cta) * BM;   // the CTA's 128 M rows
                const int a_y0 = tl.i * p.a_rows_per_expert;
                const int half = PAIR ? tl.nmma >> 1 : tl.nmma;   // token rows this CTA stages
                const int bsel = token_box_index(half);
                const int t_row = tl.tok0 + (int)cta * half;
                const uint32_t tx = (PAIR ? 2u : 1u) * (A_BYTES + (uint32_t)(16 << bsel) * BK * 2);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    if (cta == 0) mbar_arrive_expect_tx(&full[stage], tx);
                    const uint32_t fb = full_even0 + stage * 8;
                    const uint32_t a_dst = smem_u32(smem + L::a_off + stage * A_BYTES);
                    const uint32_t b_dst = smem_u32(smem + L::b_off + stage * B_BYTES);
                    if (PAIR) {
                        tma_load_2d_pair(a_dst, &maps.a, fb, a_x, a_y0 + kb * BK);
                        tma_load_2d_pair(a_dst + MN_BOX, &maps.a, fb, a_x + 64, a_y0 + kb * BK);
                        tma_load_2d_pair(b_dst, &maps.b[bsel], fb, kb * BK, t_row);
                    } else {
                        tma_load_2d(a_dst, &maps.a, fb, a_x, a_y0 + kb * BK);
                        tma_load_2d(a_dst + MN_BOX, &maps.a, fb, a_x + 64, a_y0 + kb * BK);
                        tma_load_2d(b_dst, &maps.b[bsel], fb, kb * BK, t_row);
                    }
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
                        mbar_wait<PAIR>(&full[s], (armed_parity >> s) & 1u, &no_abort, p.status);
                    }
        }
    } else if (warp == 1) {
        if (lane == 0 && cta == 0) {   // ---------------------------- MMA issuer (even CTA)
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = pair; ok && t < total; t += num_pairs) {
                const DTile tl = dtile_at<KIND>(t, mtp, eo, p.ne, p.m_tiles);
                const uint32_t idesc = make_idesc(PAIR ? PM : BM, tl.nmma) | (1u << 15);   // A MN-major
                if (!mbar_wait<PAIR>(&tempty[acc], acc_phase ^ 1u, abort_s, p.status)) break;
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait<PAIR>(&full[stage], phase, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t a_addr = smem_u32(smem + L::a_off + stage * A_BYTES);
                    const uint32_t b_addr = smem_u32(smem + L::b_off + stage * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = smem_desc_mn_sw128(a_addr + kk * 2048, p.lbo, p.sbo);
                        const uint64_t bd = smem_desc_sw128(b_addr + kk * 32);
                        if (PAIR)
                            mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                        else
                            mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                    }
                    if (PAIR)
                        commit_pair(&empty[stage]);
                    else
                        commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (PAIR)
                    commit_pair(&tfull[acc]);
                else
                    commit(&tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA done before TMEM is freed
            if (pair < total) {
                if (PAIR)
                    commit_pair(mma_done);
                else
                    commit(mma_done);
            }
        }
        if (lane == 0 && pair < total) {
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, p.status);
        }
    } else {   // ------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int etid = threadIdx.x - 64;
        const uint32_t tempty_even0 = PAIR ? mapa_shared(smem_u32(&tempty[0]), 0) : 0u;
        float *stage_f = reinterpret_cast<float *>(smem + L::epi_off);
        __nv_bfloat16 *stage_h = reinterpret_cast<__nv_bfloat16 *>(smem + L::epi_off);
        int *pair_s = reinterpret_cast<int *>(smem + L::pairs_off);
        float *wgt_s = reinterpret_cast<float *>(pair_s + BN);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = pair; t < total; t += num_pairs) {
            DTile dt = {};
            dt = dtile_at<KIND>(t, mtp, eo, p.ne, p.m_tiles);
            for (int j = etid; j < dt.nmma; j += 256) {
                const bool tv = j < dt.ntok;
                const int pr = tv ? p.perm[dt.tok0 + j] : -1;
                pair_s[j] = pr;
                wgt_s[j] = tv && p.topk_w != nullptr ? p.topk_w[pr] : 1.f;
            }
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_s, p.status);
            // tcgen05.ld is warp-collective and the epilogue warps share named barriers:
            // they leave together on abort
            if (!epi8_all(ok)) break;
            fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            // this CTA's 128 accumulator rows: M block 2 f + cta of the weight's columns
            const int blk = (PAIR ? 2 : 1) * dt.f + (int)cta;
            const bool blk_live = blk < p.m_blocks;
            {
                // dgrad: half h of the 8 epilogue warps takes the 16-token chunks
                // c = 16h, 16h + 32, ...; each half stages its chunk [16 tokens][128
                // features] in its own half of the staging block
                const int half = (warp - 2) >> 2;
                const int htid = etid - half * 128;   // 0..127 inside the half
                const int f = q * 32 + lane;           // accumulator row = feature of the tile
                float *sf = stage_f + half * (16 * BM);
                __nv_bfloat16 *sh = stage_h + half * (16 * BM);
                for (int c = half * 16; c < dt.nmma; c += 32) {
                    float v[16];
                    tmem_ld16(taddr + c, v);
                    if (c + 32 >= dt.nmma) {   // this warp's last read of the accumulator
                        fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (PAIR)
                                mbar_arrive_cluster_relaxed(tempty_even0 + acc * 8);
                            else
                                mbar_arrive(&tempty[acc]);
                        }
                    }
                    if (KIND == BWD_DGRAD_DOWN) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) sf[j * BM + f] = v[j];
                        half_sync(half);
                        // 16 tokens x 16 groups of 8 features: two items per thread, their
                        // gate / up vectors loaded first so the latencies overlap
                        const __nv_bfloat16 *__restrict__ gu = p.gu;
                        uint4 graw[2], uraw[2], wa_v[2];
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int item = htid + 128 * s2;
                            const int j = item >> 4, f8 = (item & 15) * 8;
                            const int i = blk * BM + f8;
                            graw[s2] = uraw[s2] = make_uint4(0u, 0u, 0u, 0u);
                            if (c + j < dt.ntok && i < p.I) {
                                const size_t r = (size_t)dt.tok0 + c + j;
                                const int gcol = (i / 64) * 128 + (i % 64);
                                graw[s2] = __ldg(reinterpret_cast<const uint4 *>(gu + r * 2 * p.Ipad + gcol));
                                uraw[s2] = __ldg(reinterpret_cast<const uint4 *>(gu + r * 2 * p.Ipad + gcol + 64));
                            }
                        }
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int item = htid + 128 * s2;
                            const int j = item >> 4, f8 = (item & 15) * 8;
                            const int i = blk * BM + f8;              // intermediate feature
                            // (a block past Ipad, the odd half of a last pair tile, has no
                            // outputs)
                            const bool tv = c + j < dt.ntok && blk_live;
                            float part = 0.f;
                            wa_v[s2] = make_uint4(0u, 0u, 0u, 0u);   // zero past the tile's tokens
                            if (tv) {
                                const size_t r = (size_t)dt.tok0 + c + j;
                                const int gcol = (i / 64) * 128 + (i % 64);   // packed column
                                uint4 dg_v = make_uint4(0u, 0u, 0u, 0u), du_v = dg_v;
                                if (i < p.I) {
                                    const float w = wgt_s[c + j];
                                    float g[8], u[8], dg[8], du[8], wa[8];
                                    Vec16<__nv_bfloat16>::to_float(graw[s2], g);
                                    Vec16<__nv_bfloat16>::to_float(uraw[s2], u);
                                    const float4 d0 = *reinterpret_cast<const float4 *>(sf + j * BM + f8);
                                    const float4 d1 = *reinterpret_cast<const float4 *>(sf + j * BM + f8 + 4);
                                    const float da[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                                    for (int x = 0; x < 8; ++x) {
                                        const float sg = __frcp_rn(1.0f + __expf(-g[x]));
                                        const float sl = g[x] * sg;
                                        const float a = sl * u[x];
                                        part += da[x] * a;
                                        const float dw = w * da[x];
                                        dg[x] = dw * u[x] * (sg * (1.0f + g[x] * (1.0f - sg)));
                                        du[x] = dw * sl;
                                        wa[x] = w * a;
                                    }
                                    dg_v = pack8_bf16(dg);
                                    du_v = pack8_bf16(du);
                                    wa_v[s2] = pack8_bf16(wa);
                                }
                                *reinterpret_cast<uint4 *>(p.dgu + r * 2 * p.Ipad + gcol) = dg_v;
                                *reinterpret_cast<uint4 *>(p.dgu + r * 2 * p.Ipad + gcol + 64) = du_v;
                            }
                            // the 16 items of token j are 16 consecutive lanes
#pragma unroll
                            for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                            if (tv && (item & 15) == 0)
                                p.dweight_part[(size_t)blk * p.rows + dt.tok0 + c + j] = part;
                        }
                        half_sync(half);   // the chunk's da values are read
                        // (w a)^T: the chunk [16 tokens][128 features] through this half's
                        // staging block, then 16 bytes (8 tokens) of a feature row per item,
                        // the two items of a feature in adjacent lanes
                        __nv_bfloat16 *swa = reinterpret_cast<__nv_bfloat16 *>(sf);
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int item = htid + 128 * s2;
                            *reinterpret_cast<uint4 *>(swa + (item >> 4) * BM + (item & 15) * 8) = wa_v[s2];
                        }
                        half_sync(half);
                        // the tile's first column: its first row's place in the expert's block
                        const int64_t colT = 64LL * pk[dt.i] + (dt.tok0 - eo[dt.i]) + c;
#pragma unroll
                        for (int s2 = 0; s2 < 2 && blk_live; ++s2) {
                            const int item = htid + 128 * s2;
                            const int ff = item >> 1, jg = (item & 1) * 8;
                            __align__(16) __nv_bfloat16 o[8];
#pragma unroll
                            for (int x = 0; x < 8; ++x) o[x] = swa[(jg + x) * BM + ff];
                            *reinterpret_cast<uint4 *>(p.waT + (size_t)(blk * BM + ff) * p.ldt + colT + jg) =
                                *reinterpret_cast<const uint4 *>(o);
                        }
                        half_sync(half);
                    } else {   // BWD_DGRAD_GU: dx of the pair, unweighted, into its slot
#pragma unroll
                        for (int j = 0; j < 16; ++j) sh[j * BM + f] = __float2bfloat16_rn(v[j]);
                        half_sync(half);
                        const int col0 = blk * BM;   // past H for a block with no outputs
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int item = htid + 128 * s2;
                            const int j = item >> 4, f8 = (item & 15) * 8;
                            const int prj = c + j < dt.ntok ? pair_s[c + j] : -1;
                            if (prj >= 0 && col0 + f8 < p.H)
                                *reinterpret_cast<uint4 *>(p.dx_slots + (size_t)prj * p.H + col0 + f8) =
                                    *reinterpret_cast<const uint4 *>(sh + j * BM + f8);
                        }
                        half_sync(half);
                    }
                }
                epi8_sync();   // both halves are done with this tile's pair ids and weights
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();   // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
    }
}

template <int KIND>
cudaError_t launch_bwd(const BwdMaps &maps, BwdParams prm, int64_t max_tiles, cudaStream_t s) {
    if (max_tiles <= 0) return cudaSuccess;
    // MN-major descriptor strides: 64-element groups are one 8 KB box apart, 8-row K
    // groups one 1024-byte swizzle atom apart
    prm.lbo = MN_BOX;
    prm.sbo = 1024;
    auto kern = grouped_gemm_bwd_kernel<KIND>;
    constexpr bool PAIR = Smem<KIND>::PAIR;
    // per device: the clusters of two (or CTAs) that fit at once, one CTA per SM, set up once
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
                                     (int)Smem<KIND>::alloc);
            if (e != cudaSuccess) return e;
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(2, 1, 1);
            cfg.blockDim = dim3(num_threads<KIND>(), 1, 1);
            cfg.dynamicSmemBytes = Smem<KIND>::alloc;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (PAIR) {
                e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            } else {
                e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            }
            if (e != cudaSuccess) return e;
            if (n < 1) return cudaErrorInvalidConfiguration;
            clusters_dev[dev] = n;
        }
        max_clusters = clusters_dev[dev];
    }
    const int clusters = (int)std::min<int64_t>(max_tiles, max_clusters);
    if (!PAIR)
        return launch_pdl(kern, dim3(clusters), dim3(num_threads<KIND>()), Smem<KIND>::alloc, s,
                          maps, prm);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(num_threads<KIND>(), 1, 1);
    cfg.dynamicSmemBytes = Smem<KIND>::alloc;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps, prm);
}

cudaError_t token_maps(BwdMaps *m, const void *t, uint64_t rows, uint64_t cols, uint64_t ld) {
    cudaError_t e = cudaSuccess;
    for (int b = 0; b < 5 && e == cudaSuccess; ++b) e = make_map(&m->b[b], t, rows, cols, ld, 16u << b);
    return e;
}

}  // namespace

cudaError_t launch_tc_dgrad_down(const LayerDims &d, const void *dout_send, const int32_t *eoff,
                                 const void *w_down, const void *gu, const int32_t *perm,
                                 const float *topk_w, void *dgu, void *waT, float *dweight_part,
                                 int32_t *status, cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    BwdMaps maps;
    // A = W_d [E*H rows (K = h), I columns (M = i)]
    cudaError_t e = make_map(&maps.a, w_down, (uint64_t)d.E * d.H, d.I, d.I, 64);
    if (e == cudaSuccess) e = token_maps(&maps, dout_send, rows, d.H, d.H);
    if (e != cudaSuccess) return e;
    BwdParams prm = {};
    prm.expert_offsets = eoff;
    prm.ne = d.E;
    prm.num_kb = ceil_div(d.H, BK);
    prm.m_blocks = d.Ipad / BM;
    prm.m_tiles = prm.m_blocks;   // one CTA per tile
    prm.a_rows_per_expert = d.H;
    prm.I = d.I;
    prm.Ipad = d.Ipad;
    prm.H = d.H;
    prm.gu = (const __nv_bfloat16 *)gu;
    prm.dgu = (__nv_bfloat16 *)dgu;
    prm.waT = (__nv_bfloat16 *)waT;
    prm.ldt = wgrad_t_cols(d);
    prm.dweight_part = dweight_part;
    prm.rows = (int)rows;
    prm.perm = perm;
    prm.topk_w = topk_w;
    prm.status = status;
    return launch_bwd<BWD_DGRAD_DOWN>(maps, prm, (ceil_div64(rows, BN) + d.E) * prm.m_tiles, s);
}

cudaError_t launch_tc_dgrad_gate_up(const LayerDims &d, const void *dgu, const int32_t *eoff,
                                    const void *packed, const int32_t *perm, void *dx_slots,
                                    int32_t *status, cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    BwdMaps maps;
    // A = packed W_gu [E*2Ipad rows (K = f), H columns (M = h)]
    cudaError_t e = make_map(&maps.a, packed, (uint64_t)d.E * 2 * d.Ipad, d.H, d.H, 64);
    if (e == cudaSuccess) e = token_maps(&maps, dgu, rows, 2 * d.Ipad, 2 * d.Ipad);
    if (e != cudaSuccess) return e;
    BwdParams prm = {};
    prm.expert_offsets = eoff;
    prm.ne = d.E;
    prm.num_kb = 2 * d.Ipad / BK;
    prm.m_blocks = ceil_div(d.H, BM);
    prm.m_tiles = ceil_div(prm.m_blocks, 2);
    prm.a_rows_per_expert = 2 * d.Ipad;
    prm.I = d.I;
    prm.Ipad = d.Ipad;
    prm.H = d.H;
    prm.rows = (int)rows;
    prm.perm = perm;
    prm.topk_w = nullptr;
    prm.dx_slots = (__nv_bfloat16 *)dx_slots;
    prm.status = status;
    return launch_bwd<BWD_DGRAD_GU>(maps, prm, (ceil_div64(rows, BN) + d.E) * prm.m_tiles, s);
}

}  // namespace moe
