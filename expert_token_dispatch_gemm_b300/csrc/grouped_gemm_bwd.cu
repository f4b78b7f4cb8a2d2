// Backward of the local experts as grouped GEMMs on the tensor cores. The chain rule
// through y = W_d (silu(g) * u), g = W_g x, u = W_u x of every kept (token, expert) pair
// (Ultralytics glossary "Expert Parallelism", step 3; an expert's weight gradient sums
// over every row it received -- Hugging Face "Expert parallelism" docs, "How the sizes
// combine"). Per send row r (pair of token t, weight w) with upstream gradient dout_t:
//   dgrad_down : da_u[i, r] = sum_h W_d[h, i] dout_t[h]       (tokens on N, K = H)
//                epilogue: a = silu(g) u, dweight_r += da_u . a (the routing weight's
//                gradient), dg = w da_u u silu'(g), du = w da_u silu(g), wa = w a
//   dgrad_gu   : dx_r[h] = sum_f W_gu[f, h] dgu_r[f]           (tokens on N, K = 2 Ipad)
//   wgrad      : dW_gu[f, h] = sum_r dgu_r[f] x_r[h]           (K = the expert's rows)
//                dW_d[h, i]  = sum_r dout_t[h] wa_r[i]
// The weights stay in their forward layouts: the dgrad GEMMs read them as MN-major A
// operands (M = the weight's column index), and the weight-gradient GEMMs read both
// token-major activations as MN-major operands (K = token rows), so nothing is
// transposed in memory.
//
// One CTA per SM (192 threads, persistent over its tiles), tcgen05.mma cta_group::1,
// M = 128 TMEM lanes, N <= 256:
//   warp 0      TMA producer, 4-stage ring (A: 128 x 64, B: up to 256 x 64; 128-byte
//               swizzle). MN-major tiles are 64-element boxes: one 128-byte row per K.
//   warp 1      TMEM (two 128 x 256 fp32 accumulators); lane 0 issues the MMAs. In the
//               weight-gradient GEMMs the warp first zeroes the rows of the last K block
//               that lie past the expert's segment, in both operands (they hold another
//               expert's rows, or unwritten memory past the kept rows).
//   warps 2..9  epilogue, two warps per TMEM lane quarter: in the weight-gradient GEMMs
//               each takes 128 of the tile's 256 columns (one TMEM load, two 64-column
//               TMA stores); in the dgrad GEMMs alternate 16-token chunks, each half
//               with its own named barrier.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel records
// MOE_DEV_TIMEOUT in the status word, stops issuing work, waits (bounded) for its own
// copies and MMAs, frees TMEM and returns.
#include <mutex>

#include "sm100.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;                 // M rows per tile (TMEM lanes)
constexpr int BN = 256;                 // max N per tile
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t MN_BOX = 64 * BK * 2;    // one 64-element x 64-row MN-major box: 8 KB
// Threads: producer warp, MMA warp and 8 epilogue warps (two per TMEM lane quarter).
template <int KIND> constexpr int num_threads() { return 320; }
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int CHUNK = 32;

enum { BWD_DGRAD_DOWN = 0, BWD_DGRAD_GU = 1, BWD_WGRAD = 2 };

// Shared-memory descriptor of an MN-major tile written by TMA in 64-element boxes with
// 128-byte swizzle: one 128-byte row per K index, 8-row groups 1024 bytes apart (stride
// byte offset), 64-element groups along M / N `lbo` bytes apart (leading byte offset).
// Advancing K by 16 adds 16 rows = 2048 bytes to the start address.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Token maps with box heights 32, 64, 128 and 256 rows (K-major B of the dgrad GEMMs).
struct BwdMaps {
    CUtensorMap a;       // MN-major A: box 64 x 64
    CUtensorMap b[4];    // dgrad: token rows (K-major); wgrad: b[0] MN-major box 64 x 64
    CUtensorMap out[2];  // wgrad: [E][rows][cols] outputs, box 64 x 32 (TMA stores)
};
__host__ __device__ constexpr int box_index(int rows) {
    return rows <= 32 ? 0 : rows <= 64 ? 1 : rows <= 128 ? 2 : 3;
}

struct BwdParams {
    const int32_t *expert_offsets;
    int ne;                  // experts (all of the layer)
    int num_kb;              // dgrad: K blocks of BK
    int m_tiles, n_tiles;    // M tiles of BM; wgrad: N tiles of BN
    int a_rows_per_expert;   // dgrad: rows between experts in A's map (K rows)
    uint32_t lbo, sbo;       // MN-major descriptor strides
    int I, Ipad, H;
    // dgrad_down
    const __nv_bfloat16 *gu;      // [rows, 2 Ipad] saved gate / up pre-activations
    __nv_bfloat16 *dgu;           // [rows, 2 Ipad] out
    __nv_bfloat16 *wa;            // [rows, Ipad] out: w * silu(g) * u
    float *dweight_part;          // [m_tiles, rows] out
    int rows;                     // send rows of the buffers (N * k)
    // dgrad_down / dgrad_gu
    const int32_t *perm;
    const float *topk_w;
    __nv_bfloat16 *dx_slots;      // dgrad_gu: [N*k, H] out (row = pair id)
    int wgrad_gu;                 // wgrad: 1 = M is packed gate/up rows (outputs dW_gate,
                                  // dW_up), 0 = M is down rows (output dW_down)
    int32_t *status;
};

// 4-stage ring. The dgrad GEMMs add a 16 KB staging block, the token tile's pair ids and
// weights and two tile tables; the weight-gradient GEMMs 32 KB of TMA-store staging (8
// warps x one 4 KB buffer) and the expert offsets only.
template <int KIND>
struct Smem {
    static constexpr bool WG = KIND == BWD_WGRAD;
    static constexpr int STAGES = 4;
    static constexpr uint32_t a_off = 0;
    static constexpr uint32_t b_off = STAGES * A_BYTES;
    static constexpr uint32_t epi_off = b_off + STAGES * B_BYTES;
    static constexpr uint32_t epi_bytes = WG ? 8 * 4096 : CHUNK * BM * 4;
    static constexpr uint32_t pairs_off = epi_off + epi_bytes;       // [BN] int + [BN] float
    static constexpr uint32_t bar_off = pairs_off + (WG ? 0 : 2 * BN * 4);
    static constexpr uint32_t misc_off = bar_off + 24 * 8;
    static constexpr uint32_t tables_off = misc_off + 16;
    static constexpr uint32_t end = tables_off + (WG ? 1 : 2) * (kMaxExperts + 1) * 4;
    static constexpr uint32_t alloc = end + 1024;
};
static_assert(Smem<BWD_WGRAD>::alloc <= 227 * 1024 && Smem<BWD_DGRAD_DOWN>::alloc <= 227 * 1024,
              "shared memory per CTA");

// Tile of a dgrad GEMM: expert i, M tile f, token tile m; tokens fastest.
struct DTile {
    int i, f, m, tok0, ntok, nmma;
};
__device__ __forceinline__ DTile dtile_at(int t, const int *mtp, const int *eo, int ne, int m_tiles) {
    DTile r;
    decode_tile(t, mtp, ne, m_tiles, r.i, r.m, r.f);
    const int seg = eo[r.i + 1] - eo[r.i];
    r.tok0 = eo[r.i] + r.m * BN;
    r.ntok = min(BN, seg - r.m * BN);
    r.nmma = (r.ntok + 31) & ~31;
    return r;
}
// Tile of a weight-gradient GEMM: expert e, M tile mt, N tile nt; K = the expert's rows.
struct WTile {
    int e, mt, nt, row0, nrows, nkb;
};
__device__ __forceinline__ WTile wtile_at(int t, const int *eo, int m_tiles, int n_tiles) {
    WTile r;
    const int per = m_tiles * n_tiles;
    r.e = t / per;
    const int l = t - r.e * per;
    r.mt = l / n_tiles;          // N fastest: concurrent tiles share the A rows in L2
    r.nt = l - r.mt * n_tiles;
    r.row0 = eo[r.e];
    r.nrows = eo[r.e + 1] - r.row0;
    r.nkb = (r.nrows + BK - 1) / BK;
    return r;
}

// 128 consecutive fp32 accumulator columns of this thread's TMEM lane (one load, one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float *v) {
    uint32_t r[128];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barriers of the 8 dgrad epilogue warps: id 1 + half for one half (128 threads),
// id 3 for all 256 (also a vote: returns whether `ok` holds in every thread).
__device__ __forceinline__ void half_sync(int half) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + half) : "memory");
}
__device__ __forceinline__ void epi8_sync() { asm volatile("bar.sync 3, 256;" ::: "memory"); }
__device__ __forceinline__ bool epi8_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 3, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

template <int KIND>
__global__ void __launch_bounds__(num_threads<KIND>(), 1)
grouped_gemm_bwd_kernel(const __grid_constant__ BwdMaps maps, const BwdParams p) {
    constexpr bool WG = KIND == BWD_WGRAD;
    using L = Smem<KIND>;
    constexpr int STAGES = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *full = bars;                  // [STAGES]
    uint64_t *empty = bars + STAGES;        // [STAGES]
    uint64_t *tfull = bars + 2 * STAGES;    // [2]
    uint64_t *tempty = tfull + 2;           // [2] (4 epilogue warps)
    uint64_t *mma_done = tempty + 2;        // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);
    int *eo = reinterpret_cast<int *>(smem + L::tables_off);
    int *mtp = eo + (kMaxExperts + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0) {
        if (lane < 5) tma_prefetch_desc(lane == 0 ? &maps.a : &maps.b[lane - 1]);
    } else if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else if (warp == 2 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);   // one arrival per epilogue warp
        }
        mbar_init(mma_done, 1);
        *abort_s = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dep_wait();
    grid_dep_trigger();
    if (warp == 0) {
        if (WG) {
            for (int e = lane; e <= p.ne; e += 32) eo[e] = p.expert_offsets[e];
        } else {
            build_tile_tables(p.expert_offsets, 0, p.ne, BN, eo, mtp);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // One CTA per tile, persistent over the tiles t = blockIdx.x + j * gridDim.x.
    const int tile0 = (int)blockIdx.x;
    const int tstride = (int)gridDim.x;
    const int total = WG ? p.ne * p.m_tiles * p.n_tiles : mtp[p.ne] * p.m_tiles;
    auto wtile = [&](int t) { return wtile_at(t, eo, p.m_tiles, p.n_tiles); };

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            bool ok = true;
            for (int t = tile0; ok && t < total; t += tstride) {
                int nkb, a_x, a_y0, b_x, b_y0, bsel;
                uint32_t tx;
                if (WG) {
                    const WTile tl = wtile(t);
                    nkb = tl.nkb;
                    a_x = tl.mt * BM;
                    b_x = tl.nt * BN;
                    a_y0 = b_y0 = tl.row0;
                    bsel = 0;
                    tx = A_BYTES + B_BYTES;
                } else {
                    const DTile tl = dtile_at(t, mtp, eo, p.ne, p.m_tiles);
                    nkb = p.num_kb;
                    a_x = tl.f * BM;
                    a_y0 = tl.i * p.a_rows_per_expert;
                    b_y0 = tl.tok0;
                    bsel = box_index(tl.nmma);
                    b_x = 0;
                    tx = A_BYTES + (uint32_t)(32 << bsel) * BK * 2;
                }
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_s, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], tx);
                    const uint32_t fb = smem_u32(&full[stage]);
                    const uint32_t a_dst = smem_u32(smem + L::a_off + stage * A_BYTES);
                    const uint32_t b_dst = smem_u32(smem + L::b_off + stage * B_BYTES);
                    tma_load_2d(a_dst, &maps.a, fb, a_x, a_y0 + kb * BK);
                    tma_load_2d(a_dst + MN_BOX, &maps.a, fb, a_x + 64, a_y0 + kb * BK);
                    if (WG) {   // the B tile: four 64-column MN-major boxes
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            tma_load_2d(b_dst + q * MN_BOX, &maps.b[0], fb, b_x + 64 * q,
                                        b_y0 + kb * BK);
                    } else {
                        tma_load_2d(b_dst, &maps.b[bsel], fb, kb * BK, b_y0);
                    }
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if ((armed >> s) & 1u) {
                    volatile int no_abort = 0;
                    mbar_wait(&full[s], (armed_parity >> s) & 1u, &no_abort, p.status);
                }
        }
    } else if (warp == 1) {   // ------------------------------------- MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        const uint32_t idesc_mn = (1u << 15) | (WG ? (1u << 16) : 0u);
        for (int t = tile0; ok && t < total; t += tstride) {
            int nkb, nmma, tail;
            if (WG) {
                const WTile tl = wtile(t);
                nkb = tl.nkb;
                nmma = BN;
                tail = tl.nrows - (tl.nkb - 1) * BK;   // valid rows of the last K block
            } else {
                const DTile tl = dtile_at(t, mtp, eo, p.ne, p.m_tiles);
                nkb = p.num_kb;
                nmma = tl.nmma;
                tail = BK;
            }
            const uint32_t idesc = make_idesc(BM, nmma) | idesc_mn;
            if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_s, p.status))) break;
            fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < nkb; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, abort_s, p.status))) {
                    ok = false;
                    break;
                }
                uint8_t *a_tile = smem + L::a_off + stage * A_BYTES;
                uint8_t *b_tile = smem + L::b_off + stage * B_BYTES;
                // the last K block of a weight-gradient tile: only its 16-row slices
                // that hold rows of the segment are multiplied, and the rows past the
                // segment inside the last of them read as zero (both operands)
                int kslices = BK / 16;
                if (WG && kb == nkb - 1 && tail < BK) {
                    kslices = (tail + 15) / 16;
                    const int zr = kslices * 16 - tail;
                    if (zr > 0) {
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                        for (int c = lane; c < 6 * zr * 8; c += 32) {
                            const int box = c / (zr * 8), rem = c - box * zr * 8;
                            const int row = tail + rem / 8, ch = rem % 8;
                            uint8_t *base = box < 2 ? a_tile + box * MN_BOX : b_tile + (box - 2) * MN_BOX;
                            *reinterpret_cast<uint4 *>(base + row * 128 + ch * 16) = z;
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    fence_after();
                    const uint32_t a_addr = smem_u32(a_tile);
                    const uint32_t b_addr = smem_u32(b_tile);
                    for (int kk = 0; kk < kslices; ++kk) {
                        const uint64_t ad = smem_desc_mn_sw128(a_addr + kk * 2048, p.lbo, p.sbo);
                        const uint64_t bd = WG ? smem_desc_mn_sw128(b_addr + kk * 2048, p.lbo, p.sbo)
                                               : smem_desc_sw128(b_addr + kk * 32);
                        mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                    }
                    commit(&empty[stage]);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (lane == 0) commit(&tfull[acc]);   // after no K block: arrives at once
            __syncwarp();
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) {
            commit(mma_done);   // every MMA done before TMEM is freed
            volatile int no_abort = 0;
            mbar_wait(mma_done, 0, &no_abort, p.status);
        }
    } else {   // ------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int etid = threadIdx.x - 64;
        float *stage_f = reinterpret_cast<float *>(smem + L::epi_off);
        __nv_bfloat16 *stage_h = reinterpret_cast<__nv_bfloat16 *>(smem + L::epi_off);
        int *pair_s = reinterpret_cast<int *>(smem + L::pairs_off);
        float *wgt_s = reinterpret_cast<float *>(pair_s + BN);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = tile0; t < total; t += tstride) {
            DTile dt = {};
            WTile wt = {};
            if (WG) {
                wt = wtile(t);
            } else {
                dt = dtile_at(t, mtp, eo, p.ne, p.m_tiles);
                for (int j = etid; j < dt.nmma; j += 256) {
                    const bool tv = j < dt.ntok;
                    const int pr = tv ? p.perm[dt.tok0 + j] : -1;
                    pair_s[j] = pr;
                    wgt_s[j] = tv && p.topk_w != nullptr ? p.topk_w[pr] : 1.f;
                }
            }
            const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_s, p.status);
            // tcgen05.ld is warp-collective and the epilogue warps share named barriers:
            // they leave together on abort
            if (!epi8_all(ok)) break;
            fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            if (WG) {
                // The warp's 32 accumulator rows are 32 consecutive rows of one output;
                // half h of the 8 epilogue warps takes accumulator columns 128 h ..
                // 128 h + 127 in one TMEM load and stores them as two 64-column chunks,
                // each through the warp's 128-byte-swizzled staging block [32 rows][128
                // bytes] into a TMA store (rows past I / H and columns past the output's
                // width are clipped by the 3-D map).
                const int half = (warp - 2) >> 2;
                const int m0 = wt.mt * BM + q * 32;
                int sel = 0, r0 = m0, ncols = p.I;
                if (p.wgrad_gu) {
                    sel = q >= 2 ? 1 : 0;                  // gate rows, then up rows
                    r0 = wt.mt * 64 + (q & 1) * 32;
                    ncols = p.H;
                }
                const bool live = r0 < (p.wgrad_gu ? p.I : p.H);
                uint8_t *buf = smem + L::epi_off + (warp - 2) * 4096;
                const int c2 = 128 * half;
                const bool cols_live = wt.nt * BN + c2 < ncols;   // uniform over the warp
                float v[128];
                if (cols_live) {
                    if (wt.nkb > 0) {
                        tmem_ld128(taddr + c2, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 128; ++j) v[j] = 0.f;   // an expert with no rows
                    }
                }
                // the warp's accumulator columns are read: hand them back
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
                if (live && cols_live) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col0 = wt.nt * BN + c2 + 64 * h;
                        if (col0 >= ncols) break;
                        // the store that last read the staging block is done
                        if (lane == 0) tma_store_wait_read();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4 *>(buf + lane * 128 + ((j ^ (lane & 7)) * 16)) =
                                pack8_bf16(v + 64 * h + 8 * j);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) tma_store_3d(&maps.out[sel], smem_u32(buf), col0, r0, wt.e);
                    }
                }
            } else {
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
                        if (lane == 0) mbar_arrive(&tempty[acc]);
                    }
                    if (KIND == BWD_DGRAD_DOWN) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) sf[j * BM + f] = v[j];
                        half_sync(half);
                        // 16 tokens x 16 groups of 8 features: two items per thread, their
                        // gate / up vectors loaded first so the latencies overlap
                        const __nv_bfloat16 *__restrict__ gu = p.gu;
                        uint4 graw[2], uraw[2];
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            const int item = htid + 128 * s2;
                            const int j = item >> 4, f8 = (item & 15) * 8;
                            const int i = dt.f * BM + f8;
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
                            const int i = dt.f * BM + f8;             // intermediate feature
                            const bool tv = c + j < dt.ntok;
                            float part = 0.f;
                            if (tv) {
                                const size_t r = (size_t)dt.tok0 + c + j;
                                const int gcol = (i / 64) * 128 + (i % 64);   // packed column
                                uint4 dg_v = make_uint4(0u, 0u, 0u, 0u), du_v = dg_v, wa_v = dg_v;
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
                                    wa_v = pack8_bf16(wa);
                                }
                                *reinterpret_cast<uint4 *>(p.dgu + r * 2 * p.Ipad + gcol) = dg_v;
                                *reinterpret_cast<uint4 *>(p.dgu + r * 2 * p.Ipad + gcol + 64) = du_v;
                                *reinterpret_cast<uint4 *>(p.wa + r * p.Ipad + i) = wa_v;
                            }
                            // the 16 items of token j are 16 consecutive lanes
#pragma unroll
                            for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                            if (tv && (item & 15) == 0)
                                p.dweight_part[(size_t)dt.f * p.rows + dt.tok0 + c + j] = part;
                        }
                        half_sync(half);
                    } else {   // BWD_DGRAD_GU: dx of the pair, unweighted, into its slot
#pragma unroll
                        for (int j = 0; j < 16; ++j) sh[j * BM + f] = __float2bfloat16_rn(v[j]);
                        half_sync(half);
                        const int col0 = dt.f * BM;
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

    if (WG && warp >= 2 && lane == 0) tma_store_wait_all();   // stores done, staging free
    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
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
    // per device: the SM count (one persistent CTA per SM), set up once
    static std::mutex mu;
    static int sms_dev[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (sms_dev[dev] == 0) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)Smem<KIND>::alloc);
            if (e != cudaSuccess) return e;
            int n = 0;
            e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            sms_dev[dev] = n > 0 ? n : 148;
        }
        sms = sms_dev[dev];
    }
    const int grid = (int)std::min<int64_t>(max_tiles, sms);
    return launch_pdl(kern, dim3(grid), dim3(num_threads<KIND>()), Smem<KIND>::alloc, s, maps, prm);
}

cudaError_t token_maps(BwdMaps *m, const void *t, uint64_t rows, uint64_t cols, uint64_t ld) {
    cudaError_t e = cudaSuccess;
    for (int b = 0; b < 4 && e == cudaSuccess; ++b) e = make_map(&m->b[b], t, rows, cols, ld, 32u << b);
    return e;
}

}  // namespace

cudaError_t launch_tc_dgrad_down(const LayerDims &d, const void *dout_send, const int32_t *eoff,
                                 const void *w_down, const void *gu, const int32_t *perm,
                                 const float *topk_w, void *dgu, void *wa, float *dweight_part,
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
    prm.m_tiles = d.Ipad / BM;
    prm.a_rows_per_expert = d.H;
    prm.I = d.I;
    prm.Ipad = d.Ipad;
    prm.H = d.H;
    prm.gu = (const __nv_bfloat16 *)gu;
    prm.dgu = (__nv_bfloat16 *)dgu;
    prm.wa = (__nv_bfloat16 *)wa;
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
    prm.m_tiles = ceil_div(d.H, BM);
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

cudaError_t launch_tc_wgrad_gate_up(const LayerDims &d, const void *dgu, const void *send,
                                    const int32_t *eoff, void *dw_gate, void *dw_up,
                                    int32_t *status, cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    BwdMaps maps = {};
    cudaError_t e = make_map(&maps.a, dgu, rows, 2 * d.Ipad, 2 * d.Ipad, 64);
    if (e == cudaSuccess) e = make_map(&maps.b[0], send, rows, d.H, d.H, 64);
    for (int b = 1; b < 4 && e == cudaSuccess; ++b) maps.b[b] = maps.b[0];
    if (e == cudaSuccess) e = make_store_map_3d(&maps.out[0], dw_gate, d.H, d.I, d.E, 64, 32);
    if (e == cudaSuccess) e = make_store_map_3d(&maps.out[1], dw_up, d.H, d.I, d.E, 64, 32);
    if (e != cudaSuccess) return e;
    BwdParams prm = {};
    prm.expert_offsets = eoff;
    prm.ne = d.E;
    prm.m_tiles = 2 * d.Ipad / BM;
    prm.n_tiles = ceil_div(d.H, BN);
    prm.I = d.I;
    prm.Ipad = d.Ipad;
    prm.H = d.H;
    prm.rows = (int)rows;
    prm.wgrad_gu = 1;
    prm.status = status;
    return launch_bwd<BWD_WGRAD>(maps, prm, (int64_t)d.E * prm.m_tiles * prm.n_tiles, s);
}

cudaError_t launch_tc_wgrad_down(const LayerDims &d, const void *dout_send, const void *wa,
                                 const int32_t *eoff, void *dw_down, int32_t *status,
                                 cudaStream_t s) {
    const int64_t rows = (int64_t)d.N * d.k;
    BwdMaps maps = {};
    cudaError_t e = make_map(&maps.a, dout_send, rows, d.H, d.H, 64);
    if (e == cudaSuccess) e = make_map(&maps.b[0], wa, rows, d.Ipad, d.Ipad, 64);
    for (int b = 1; b < 4 && e == cudaSuccess; ++b) maps.b[b] = maps.b[0];
    if (e == cudaSuccess) e = make_store_map_3d(&maps.out[0], dw_down, d.I, d.H, d.E, 64, 32);
    if (e == cudaSuccess) maps.out[1] = maps.out[0];
    if (e != cudaSuccess) return e;
    BwdParams prm = {};
    prm.expert_offsets = eoff;
    prm.ne = d.E;
    prm.m_tiles = ceil_div(d.H, BM);
    prm.n_tiles = ceil_div(d.I, BN);
    prm.I = d.I;
    prm.Ipad = d.Ipad;
    prm.H = d.H;
    prm.rows = (int)rows;
    prm.wgrad_gu = 0;
    prm.status = status;
    return launch_bwd<BWD_WGRAD>(maps, prm, (int64_t)d.E * prm.m_tiles * prm.n_tiles, s);
}

}  // namespace moe
