// Step 1 on the tensor cores -- routing for bf16 layers (Ultralytics glossary "Expert
// Parallelism", section "How tokens move between GPUs", step 1 and its routing example):
// logits = x W_r^T (+ b) accumulate in TMEM, M = 128 tokens by N = E rounded up to 16;
// each epilogue thread owns one token's logits, keeps its top-k in registers (ties to
// the lower expert id), applies the softmax over the k chosen logits and adds the
// token's experts to the per-segment histogram that the dispatch scan consumes.
//
// One CTA per 128-token tile, or (KSPLIT = 2, when there are fewer tiles than SMs) a
// cluster of two CTAs per tile that split the hidden dimension: CTA r accumulates the
// partial logits of K blocks [r * ceil(kb/2), ...) for all 128 tokens, keeps the 64
// tokens of histogram segment 2 * tile + r and sends its partials of the other 64 rows to
// the peer's shared memory (st.shared::cluster, then a release arrive on the peer's
// mbarrier). Each CTA adds own + received partials (fp32 addition commutes, so both see
// the same sums) and finishes the top-k of its 64 tokens. Twice the SMs stream x.
// The top-k runs over column slices: with SLICES groups of four epilogue warps, group g
// selects each token's top-k among its slice of the experts and group 0 merges the other
// groups' lists in expert order, which keeps the ordering (value descending, ties to the
// lower id).
//
// Per CTA (64 + 128 * SLICES threads, one tile):
//   warp 0      TMA producer: 128x64 x tile + round16(E) x 64 router tile per stage,
//               128-byte swizzle, a ring of 2..8 stages (as many as the shared memory
//               left to the CTA holds: the copies in flight per SM set the streaming
//               rate) guarded by full/empty mbarriers;
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
#include <algorithm>
#include <mutex>

#include "sm100.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = kTcBlockM;   // 128 tokens per tile
constexpr int MAX_STAGES = 8;
constexpr uint32_t A_BYTES = BM * BK * 2;
static_assert(BM == 2 * kSegTokens, "a route tile covers two histogram segments");

// Routing variants (template MODE): 0 plain top-k of the logits; 1 selection on
// logits + selection bias, weights from the logits; 2 as 1 within the group_limit best
// partitions (one column slice, two passes over the accumulator).
enum { ROUTE_PLAIN = 0, ROUTE_SELBIAS = 1, ROUTE_GROUP = 2 };

struct RouteParams {
    int rows;                // tokens
    int bn;                  // MMA N (E rounded up to 16)
    int stages;              // ring depth, 2..MAX_STAGES
    int kb_half;             // KSPLIT = 2: K blocks of CTA 0 (CTA 1 takes the rest)
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

// Shared-memory layout for a given MMA N and ring depth.
// KSPLIT = 2 adds the receive buffer of the peer's partial logits, [bn / 4][64 rows][4]
// fp32 (a warp's 32 rows of 4 columns are 512 contiguous bytes), and its mbarrier.
struct RouteSmem {
    uint32_t b_off, recv_off, bar_off, misc_off, bias_off, sbias_off, hist_off, alloc;
};
__host__ __device__ inline RouteSmem route_smem(int bn, int E, int stages, int ksplit) {
    RouteSmem m;
    m.b_off = (uint32_t)stages * A_BYTES;
    m.recv_off = m.b_off + (uint32_t)stages * (uint32_t)bn * BK * 2;
    m.bar_off = m.recv_off + (ksplit == 2 ? 64u * (uint32_t)bn * 4u : 0u);
    m.misc_off = m.bar_off + (2 * MAX_STAGES + 2) * 8;
    m.bias_off = m.misc_off + 16;
    m.sbias_off = m.bias_off + (uint32_t)(E + 3) / 4 * 16;
    m.hist_off = m.sbias_off + (uint32_t)(E + 3) / 4 * 16;
    m.alloc = m.hist_off + 2 * (uint32_t)E * 4 + 1024;   // + slack to align the base
    return m;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
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

// Plain routing ranks candidates by (logit desc, expert id asc) through order-preserving
// 32-bit keys: a NaN ranks as -inf, -0 as +0, and every real key is above 0, the key of
// an empty candidate. A top-k is then k rounds of: the largest key (a max tree), the
// lowest id among the candidates holding it (a min tree), that candidate cleared -- a
// depth of log2(N) per round instead of one long chain of list insertions.
__device__ __forceinline__ uint32_t rank_key(float v) {
    if (isnan(v)) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
template <int N>
__device__ __forceinline__ uint32_t tree_max_u32(const uint32_t (&a)[N]) {
    static_assert((N & (N - 1)) == 0, "power of two");
    uint32_t t[N];
#pragma unroll
    for (int j = 0; j < N; ++j) t[j] = a[j];
#pragma unroll
    for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) t[j] = max(t[j], t[j + w]);
    return t[0];
}
template <int N>
__device__ __forceinline__ int tree_min_i32(const int (&a)[N]) {
    int t[N];
#pragma unroll
    for (int j = 0; j < N; ++j) t[j] = a[j];
#pragma unroll
    for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) t[j] = min(t[j], t[j + w]);
    return t[0];
}
// The KMAX best of N (key, id) candidates, in ranking order, into (ok, oi); the
// candidates' keys are consumed. An entry with key 0 is empty (id -1).
template <int N, int KMAX>
__device__ __forceinline__ void top_by_key(uint32_t (&o)[N], const int (&id)[N], uint32_t (&ok)[KMAX],
                                           int (&oi)[KMAX]) {
#pragma unroll
    for (int t = 0; t < KMAX; ++t) {
        const uint32_t m = tree_max_u32<N>(o);
        int c[N];
#pragma unroll
        for (int j = 0; j < N; ++j) c[j] = (o[j] == m) ? id[j] : 0x7fffffff;
        const int bi = tree_min_i32<N>(c);
#pragma unroll
        for (int j = 0; j < N; ++j) o[j] = (id[j] == bi) ? 0u : o[j];
        ok[t] = m;
        oi[t] = m != 0u ? bi : -1;
    }
}

// SLICES = 2 runs two CTAs per SM: at most 102 registers per thread
template <int KMAX, int SLICES, int MODE, int KSPLIT>
__global__ void __launch_bounds__(64 + 128 * SLICES, SLICES == 2 ? 2 : 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w, const RouteParams p) {
    constexpr int NT = 128 * SLICES;   // epilogue threads
    static_assert(KSPLIT == 1 || (KSPLIT == 2 && MODE != ROUTE_GROUP), "split routing modes");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const RouteSmem L = route_smem(p.bn, p.E, p.stages, KSPLIT);
    const int STAGES = p.stages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *full = bars;                  // [STAGES]
    uint64_t *empty = bars + STAGES;        // [STAGES]
    uint64_t *tfull = bars + 2 * STAGES;    // [1]
    uint64_t *recv_full = tfull + 1;        // [1] KSPLIT = 2: the peer's partials landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    volatile int *abort_s = reinterpret_cast<volatile int *>(smem + L.misc_off + 4);
    float *bias_s = reinterpret_cast<float *>(smem + L.bias_off);
    float *sbias_s = reinterpret_cast<float *>(smem + L.sbias_off);
    int *hist_s = reinterpret_cast<int *>(smem + L.hist_off);   // [2][E]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int tile = KSPLIT == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const uint32_t crank = KSPLIT == 2 ? cluster_ctarank() : 0u;
    // this CTA's K blocks
    const int kb0 = KSPLIT == 2 && crank == 1 ? p.kb_half : 0;
    const int kb1 = KSPLIT == 2 && crank == 0 ? p.kb_half : p.num_kb;
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
        if (KSPLIT == 2) mbar_init(recv_full, 64 * SLICES);   // every sending thread
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
    if (KSPLIT == 2) cluster_sync_all();   // the peer's barriers exist before any arrival
    fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, armed = 0, armed_parity = 0;
            const uint32_t tx = A_BYTES + (uint32_t)p.bn * BK * 2;
            for (int kb = kb0; kb < kb1; ++kb) {
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
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(&full[stage], phase, abort_s, p.status)) break;
                fence_after();
                const uint32_t a_addr = smem_u32(smem + stage * A_BYTES);
                const uint32_t b_addr = smem_u32(smem + L.b_off + stage * (uint32_t)p.bn * BK * 2);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    mma_bf16(tmem_base, smem_desc_sw128(a_addr + kk * 32),
                             smem_desc_sw128(b_addr + kk * 32), p.idesc, ((kb - kb0) | kk) != 0);
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
        // KSPLIT = 2: rows 64 crank .. 64 crank + 63 are this CTA's; its other rows' partials
        // go to the peer
        const bool own = KSPLIT == 1 || (q >> 1) == (int)crank;
        const int cps = (p.bn + 32 * SLICES - 1) / (32 * SLICES) * 32;   // columns per slice
        const int cs0 = slice * cps, cs1 = min(p.bn, (slice + 1) * cps);
        // tcgen05.ld is warp-collective and the epilogue warps share named barriers:
        // all of them decide together
        const bool ok = epilogue_all<NT>(mbar_wait(tfull, 0, abort_s, p.status) && *abort_s == 0);
        fence_after();
        if (KSPLIT == 2 && !own) {
            // send this slice's partials of the peer's rows, then arrive on its barrier
            // (also after an abort, so that the peer does not wait for them)
            const uint32_t peer = crank ^ 1u;
            const int prow = (q & 1) * 32 + lane;   // row inside the peer's 64
            if (ok) {
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
                const uint32_t recv = mapa_shared(smem_u32(smem + L.recv_off), peer);
                for (int c = cs0; c < cs1; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        if (c + j < p.bn)
                            st_cluster_v4(recv + ((uint32_t)((c + j) >> 2) * 64u + (uint32_t)prow) * 16u,
                                          v[j], v[j + 1], v[j + 2], v[j + 3]);
                }
            }
            mbar_arrive_cluster(mapa_shared(smem_u32(recv_full), peer));
        }
        float val[KMAX], raw[KMAX];   // raw: the entry's logit (MODE > ROUTE_PLAIN)
        int idx[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            val[j] = -INFINITY;
            raw[j] = -INFINITY;
            idx[j] = -1;
        }
        // plain routing with k <= 4 selects by rank keys; larger lists (whose key trees
        // spill registers) and the routing variants by list insertion
        constexpr bool KEYED = MODE == ROUTE_PLAIN && KMAX <= 4;
        uint32_t kk[KMAX];
        int ki[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            kk[j] = 0u;
            ki[j] = -1;
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
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c + j < p.E) dst[j] = v[j] + bias_s[c + j];
            }
        };
        // the peer's partial logits of one of this CTA's rows, columns c .. c + 3
        const int lrow = (q & 1) * 32 + lane;
        auto add_recv = [&](float (&v)[32], int c) {
            if constexpr (KSPLIT == 2) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    if (c + j < p.bn) {
                        const float4 pv = *reinterpret_cast<const float4 *>(
                            smem + L.recv_off + ((size_t)((c + j) >> 2) * 64 + lrow) * 16);
                        v[j] += pv.x;
                        v[j + 1] += pv.y;
                        v[j + 2] += pv.z;
                        v[j + 3] += pv.w;
                    }
            }
        };
        if (ok) {
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
            if (KSPLIT == 2 && own) mbar_wait<true>(recv_full, 0, abort_s, p.status);
            if (!own) {
                // KSPLIT = 2: sent above; only the merge barriers remain
            } else if (MODE == ROUTE_GROUP) {
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
            } else if (KEYED) {
                // the slice's candidates 32 columns at a time: the chunk's best KMAX, then
                // (after the first chunk) merged with the running list
                for (int c = cs0; c < cs1; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
                    add_recv(v, c);
                    store_logits(v, c);
                    uint32_t o[32];
                    int id[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        id[j] = c + j;
                        o[j] = c + j < p.E ? rank_key(v[j] + bias_s[c + j]) : 0u;
                    }
                    if (c == cs0) {
                        top_by_key<32, KMAX>(o, id, kk, ki);
                    } else {
                        uint32_t co[KMAX];
                        int ci[KMAX];
                        top_by_key<32, KMAX>(o, id, co, ci);
                        uint32_t mo[2 * KMAX];
                        int mi[2 * KMAX];
#pragma unroll
                        for (int j = 0; j < KMAX; ++j) {
                            mo[j] = kk[j];
                            mi[j] = ki[j];
                            mo[KMAX + j] = co[j];
                            mi[KMAX + j] = ci[j];
                        }
                        top_by_key<2 * KMAX, KMAX>(mo, mi, kk, ki);
                    }
                }
            } else {
                for (int c = cs0; c < cs1; c += 32) {
                    float v[32];
                    tmem_ld32(taddr + c, v);
                    add_recv(v, c);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int e = c + j;
                        if (e < p.E) push(v[j], e);
                    }
                    store_logits(v, c);
                }
            }
            if (KEYED && SLICES > 1) {
                // keyed lists of slices 1.. into the stage ring (every MMA has read it);
                // group 0 takes the best KMAX of all SLICES lists
                uint32_t *lk = reinterpret_cast<uint32_t *>(smem);   // [SLICES-1][BM][KMAX]
                int *lki = reinterpret_cast<int *>(lk + (SLICES - 1) * BM * KMAX);
                if (slice > 0 && own)
#pragma unroll
                    for (int j = 0; j < KMAX; ++j) {
                        lk[((slice - 1) * BM + r) * KMAX + j] = kk[j];
                        lki[((slice - 1) * BM + r) * KMAX + j] = ki[j];
                    }
                epilogue_sync<NT>();
                if (slice == 0 && own) {
                    constexpr int NC = SLICES * KMAX;   // 2..32, a power of two
                    uint32_t mo[NC];
                    int mi[NC];
#pragma unroll
                    for (int j = 0; j < KMAX; ++j) {
                        mo[j] = kk[j];
                        mi[j] = ki[j];
                    }
#pragma unroll
                    for (int g = 0; g < SLICES - 1; ++g)
#pragma unroll
                        for (int j = 0; j < KMAX; ++j) {
                            mo[(g + 1) * KMAX + j] = lk[(g * BM + r) * KMAX + j];
                            mi[(g + 1) * KMAX + j] = lki[(g * BM + r) * KMAX + j];
                        }
                    top_by_key<NC, KMAX>(mo, mi, kk, ki);
                }
            } else if (SLICES > 1) {
                // lists of slices 1.. into the stage ring (every MMA has read it), then
                // group 0 pushes them in slice order, i.e. in increasing expert id
                float *lv = reinterpret_cast<float *>(smem);   // [SLICES-1][BM][KMAX]
                float *lr = lv + (SLICES - 1) * BM * KMAX;
                int *li = reinterpret_cast<int *>(lr + (SLICES - 1) * BM * KMAX);
                if (slice > 0 && own)
#pragma unroll
                    for (int j = 0; j < KMAX; ++j) {
                        lv[((slice - 1) * BM + r) * KMAX + j] = val[j];
                        lr[((slice - 1) * BM + r) * KMAX + j] = raw[j];
                        li[((slice - 1) * BM + r) * KMAX + j] = idx[j];
                    }
                epilogue_sync<NT>();
                if (slice == 0 && own)
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
            if (KEYED) {
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    val[j] = key_value(kk[j]);
                    idx[j] = ki[j];
                }
            }
            if (slice == 0 && own && tok < p.rows) {
                // softmax over the chosen experts' logits
                float lg[KMAX];
#pragma unroll
                for (int j = 0; j < KMAX; ++j) lg[j] = MODE == ROUTE_PLAIN ? val[j] : raw[j];
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
                // KSPLIT = 2: the CTA's own segment only (the peer writes the other)
                for (int j = etid; j < 2 * p.E; j += NT) {
                    const int seg = 2 * tile + j / p.E;
                    if (KSPLIT == 2 && j / p.E != (int)crank) continue;
                    if (seg < p.nseg) p.seg_hist[(size_t)seg * p.E + j % p.E] = hist_s[j];
                }
            }
        }
    }

    fence_before();
    __syncthreads();
    if (KSPLIT == 2) cluster_sync_all();   // no CTA leaves while its peer may still write to it
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(p.tmem_cols)
                     : "memory");
    }
}

// Ring depth: as many stages as the shared memory of one CTA (SLICES = 4: one CTA per SM)
// or of half an SM (SLICES <= 2: two per SM) holds, at least enough to stage the slices'
// top-k lists for the merge; 0 when fewer than two stages fit.
int ring_stages(int bn, int E, int slices, int kmax, int ksplit) {
    const uint32_t limit = (slices == 4 ? 227u : 113u) * 1024u;
    const uint32_t fixed = route_smem(bn, E, 0, ksplit).alloc;
    if (fixed >= limit) return 0;
    const uint32_t stage_bytes = A_BYTES + (uint32_t)bn * BK * 2;
    const int lists = (slices - 1) * BM * kmax * 12;
    int st = (int)std::min<uint32_t>(MAX_STAGES, (limit - fixed) / stage_bytes);
    while (st * (int)stage_bytes < lists) ++st;
    if (st < 2 || st > MAX_STAGES || route_smem(bn, E, st, ksplit).alloc > limit) return 0;
    return st;
}

template <int KMAX, int SLICES, int MODE, int KSPLIT>
cudaError_t launch_route_tc(const CUtensorMap &mx, const CUtensorMap &mw, const RouteParams &prm,
                            int tiles, cudaStream_t s) {
    auto kern = route_tc_kernel<KMAX, SLICES, MODE, KSPLIT>;
    RouteParams p = prm;
    p.kb_half = (p.num_kb + 1) / 2;
    p.stages = ring_stages(p.bn, p.E, SLICES, KMAX, KSPLIT);
    if (p.stages == 0) return cudaErrorInvalidConfiguration;
    const RouteSmem L = route_smem(p.bn, p.E, p.stages, KSPLIT);
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
    if (KSPLIT == 1)
        return launch_pdl(kern, dim3(tiles), dim3(64 + 128 * SLICES), L.alloc, s, mx, mw, p);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * tiles, 1, 1);
    cfg.blockDim = dim3(64 + 128 * SLICES, 1, 1);
    cfg.dynamicSmemBytes = L.alloc;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, mx, mw, p);
}

// Tiles fewer than the SMs: split the hidden dimension over a cluster of two CTAs per tile
// (at least two K blocks); four column slices while one CTA per SM covers every CTA, two
// otherwise (two CTAs of 320 threads fit on an SM). Lists longer than 8, and the
// group-limited routing, run one unsplit, unsliced CTA per tile.
template <int KMAX>
cudaError_t launch_route_k(const CUtensorMap &mx, const CUtensorMap &mw, const RouteParams &prm,
                           int tiles, int num_sms, cudaStream_t s) {
    if (tiles <= 0) return cudaSuccess;
    if (prm.group_limit > 0) return launch_route_tc<KMAX, 1, ROUTE_GROUP, 1>(mx, mw, prm, tiles, s);
    if constexpr (KMAX > 8) {
        (void)num_sms;
        if (prm.sel_bias != nullptr)
            return launch_route_tc<KMAX, 1, ROUTE_SELBIAS, 1>(mx, mw, prm, tiles, s);
        return launch_route_tc<KMAX, 1, ROUTE_PLAIN, 1>(mx, mw, prm, tiles, s);
    } else {
        const bool wide_split = 2 * tiles <= num_sms;
        const bool split = tiles < num_sms && prm.num_kb >= 2 &&
                           ring_stages(prm.bn, prm.E, wide_split ? 4 : 2, KMAX, 2) > 0;
        const int ctas = split ? 2 * tiles : tiles;
        const bool wide = ctas <= num_sms;
        const bool sb = prm.sel_bias != nullptr;
        if (split) {
            if (sb)
                return wide ? launch_route_tc<KMAX, 4, ROUTE_SELBIAS, 2>(mx, mw, prm, tiles, s)
                            : launch_route_tc<KMAX, 2, ROUTE_SELBIAS, 2>(mx, mw, prm, tiles, s);
            return wide ? launch_route_tc<KMAX, 4, ROUTE_PLAIN, 2>(mx, mw, prm, tiles, s)
                        : launch_route_tc<KMAX, 2, ROUTE_PLAIN, 2>(mx, mw, prm, tiles, s);
        }
        if (sb)
            return wide ? launch_route_tc<KMAX, 4, ROUTE_SELBIAS, 1>(mx, mw, prm, tiles, s)
                        : launch_route_tc<KMAX, 2, ROUTE_SELBIAS, 1>(mx, mw, prm, tiles, s);
        return wide ? launch_route_tc<KMAX, 4, ROUTE_PLAIN, 1>(mx, mw, prm, tiles, s)
                    : launch_route_tc<KMAX, 2, ROUTE_PLAIN, 1>(mx, mw, prm, tiles, s);
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
