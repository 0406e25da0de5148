// Self-Saliency score on the tensor cores.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", section "Self-Saliency Score: Predicting Future Utility from
// Local Context": the KL sensitivity between the window distribution with the
// token's own key (a^diag) and without it (a^nodiag), in the closed form
// -log(1 - p_t + 1e-6), averaged over the query heads of a kv head.
//
// Persistent CTAs walk tiles of 32 tokens of one (sequence, kv head): the
// G <= 4 query heads x 32 tokens form the M = 128 rows of one MMA against the
// band of keys [t0 - Wr, t0 + 32) that holds every window of the tile.  One
// thread of a fourth warpgroup issues the TMA copies and the MMAs, tiles
// pipelined over up to four shared-memory / TMEM stages; two groups of four
// row warps take alternate tiles, one thread per row, and reduce each row to its
// off-diagonal window mass relative to the token's own logit while the next
// tiles load and multiply.
#include "sm100.cuh"
#include "tma_host.cuh"

namespace still {

using namespace sm100;

namespace {
constexpr int SC_MAX_NB = 8;         // band blocks of 32 keys (W <= 225)
constexpr int SC_MAX_STAGES = 4;     // tiles in flight
constexpr int SC_ROWS = 256;         // row threads: SC_GROUPS groups of four warps
constexpr int SC_GROUPS = 2;
constexpr int SC_THREADS = SC_ROWS + 128;
constexpr size_t SC_SMEM_CAP = 227 * 1024 - 4096;   // dynamic share of the 227 KB per-block limit
}

struct ScoreTCParams {
    Dims dm;
    int Wr, nb;        // band [t0 - Wr, t0 + 32), nb blocks of 32 keys
    int tiles_per_unit, total_tiles;
    int stages;        // tiles in flight (shared-memory and TMEM stages)
    uint32_t stage_bytes, tmem_stride;
    float *scores;
    int diag;          // 1: write the mean self probability p_t (diagonal attention) instead of the score
    // the prefill's set-up, done by this kernel's threads when kslot is set:
    // status word = 0, slot map = -1, kept tables = 0, W_f^T in bf16
    const float *Wf;
    uint16_t *wft;
    int32_t *kslot;
    // device status word (nullable): a bounded wait that gives up writes
    // STILL_ERR_TIMEOUT here; the row warps' waits give up after
    // row_wait_limit cycles, the issuing thread's after WAIT_LIMIT_CYCLES
    int32_t *status;
    long long row_wait_limit;
    size_t nkslot, nkept16;
    uint4 *kept;
};

// q: boxes of 32 tokens x 64 columns x G heads; k: the nb band blocks in one box
struct ScoreTCMaps {
    CUtensorMap q, k;
};

template <int D, int NB>
__global__ void __launch_bounds__(SC_THREADS, 1) score_tc_kernel(const __grid_constant__ ScoreTCMaps maps, ScoreTCParams P)
{
    constexpr int CBD = D / 64;
    constexpr uint32_t QB = CBD * 16384;          // Q tile bytes
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    // full: a stage's Q and K arrived; mma: its logits are in TMEM (and its
    // shared memory is free); tfree: the rows have read its TMEM columns
    __shared__ uint64_t bar_full[SC_MAX_STAGES], bar_mma[SC_MAX_STAGES], bar_tfree[SC_MAX_STAGES], bar_drain;
    __shared__ uint32_t tmem_base;
    __shared__ float hsc[SC_GROUPS][2][4 * 32];   // per group, two tiles: head scores by (head, token)
    __shared__ int s_abort;

    const Dims &dm = P.dm;
    const int NS = P.stages;
    const uint32_t STB = P.stage_bytes, KBB = P.nb * 4096;   // bytes of a stage, of one K column block
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int first = blockIdx.x, step = gridDim.x;
    const int my_tiles = first < P.total_tiles ? (P.total_tiles - first + step - 1) / step : 0;

    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&bar_full[i], 1);
            mbar_init(&bar_mma[i], 1);
            mbar_init(&bar_tfree[i], SC_ROWS / SC_GROUPS);
        }
        mbar_init(&bar_drain, 1);
        fence_barrier_init();
        s_abort = 0;
    }
    // padding rows of absent heads: zero in every stage buffer, never written again
    for (int st = 0; st < NS; ++st)
        for (int i = tid; i < (int)(QB / 16); i += SC_THREADS) {
            const int row = (i * 16 % 16384) / 128;
            if (row >= dm.G * 32) reinterpret_cast<uint4 *>(sm + st * STB)[i] = make_uint4(0, 0, 0, 0);
        }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    grid_dep_sync();   // the previous kernel's writes are visible from here on
    if (P.kslot) {
        const size_t gt = (size_t)blockIdx.x * SC_THREADS + tid, nt = (size_t)gridDim.x * SC_THREADS;
        for (size_t i = gt; i < P.nkslot / 4; i += nt) reinterpret_cast<int4 *>(P.kslot)[i] = make_int4(-1, -1, -1, -1);
        for (size_t i = P.nkslot / 4 * 4 + gt; i < P.nkslot; i += nt) P.kslot[i] = -1;
        for (size_t i = gt; i < P.nkept16; i += nt) P.kept[i] = make_uint4(0, 0, 0, 0);
        for (size_t i = gt; i < (size_t)dm.d * dm.df; i += nt) {
            const int f = (int)(i / dm.d), e = (int)(i % dm.d);
            P.wft[i] = f2bf(P.Wf[(size_t)e * dm.df + f]);
        }
    }

    // bounded wait; gives up early once another thread has given up.  A limit
    // below the default (a test of this path) polls without the suspension
    // mbarrier.try_wait may take, so that the clock limit is what decides.
    auto wait = [&](uint64_t *bar, uint32_t parity, long long limit) -> bool {
        const bool poll = limit < WAIT_LIMIT_CYCLES;
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        const long long c0 = clock64();
        while (!(poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))) {
            if (*(volatile int *)&s_abort) return false;
            if (clock64() - c0 > limit) {
                set_status(P.status, STILL_ERR_TIMEOUT);
                *(volatile int *)&s_abort = 1;
                return false;
            }
        }
        return true;
    };
    auto tile_coords = [&](int i, int &unit, int &t0) {
        const int tile = first + i * step;
        unit = tile / P.tiles_per_unit;
        t0 = (tile % P.tiles_per_unit) * 32;
    };

    if (warp >= SC_ROWS / 32) {
        // ======================= the issuing warpgroup =======================
        regs_dec<56>();
        if (warp == SC_ROWS / 32 && lane == 0 && my_tiles > 0) {
            const uint32_t idesc = idesc_bf16(128, P.nb * 32, 0, 0);
            const uint64_t d0 = sdesc(sb, 16, 1024);
            auto issue_load = [&](int i) {
                int unit, t0;
                tile_coords(i, unit, t0);
                const int st = i % NS;
                uint8_t *qd = sm + st * STB;
                uint8_t *kd = qd + QB;
                const int b = unit / dm.Hkv, g = unit % dm.Hkv;
                mbar_expect_tx(&bar_full[st], dm.G * CBD * 4096 + P.nb * CBD * 4096);
                for (int cb = 0; cb < CBD; ++cb) {
                    tma_load_3d(qd + cb * 16384, &maps.q, &bar_full[st], cb * 64, t0, b * dm.Hq + g * dm.G);
                    tma_load_3d(kd + cb * KBB, &maps.k, &bar_full[st], cb * 64, t0 - P.Wr, unit);
                }
            };
            uint32_t ph_full = 0, ph_mma = 0, ph_tf = 0;   // one parity bit per stage
            int loaded = 0, arrived = 0;                  // tiles whose copies were issued / waited for
            bool ok = true;
            for (int i = 0; i < NS && i < my_tiles; ++i, ++loaded) issue_load(i);
            for (int i = 0; i < my_tiles && ok; ++i) {
                const int st = i % NS;
                ok &= wait(&bar_full[st], (ph_full >> st) & 1u, WAIT_LIMIT_CYCLES);
                if (!ok) break;
                ++arrived;
                ph_full ^= 1u << st;
                if (i >= NS) {   // the rows are done with tile i - NS in this TMEM stage
                    ok &= wait(&bar_tfree[st], (ph_tf >> st) & 1u, WAIT_LIMIT_CYCLES);
                    if (!ok) break;
                    ph_tf ^= 1u << st;
                }
                tc_fence_after();
                const uint64_t qa = d0 + ((st * STB) >> 4), ka = qa + (QB >> 4);
#pragma unroll 1
                for (int k = 0; k < D; k += 16)
                    mma_ss(tmem + st * P.tmem_stride, qa + (((k / 64) * 16384 + (k % 64) * 2) >> 4),
                           ka + (((k / 64) * KBB + (k % 64) * 2) >> 4), idesc, k > 0);
                mma_commit(&bar_mma[st]);
                if (i + NS < my_tiles) {
                    // the stage's shared memory is free once this MMA has read it
                    ok &= wait(&bar_mma[st], (ph_mma >> st) & 1u, WAIT_LIMIT_CYCLES);
                    if (!ok) break;
                    issue_load(i + NS);
                    ++loaded;
                }
                ph_mma ^= 1u << st;
            }
            // Every MMA and copy this thread issued completes before the block's shared and
            // tensor memory are released, also when the block gave up (these waits ignore the
            // abort flag; on the normal path they find everything complete).
            mma_commit(&bar_drain);
            mbar_wait(&bar_drain, 0, P.status);
            for (int j = arrived; j < loaded; ++j) mbar_wait(&bar_full[j % NS], (uint32_t)(j / NS) & 1u, P.status);
        }
        __syncwarp();
    } else {
        // ============================= the row warps =============================
        // Two groups of four warps take alternate tiles; in a group, warp q
        // serves TMEM lane quarter q (query head q of the tile) and each thread
        // one whole row, so the only exchange is the head mean.
        regs_inc<224>();
        const int quarter = warp & 3, grp = warp >> 2;
        const int hh = quarter, tt = lane;
        constexpr int BC = NB * 32;   // band columns
        const int W = dm.W;
        const float l2s = 1.4426950408889634f * rsqrtf((float)D);   // log2(e) / sqrt(d)
        const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16);
        for (int i = grp, n = 0; i < my_tiles; i += SC_GROUPS, ++n) {
            const int st = i % NS;
            int unit, t0;
            tile_coords(i, unit, t0);
            // the k-th use of a stage completes phase k of its barrier; this group
            // has seen tile i - 2 complete, so every earlier use of the stage has too
            bool bad = !wait(&bar_mma[st], (uint32_t)(i / NS) & 1u, P.row_wait_limit);
            tc_fence_after();
            float v[BC];
#pragma unroll
            for (int c0 = 0; c0 < BC; c0 += 32)
                tmem_ld32(tlane + st * P.tmem_stride + c0, *reinterpret_cast<float(*)[32]>(v + c0));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bar_tfree[st]);

            // window columns [lo, self_c): the keys other than the token itself; the
            // token's own logit is at self_c = Wr + tt, in the last band block.  The
            // masses are taken relative to the token's own logit, so no row maximum
            // is needed: a mass that overflows to +inf gives p = 0 exactly.
            const int t = t0 + tt;
            const int band_lo = t0 - P.Wr;
            const int lo = max(max(t - W + 1, 0) - band_lo, 0);
            const int self_c = P.Wr + tt;
            float sself = 0.f;
#pragma unroll
            for (int x = BC - 32; x < BC; ++x)
                if (x == self_c) sself = v[x];
            const float ms = sself * l2s;
            float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int x = 0; x < BC - 32; ++x) {   // before the last block: every column is below self_c
                const float e = exp2_mufu(fmaf(v[x], l2s, -ms));
                o4[x & 3] += x >= lo ? e : 0.f;
            }
#pragma unroll
            for (int x = BC - 32; x < BC; ++x) {
                const float e = exp2_mufu(fmaf(v[x], l2s, -ms));
                o4[x & 3] += (x >= lo && x < self_c) ? e : 0.f;
            }
            const float oth = (o4[0] + o4[1]) + (o4[2] + o4[3]);
            float *hs = hsc[grp][n & 1];
            hs[hh * 32 + tt] = (hh < dm.G && t < dm.N) ? (P.diag ? 1.f / (1.f + oth) : saliency_from_stats(oth, 1.f)) : 0.f;
            // the group's four heads are in; the other half of hsc[grp] was read
            // before this barrier by the warp that reads this half after it
            if (named_sync_or(1 + grp, 128, bad || *(volatile int *)&s_abort)) break;
            if (quarter == 0 && t < dm.N) {
                float a = 0.f;
                for (int h = 0; h < dm.G; ++h) a += hs[h * 32 + tt];
                P.scores[(size_t)unit * dm.N + t] = a / dm.G;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

bool score_tc_supported(const Dims &dm)
{
    if (dm.d != 64 && dm.d != 128) return false;
    if (dm.G != 1 && dm.G != 2 && dm.G != 4) return false;
    if (dm.W < 1) return false;
    const int Wr = (dm.W - 1 + 31) / 32 * 32;
    return (Wr + 32) / 32 <= SC_MAX_NB;
}

cudaError_t launch_score_tc(const Dims &dm, const uint16_t *q, const uint16_t *k, float *scores, cudaStream_t s,
                            const PrepArgs *prep, int diag)
{
    KTimer tm("score", s);
    ScoreTCMaps m;
    const int D = dm.d;
    uint64_t dq[3] = {(uint64_t)D, (uint64_t)dm.N, (uint64_t)dm.B * dm.Hq};
    uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * dm.N};
    ScoreTCParams p;
    p.dm = dm;
    p.Wr = (dm.W - 1 + 31) / 32 * 32;
    p.nb = (p.Wr + 32) / 32;
    uint32_t boxq[3] = {64, 32, (uint32_t)dm.G}, boxk[3] = {64, (uint32_t)(32 * p.nb), 1};
    bool ok = make_tma_map(&m.q, q, 3, dq, sq, boxq, true);
    uint64_t dk[3] = {(uint64_t)D, (uint64_t)dm.N, (uint64_t)dm.B * dm.Hkv};
    ok = ok && make_tma_map(&m.k, k, 3, dk, sq, boxk, true);
    if (!ok) return cudaErrorInvalidValue;
    p.tiles_per_unit = (dm.N + 31) / 32;
    p.total_tiles = p.tiles_per_unit * dm.B * dm.Hkv;
    p.scores = scores;
    p.diag = diag;
    p.Wf = prep ? prep->Wf : nullptr;
    p.wft = prep ? prep->wft : nullptr;
    p.status = prep ? prep->status : nullptr;
    p.row_wait_limit = consumer_wait_limit();
    p.kslot = prep ? prep->kslot : nullptr;
    p.nkslot = prep ? (size_t)dm.B * dm.Hkv * dm.N : 0;
    p.kept = prep ? reinterpret_cast<uint4 *>(prep->kept) : nullptr;
    p.nkept16 = prep ? prep->kept_bytes / 16 : 0;
    const uint32_t qb = (uint32_t)(D / 64) * 16384, kbytes = (uint32_t)p.nb * 32 * D * 2;
    p.stage_bytes = (qb + kbytes + 1023) & ~1023u;
    p.tmem_stride = p.nb * 32 <= 128 ? 128 : 256;
    int ns = (int)((SC_SMEM_CAP - 1024) / p.stage_bytes);
    if (ns > SC_MAX_STAGES) ns = SC_MAX_STAGES;
    if (ns > (int)(512 / p.tmem_stride)) ns = 512 / p.tmem_stride;
    p.stages = ns;
    int dev = 0, nsm = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int grid = p.total_tiles < nsm ? p.total_tiles : nsm;
    const size_t smem = (size_t)ns * p.stage_bytes + 1024;
    cudaError_t e = cudaSuccess;
#define STILL_SCORE(DD, NBB)                                                                                    \
    e = cudaFuncSetAttribute(score_tc_kernel<DD, NBB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);  \
    if (e != cudaSuccess) return e;                                                                             \
    e = launch_kernel(score_tc_kernel<DD, NBB>, grid, dim3(SC_THREADS), smem, s, m, p);                       \
    if (e != cudaSuccess) return e;
#define STILL_SCORE_NB(DD)                                                                                      \
    switch (p.nb) {                                                                                             \
    case 1: STILL_SCORE(DD, 1) break;                                                                           \
    case 2: STILL_SCORE(DD, 2) break;                                                                           \
    case 3: STILL_SCORE(DD, 3) break;                                                                           \
    case 4: STILL_SCORE(DD, 4) break;                                                                           \
    case 5: STILL_SCORE(DD, 5) break;                                                                           \
    case 6: STILL_SCORE(DD, 6) break;                                                                           \
    case 7: STILL_SCORE(DD, 7) break;                                                                           \
    default: STILL_SCORE(DD, 8) break;                                                                          \
    }
    if (D == 64) { STILL_SCORE_NB(64) }
    else { STILL_SCORE_NB(128) }
#undef STILL_SCORE_NB
#undef STILL_SCORE
    return cudaGetLastError();
}

}  // namespace still
