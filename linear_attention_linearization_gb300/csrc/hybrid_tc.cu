// Tensor-core hybrid attention of the prefill (tcgen05 + TMEM, fed by TMA).
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", sections "Content-Aware Routing with Fixed Budget", "Delayed
// Chunk-Level Selection for Unified Training-Inference Parallelism" and
// "NP-Map: Norm-Preserving Feature Map":
//   SA(t) = {t-W < j <= t} U {j kept by chunk(j) < chunk(t), j <= t-W}
//   LA(t) = {j <= t-W} minus SA(t)
//   y_t   = (sum_SA e^{s-c} v + phi(q)^T S_LA) / (sum_SA e^{s-c} + phi(q)^T z_LA)
//
// One CTA (one per SM) walks the 32-token tiles of one segment of one
// (sequence, kv head).  A tile is M = 128 rows: the G <= 4 query heads of the
// group x 32 tokens (rows of absent heads are padding).  Per tile:
//   U   = Q Wf              -> phi(Q) = ||q|| u / ||u||, u = softmax(U)    (TMEM -> smem)
//   S   = Q [K_band | K_kept]^T, one MMA per block of 32 keys             (TMEM)
//         band = the 32-key blocks covering [t0-W+1, t0+31]; kept = the
//         kept tokens of earlier chunks, a contiguous prefix of the kept table
//   A   = phi(Q) [phi(K_lag) | phi(K_extra)]^T                             (TMEM)
//         lag = the 32 keys [t0-W, t0-W+32) that leave the window during the
//         tile (rows of slotted keys are zero in the feature table); extra =
//         the kept tokens of the tile's own chunk, which are still linear keys
//   O   = A V_lagx + sum_kb P_kb V_kb + phi(Q) S_run                       (TMEM)
//         P = exp(S - c) masked, c = exact row maximum over the softmax keys;
//         masked A and P are written back to TMEM as bf16 pairs over the
//         columns they came from (each thread within the columns it read
//         itself) and feed the MMAs from there
//   dS  = phi(K_lag)^T V_lag, dz = phi(K_lag)^T 1 -> S_run += dS, z_run += dz
//         (fp32 in registers and shared memory, bf16 copy of S_run in smem)
//   y   = O / (sum P + sum A + phi(Q).z_run)                              (TMA store)
// Masks (window, causal lag, chunk of the kept tokens) are applied to the
// logits in TMEM by the row threads -- four warps per TMEM lane quarter, each
// owning a quarter of U, O and dS and every fourth block of 32 keys -- and one
// thread issues every TMA and MMA.
#include <climits>

#include "sm100.cuh"
#include "tma_host.cuh"

namespace still {

using namespace sm100;

struct TCParams {
    Dims dm;
    SegPlan sp;
    int Wr;        // the band starts at t0 - Wr
    int nb;        // band blocks of 32 keys
    int KP;        // rows of the kept tables per (sequence, kv head)
    const int32_t *fsel;
    const float *dS;
    const float *dz;
    int32_t *status;
    long long row_wait_limit;   // limit of the row warps' waits (the issuing thread's: WAIT_LIMIT_CYCLES)
    // gated layer (nullable): pre-activations of the linear branch's per-channel gate,
    // [B, Hq, N, d] bf16; y = (softmax numerator + sigmoid(gate) * linear numerator) / den
    const uint16_t *gate;
};

// q and out: boxes of 32 tokens x 64 columns x G heads.  kband / vband: the
// nb band blocks of a tile in one box; kk<n> / vk<n>: n blocks of 32 rows of
// the kept tables; v / phik: the 32 lag rows; vk16 / phk16: the 16 rows of
// the own-chunk kept tokens.
struct TCMaps {
    CUtensorMap q, out, kband, vband, kk32, kk64, kk128, vk32, vk64, vk128, v, vk16, phik, phk16, wft;
};

// logits (and, once P V is done, dS at 0 and dz at TM_DZ), O, A, row exchange:
// the NP-Map statistics at TM_X share the A columns (they are read before the
// A MMA is issued), row maxima and denominator shares at TM_X2
constexpr int TM_S = 0, TM_DZ = 256, TM_O = 320, TM_A = 448, TM_X = 448, TM_X2 = 496, TM_COLS = 512;
// the gated layer's linear numerator, in logit columns free once P V is done
// (dS takes 0 .. 127 and dz 256 .. 271)
constexpr int TM_LIN = 128;
constexpr int MAX_KEY_BLOCKS = 10;   // 320 logit columns: every block of a tile stays resident
constexpr int NX = 16;               // extra (kept, own chunk) rows per tile

constexpr int RING_SLOTS = 9;        // K (then V) blocks of 32 keys resident; more come in a second batch

template <int D, int DF>
struct TCLayout {
    static constexpr int CBD = D / 64, CBF = DF / 64;
    static constexpr uint32_t Q = 0;
    static constexpr uint32_t WF = Q + CBD * 16384;
    static constexpr uint32_t PHIQ = WF + CBD * DF * 128;
    static constexpr uint32_t SRUN = PHIQ + (CBD > CBF ? CBD : CBF) * 16384;
    static constexpr uint32_t RING = SRUN + CBD * DF * 128;   // CBD regions of RING_SLOTS x 32 rows x 128 B
    static constexpr uint32_t RSTRIDE = RING_SLOTS * 4096;     // bytes between the column-block regions
    // one 1024-byte swizzle atom whose row 0 is 64 bf16 ones: the B operand of
    // phi(K_lag)^T 1 (rows 1..15 feed output columns that are never read)
    static constexpr uint32_t ONES = RING + CBD * RSTRIDE;
    static constexpr uint32_t PHIK = ONES + 1024;
    static constexpr uint32_t VLAG = PHIK + CBF * 6144;
    static constexpr uint32_t XPOS = VLAG + CBD * 6144;
    static constexpr uint32_t ZRUN = XPOS + NX * 4;
    static constexpr uint32_t TOTAL = ZRUN + DF * 4;
};

constexpr int HT_PARTS = 4;                // row warps per TMEM lane quarter
constexpr int HT_ROWS = 128 * HT_PARTS;    // row threads: 16 warps
constexpr int HT_THREADS = HT_ROWS + 128;  // and a warpgroup whose first thread issues every TMA copy and MMA
// registers per thread after the split: the launch gives 96 x 640 = 61440; the
// row warps take 104 x 512 = 53248 and the issuing warpgroup keeps 64 x 128 = 8192
constexpr int HT_LAUNCH_REGS = 96, HT_ROW_REGS = 104, HT_ISSUE_REGS = 64;
static_assert(HT_ROWS * HT_ROW_REGS + 128 * HT_ISSUE_REGS <= HT_THREADS * HT_LAUNCH_REGS,
              "the register split exceeds what the block is launched with");

template <int D, int DF, bool GATED>
__global__ void __launch_bounds__(HT_THREADS, 1) hybrid_tc_kernel(const __grid_constant__ TCMaps maps, TCParams P)
{
    using Lay = TCLayout<D, DF>;
    constexpr int CBD = Lay::CBD, CBF = Lay::CBF;
    constexpr float LOG2E = 1.4426950408889634f;
    constexpr uint32_t SLOT = CBD * 4096;     // bytes of one ring slot (32 keys x D)
    constexpr uint32_t RSTRIDE = Lay::RSTRIDE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    int32_t *xpos = (int32_t *)(sm + Lay::XPOS);
    float *zrun = (float *)(sm + Lay::ZRUN);

    // issuer -> rows: U, S, A (+ phi(Q) S_run), O, dS complete; rows -> issuer:
    // phi(Q) written, A masked, P written, tile finished (O and dS read,
    // output staged, S_run updated); issuer -> rows: output staging free
    __shared__ uint64_t bar_q, bar_wf, bar_lag, bar_u, bar_s, bar_a, bar_o, bar_ds, bar_k, bar_v;
    __shared__ uint64_t bar_s1, bar_pv1, bar_drain;   // the issuer's own: first-batch S and P V, the drain
    __shared__ uint64_t rdy_phiq, rdy_a, rdy_p1, rdy_p, rdy_epi, stg_free;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    const Dims &dm = P.dm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int unit = b * dm.Hkv + g;
    const int W = dm.W, C = dm.C, lam = dm.lam;
    const int tbeg = P.sp.begin[s], tend = P.sp.begin[s + 1];
    const int ntiles = (tend - tbeg + 31) / 32;
    const int32_t *fs = P.fsel + (size_t)unit * P.KP;
    constexpr bool gated = GATED;

    if (warp == 0) {
        tmem_alloc(&tmem_base, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (uint64_t *bb : {&bar_q, &bar_wf, &bar_lag, &bar_u, &bar_s, &bar_a, &bar_o, &bar_ds, &bar_k, &bar_v, &stg_free,
                             &bar_s1, &bar_pv1, &bar_drain})
            mbar_init(bb, 1);
        for (uint64_t *bb : {&rdy_phiq, &rdy_a, &rdy_p1, &rdy_p, &rdy_epi}) mbar_init(bb, HT_ROWS);
        fence_barrier_init();
        s_abort = 0;
    }
    // the ones row (and zero rows below it)
    for (int i = tid; i < 1024 / 16; i += HT_THREADS) {
        const uint32_t one2 = 0x3f803f80u;   // two bf16 ones
        reinterpret_cast<uint4 *>(sm + Lay::ONES)[i] = i < 8 ? make_uint4(one2, one2, one2, one2) : make_uint4(0, 0, 0, 0);
    }
    // padding rows of absent heads stay zero for the whole kernel
    for (int i = tid; i < CBD * 16384 / 16; i += HT_THREADS) {
        const int row = (i * 16 % 16384) / 128;
        if (row >= dm.G * 32) reinterpret_cast<uint4 *>(sm + Lay::Q)[i] = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    grid_dep_sync();   // the previous kernel's writes are visible from here on

    // bounded wait; gives up early once the other side has given up.  The row
    // warps wait at most P.row_wait_limit cycles, the issuing thread
    // WAIT_LIMIT_CYCLES; a limit below the default (a test of this path) polls
    // without the suspension mbarrier.try_wait may take.
    const bool is_row = warp < HT_ROWS / 32;
    const long long limit = is_row ? P.row_wait_limit : WAIT_LIMIT_CYCLES;
    const bool poll = limit < WAIT_LIMIT_CYCLES;
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
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

    if (warp >= HT_ROWS / 32) {
        // ======================== the issuing warpgroup =========================
        regs_dec<HT_ISSUE_REGS>();
        if (warp == HT_ROWS / 32 && lane == 0 && ntiles > 0) {
            int loads_q = 0, loads_lag = 0;   // copies issued per barrier (for the drain)
            auto load_q = [&](int t0) {
                ++loads_q;
                mbar_expect_tx(&bar_q, dm.G * CBD * 4096);
                for (int cb = 0; cb < CBD; ++cb)
                    tma_load_3d(sm + Lay::Q + cb * 16384, &maps.q, &bar_q, cb * 64, t0, b * dm.Hq + g * dm.G);
            };
            auto load_lag = [&](int t0) {
                const int ct = t0 / C;
                const int xrow = ct < dm.T_max ? ct * lam : P.KP;   // past the table: zero fill
                ++loads_lag;
                mbar_expect_tx(&bar_lag, CBF * (4096 + 2048) + CBD * (4096 + 2048));
                for (int cb = 0; cb < CBF; ++cb) {
                    tma_load_3d(sm + Lay::PHIK + cb * 6144, &maps.phik, &bar_lag, cb * 64, t0 - W, unit);
                    tma_load_3d(sm + Lay::PHIK + cb * 6144 + 4096, &maps.phk16, &bar_lag, cb * 64, xrow, unit);
                }
                for (int cb = 0; cb < CBD; ++cb) {
                    tma_load_3d(sm + Lay::VLAG + cb * 6144, &maps.v, &bar_lag, cb * 64, t0 - W, unit);
                    tma_load_3d(sm + Lay::VLAG + cb * 6144 + 4096, &maps.vk16, &bar_lag, cb * 64, xrow, unit);
                }
            };
            // key blocks [k0, k1) of the tile at t0 into ring slots 0 .. k1-k0-1: K (kv = 0) or
            // V (kv = 1); the band (blocks below nb, first batch only) in one box per column
            // block, the kept prefix in boxes of 4, 2 and 1 blocks
            int loads_k = 0, loads_v = 0;   // copies issued per barrier (for the drain)
            auto load_keys = [&](int t0, int k0, int k1, int kv) {
                uint64_t *bar = kv ? &bar_v : &bar_k;
                ++(kv ? loads_v : loads_k);
                mbar_expect_tx(bar, (k1 - k0) * SLOT);
                for (int cb = 0; cb < CBD; ++cb) {
                    uint8_t *dst = sm + Lay::RING + cb * RSTRIDE;
                    if (k0 == 0) tma_load_3d(dst, kv ? &maps.vband : &maps.kband, bar, cb * 64, t0 - P.Wr, unit);
                    int kb = max(k0, P.nb);
                    while (kb < k1) {
                        const int n = k1 - kb >= 4 ? 4 : (k1 - kb >= 2 ? 2 : 1);
                        const CUtensorMap *mp = n == 4 ? (kv ? &maps.vk128 : &maps.kk128)
                                              : n == 2 ? (kv ? &maps.vk64 : &maps.kk64) : (kv ? &maps.vk32 : &maps.kk32);
                        tma_load_3d(dst + (kb - k0) * 4096, mp, bar, cb * 64, 32 * (kb - P.nb), unit);
                        kb += n;
                    }
                }
            };
            auto store_out = [&](int t0) {
                for (int cb = 0; cb < CBD; ++cb)
                    tma_store_3d(&maps.out, sm + Lay::PHIQ + cb * 16384, cb * 64, t0, b * dm.Hq + g * dm.G);
                tma_store_commit();
            };
            auto nkb_of = [&](int t0) { return P.nb + (min(t0 / C, dm.T_max) * lam + 31) / 32; };
            uint32_t ph_q = 0, ph_lag = 0, ph_s = 0, ph_o = 0, ph_k = 0, ph_v = 0;
            uint32_t pe_phiq = 0, pe_a = 0, pe_p1 = 0, pe_p = 0, pe_epi = 0;
            const uint32_t id_u = idesc_bf16(128, DF, 0, 0);
            const uint32_t id_a = idesc_bf16(128, 32 + NX, 0, 0);
            const uint32_t id_o = idesc_bf16(128, D, 0, 1);
            const uint32_t id_ds = idesc_bf16(128, D, 1, 1);
            const uint32_t id_dz = idesc_bf16(128, 16, 1, 0);   // phi(K_lag)^T 1
            auto koff = [](int k, uint32_t blockbytes) { return (uint64_t)(((k / 64) * blockbytes + (k % 64) * 2) >> 4); };
            auto kdesc = [&](uint32_t base, int k, uint32_t blockbytes) {   // K-major operand, K step k
                return sdesc(base + (k / 64) * blockbytes + (k % 64) * 2, 16, 1024);
            };
            // descriptors advance by adding (byte offset >> 4) to the start-address field
            const uint64_t dQ = sdesc(sb + Lay::Q, 16, 1024), dWF = sdesc(sb + Lay::WF, 16, 1024);
            const uint64_t dKR = sdesc(sb + Lay::RING, 16, 1024);               // K-major ring (keys as N)
            const uint64_t dVR = sdesc(sb + Lay::RING, RSTRIDE, 1024);          // MN-major ring (keys as K)
            const uint64_t dVL = sdesc(sb + Lay::VLAG, 6144, 1024);
            const uint64_t dPQ = sdesc(sb + Lay::PHIQ, 16, 1024), dSR = sdesc(sb + Lay::SRUN, DF * 128, 1024);

            tma_prefetch_desc(&maps.q);
            mbar_expect_tx(&bar_wf, CBD * DF * 128);
            for (int cb = 0; cb < CBD; ++cb) tma_load_2d(sm + Lay::WF + cb * DF * 128, &maps.wft, &bar_wf, cb * 64, 0);
            load_q(tbeg);
            load_lag(tbeg);
            load_keys(tbeg, 0, min(nkb_of(tbeg), RING_SLOTS), 0);
            mbar_arrive(&stg_free);   // the staging buffer starts free
            bool ok = wait(&bar_wf, 0);
            uint32_t ph_s1 = 0, ph_pv1 = 0;

            for (int it = 0; it < ntiles && ok; ++it) {
                const int t0 = tbeg + it * 32;
                const int nkb = nkb_of(t0);
                const int B1 = min(nkb, RING_SLOTS);   // blocks of the first batch through the ring
                const bool has_next = it + 1 < ntiles;
                if (it > 0) {
                    // the rows are done with the previous tile (O and dS read, output staged)
                    if (!(ok = wait(&rdy_epi, pe_epi))) break;
                    pe_epi ^= 1;
                }
                // the previous output leaves, U = Q Wf (the rows wait on it), the staging buffer
                // is handed back once the store has read it, then S = Q K^T: blocks 0 .. B1-1
                // in consecutive slots, one MMA of N = 32 min(B1, 8) per K step and one more for
                // a ninth slot; blocks past the ring come in a second batch once these are read
                if (it > 0) store_out(t0 - 32);
                if (!(ok = wait(&bar_q, ph_q))) break;
                ph_q ^= 1;
                tc_fence_after();
#pragma unroll 1
                for (int k = 0; k < D; k += 16)
                    mma_ss(tmem + TM_O, dQ + koff(k, 16384), dWF + koff(k, DF * 128), id_u, k > 0);
                mma_commit(&bar_u);
                if (it > 0) {
                    tma_store_wait_read();
                    mbar_arrive(&stg_free);
                }
                if (!(ok = wait(&bar_k, ph_k))) break;
                ph_k ^= 1;
                tc_fence_after();
                const int na = B1 < 8 ? B1 : 8;
                const uint32_t id_sa = idesc_bf16(128, 32 * na, 0, 0);
#pragma unroll 1
                for (int k = 0; k < D; k += 16)
                    mma_ss(tmem + TM_S, dQ + koff(k, 16384), dKR + koff(k, RSTRIDE), id_sa, k > 0);
                if (B1 > 8) {
                    const uint32_t id_sb = idesc_bf16(128, 32 * (B1 - 8), 0, 0);
#pragma unroll 1
                    for (int k = 0; k < D; k += 16)
                        mma_ss(tmem + TM_S + 256, dQ + koff(k, 16384), dKR + koff(k, RSTRIDE) + (uint64_t)(8 * 4096 >> 4),
                               id_sb, k > 0);
                }
                if (nkb > B1) {
                    // the second batch: its K blocks replace the first batch's once those are read
                    mma_commit(&bar_s1);
                    if (!(ok = wait(&bar_s1, ph_s1))) break;
                    ph_s1 ^= 1;
                    load_keys(t0, B1, nkb, 0);
                    if (!(ok = wait(&bar_k, ph_k))) break;
                    ph_k ^= 1;
                    tc_fence_after();
                    const uint32_t id_sc = idesc_bf16(128, 32 * (nkb - B1), 0, 0);
#pragma unroll 1
                    for (int k = 0; k < D; k += 16)
                        mma_ss(tmem + TM_S + 32 * B1, dQ + koff(k, 16384), dKR + koff(k, RSTRIDE), id_sc, k > 0);
                }
                mma_commit(&bar_s);
                if (it > 0) load_lag(t0);   // the previous tile's A, dS and z_run are done with it
                // S complete: the ring takes this tile's V blocks (the first batch)
                if (!(ok = wait(&bar_s, ph_s))) break;
                ph_s ^= 1;
                load_keys(t0, 0, B1, 1);
                // phi(Q) written (and every row has read Q): A, O = phi(Q) S_run; the next Q
                if (!(ok = wait(&rdy_phiq, pe_phiq))) break;
                pe_phiq ^= 1;
                if (has_next) load_q(t0 + 32);
                if (!(ok = wait(&bar_lag, ph_lag))) break;
                ph_lag ^= 1;
                tc_fence_after();
                for (int k = 0; k < DF; k += 16)
                    mma_ss(tmem + TM_A, kdesc(sb + Lay::PHIQ, k, 16384), kdesc(sb + Lay::PHIK, k, 6144), id_a, k > 0);
                // the linear numerator: phi(Q) S_run, then (once A is masked) A V_lagx -- into O
                // with the softmax part, or, for the gated layer, into logit columns of its own
                // once every P V MMA has been issued
                auto lin_state = [&](uint32_t d, uint32_t acc0) {
#pragma unroll 1
                    for (int k = 0; k < DF; k += 16)
                        mma_ss(d, dPQ + koff(k, 16384), dSR + (uint64_t)(k * 128 >> 4), id_o, k > 0 ? 1u : acc0);
                };
                auto lin_lag = [&](uint32_t d) {
                    // packed lag pairs in columns 0 .. 15 of A, packed extras in 32 .. 39 (each half
                    // packs within the columns it read, so neither overwrites what the other reads)
#pragma unroll 1
                    for (int kk = 0; kk < 32 + NX; kk += 16)
                        mma_ts(d, tmem + TM_A + (kk < 32 ? kk / 2 : kk), dVL + (uint64_t)(kk * 128 >> 4), id_o, 1);
                };
                if (!gated) lin_state(tmem + TM_O, 0);
                mma_commit(&bar_a);
                if (!(ok = wait(&rdy_a, pe_a))) break;
                pe_a ^= 1;
                tc_fence_after();
                if (!gated) lin_lag(tmem + TM_O);
                // P written, first the blocks below the split, then the rest: O += sum_kb P_kb V_kb
                // (blocks of the second batch once the first batch's V has been read); the gated
                // layer's first P V starts O
                const int split = nkb / 2;
                uint32_t o_acc = gated ? 0u : 1u;
                auto pv = [&](int kb, int slot) {
                    mma_ts(tmem + TM_O, tmem + TM_S + 32 * kb, dVR + (uint64_t)(slot * 4096 >> 4), id_o, o_acc);
                    mma_ts(tmem + TM_O, tmem + TM_S + 32 * kb + 16, dVR + (uint64_t)((slot * 4096 + 2048) >> 4), id_o, 1);
                    o_acc = 1u;
                };
                if (!(ok = wait(&bar_v, ph_v))) break;
                ph_v ^= 1;
                if (!(ok = wait(&rdy_p1, pe_p1))) break;
                pe_p1 ^= 1;
                tc_fence_after();
                for (int kb = 0; kb < min(split, B1); ++kb) pv(kb, kb);
                if (!(ok = wait(&rdy_p, pe_p))) break;
                pe_p ^= 1;
                tc_fence_after();
                for (int kb = min(split, B1); kb < B1; ++kb) pv(kb, kb);
                if (nkb > B1) {
                    mma_commit(&bar_pv1);
                    if (!(ok = wait(&bar_pv1, ph_pv1))) break;
                    ph_pv1 ^= 1;
                    load_keys(t0, B1, nkb, 1);
                    if (!(ok = wait(&bar_v, ph_v))) break;
                    ph_v ^= 1;
                    tc_fence_after();
                    for (int kb = B1; kb < nkb; ++kb) pv(kb, kb - B1);
                }
                if (gated) {
                    // the gated layer's linear numerator, behind the P V MMAs (which have read P)
                    lin_state(tmem + TM_S + TM_LIN, 0);
                    lin_lag(tmem + TM_S + TM_LIN);
                }
                mma_commit(&bar_o);
                // dS into the logit columns right behind the P V MMAs (the tensor pipe runs its
                // MMAs in issue order, so they have read P first), then the next K blocks once
                // every read of the ring is done
                for (int kk = 0; kk < 32; kk += 16) {
                    const uint64_t dphi = sdesc(sb + Lay::PHIK + kk * 128, 6144, 1024);
                    mma_ss(tmem + TM_S, dphi, sdesc(sb + Lay::VLAG + kk * 128, 6144, 1024), id_ds, kk > 0);
                    mma_ss(tmem + TM_DZ, dphi, sdesc(sb + Lay::ONES + kk * 2, 16, 1024), id_dz, kk > 0);
                }
                mma_commit(&bar_ds);
                if (!(ok = wait(&bar_o, ph_o))) break;
                ph_o ^= 1;
                if (has_next) load_keys(t0 + 32, 0, min(nkb_of(t0 + 32), RING_SLOTS), 0);
            }
            if (ok && wait(&rdy_epi, pe_epi)) store_out(tbeg + (ntiles - 1) * 32);
            tma_store_wait_all();
            // Every MMA and copy this thread issued completes before the block releases its
            // shared and tensor memory, also when the block gave up (these waits ignore the
            // abort flag; on the normal path they find everything complete).
            mma_commit(&bar_drain);
            mbar_wait(&bar_drain, 0, P.status);
            mbar_wait(&bar_wf, 0, P.status);
            if (loads_q > 0) mbar_wait(&bar_q, (uint32_t)(loads_q - 1) & 1u, P.status);
            if (loads_lag > 0) mbar_wait(&bar_lag, (uint32_t)(loads_lag - 1) & 1u, P.status);
            if (loads_k > 0) mbar_wait(&bar_k, (uint32_t)(loads_k - 1) & 1u, P.status);
            if (loads_v > 0) mbar_wait(&bar_v, (uint32_t)(loads_v - 1) & 1u, P.status);
        }
        __syncwarp();
    } else {
        // ============================ the row warps =============================
        // Four warps per TMEM lane quarter.  Part p of a row owns the columns
        // [p DQ, (p + 1) DQ) of U, O and dS, the 16-key halves u = p mod 4 of the
        // logit blocks (half u = 2 kb + h: a half's P is packed over the first 8
        // of the 16 columns its own thread read), and, on the parts with the
        // fewest halves, one piece of A (part 3 the lag keys, part 2 the
        // own-chunk extras).
        regs_inc<HT_ROW_REGS>();
        constexpr int DQ = D / HT_PARTS, FQ = DF / HT_PARTS;
        const int quarter = warp & 3, part = warp >> 2;
        const int r = quarter * 32 + lane;            // the tile row (and state row) this thread serves
        const float l2s = LOG2E * rsqrtf((float)D);
        const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16);   // this warp's TMEM lanes

        // running linear state: row f = r, columns [part*DQ, part*DQ + DQ) in fp32
        float srun[DQ];
        {
            const float *S0 = P.dS + ((size_t)unit * (P.sp.nseg + 1) + s) * (size_t)(DF * D);
            const int f = r;
#pragma unroll
            for (int c = 0; c < DQ; c += 4) {
                const float4 x = f < DF ? *reinterpret_cast<const float4 *>(S0 + (size_t)f * D + part * DQ + c)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                srun[c] = x.x;
                srun[c + 1] = x.y;
                srun[c + 2] = x.z;
                srun[c + 3] = x.w;
            }
            if (f < DF && part == 0) zrun[f] = P.dz[((size_t)unit * (P.sp.nseg + 1) + s) * DF + f];
            if (f < DF) {
#pragma unroll
                for (int c8 = 0; c8 < DQ / 8; ++c8) {
                    const int c = part * DQ + c8 * 8;
                    uint4 pk;
                    pk.x = pack_bf16(srun[c8 * 8 + 0], srun[c8 * 8 + 1]);
                    pk.y = pack_bf16(srun[c8 * 8 + 2], srun[c8 * 8 + 3]);
                    pk.z = pack_bf16(srun[c8 * 8 + 4], srun[c8 * 8 + 5]);
                    pk.w = pack_bf16(srun[c8 * 8 + 6], srun[c8 * 8 + 7]);
                    *reinterpret_cast<uint4 *>(sm + Lay::SRUN + (c / 64) * (DF * 128) + sw128(f, (c % 64) / 8)) = pk;
                }
            }
        }
        uint32_t ph_q = 0, ph_u = 0, ph_s = 0, ph_a = 0, ph_o = 0, ph_ds = 0, ph_stg = 0;
        // per-row values the four parts exchange go through TMEM columns of the
        // row's lane: NP-Map statistics of part p at [TM_X + 4p, +3), its row
        // maximum at TM_X2 + p, its share of the denominator at TM_X2 + 4 + p
        auto sync_rows = [&](bool bad) { return named_sync_or(1, HT_ROWS, bad || *(volatile int *)&s_abort); };

        for (int it = 0; it < ntiles; ++it) {
            const int t0 = tbeg + it * 32;
            const int ct = t0 / C;
            const int nkg = min(ct, dm.T_max) * lam;
            const int nkb = P.nb + (nkg + 31) / 32;
            const int band_lo = t0 - P.Wr;

            // row identity and its column ranges
            const int hh = r / 32, t = t0 + (r % 32);
            const bool row_ok = hh < dm.G && t < dm.N;
            // softmax band columns [blo, bhi]; lag columns [llo, lhi] of A
            const int blo = row_ok ? max(t - W + 1, 0) - band_lo : 1, bhi = row_ok ? t - band_lo : 0;
            const int llo = max(0, W - t0), lhi = row_ok ? t - t0 : -1;

            if (tid < NX) xpos[tid] = (ct < dm.T_max && tid < lam) ? fs[ct * lam + tid] : INT_MAX;

            // ---------------- ||q||^2 of my quarter of the row -------------------------------
            bool bad = !wait(&bar_q, ph_q);
            ph_q ^= 1;
            float qa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c8 = 0; c8 < DQ / 8; ++c8) {
                const int c = part * DQ + c8 * 8;
                const uint4 pk = *reinterpret_cast<const uint4 *>(sm + Lay::Q + (c / 64) * 16384 + sw128(r, (c % 64) / 8));
                const uint32_t w4[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                for (int h2 = 0; h2 < 4; ++h2) {
                    const float a0 = __uint_as_float(w4[h2] << 16), a1 = __uint_as_float(w4[h2] & 0xffff0000u);
                    qa[h2] = fmaf(a0, a0, fmaf(a1, a1, qa[h2]));
                }
            }
            const float qn2 = (qa[0] + qa[1]) + (qa[2] + qa[3]);

            // ---------------- phi(Q), pass 1: exponentials of my features (kept) ----------
            bad |= !wait(&bar_u, ph_u);
            ph_u ^= 1;
            tc_fence_after();
            float eu[FQ];
#pragma unroll
            for (int c0 = 0; c0 < FQ; c0 += 16)
                tmem_ld16(tlane + TM_O + part * FQ + c0, *reinterpret_cast<float(*)[16]>(eu + c0));
            tmem_ld_wait();
            float mx = eu[0];
#pragma unroll
            for (int i = 1; i < FQ; ++i) mx = fmaxf(mx, eu[i]);
            const float mu = mx * LOG2E;   // = max(u log2 e): scaling by a positive constant is monotone
            float s2 = 0.f;
#pragma unroll
            for (int i = 0; i < FQ; ++i) {
                eu[i] = exp2_mufu(fmaf(eu[i], LOG2E, -mu));
                s2 = fmaf(eu[i], eu[i], s2);
            }
            {
                const float v[4] = {mu, s2, qn2, 0.f};
                tmem_st4(tlane + TM_X + 4 * part, v);
                tmem_st_wait();
            }
            tc_fence_before();
            if (sync_rows(bad)) break;
            tc_fence_after();
            // number of kept keys (ascending table) at or before t - W, own-chunk extras likewise
            int nvk = 0, nvx = 0;
            {
                int lo = 0, hi = nkg;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldg(fs + mid) <= t - W) lo = mid + 1; else hi = mid;
                }
                nvk = row_ok ? lo : 0;
                while (nvx < NX && xpos[nvx] <= t - W) ++nvx;
                if (!row_ok) nvx = 0;
            }
            float xs[16];
            tmem_ld16(tlane + TM_X, xs);
            tmem_ld_wait();

            // ---------------- phi(Q), pass 2: write my quarter of phi, phi . z --------------
            bad = !wait(&stg_free, ph_stg);    // the previous output has left the staging buffer
            ph_stg ^= 1;
            float den = 0.f;   // my share of the denominator: phi . z here, then my A and P sums
            {
                // the four parts' statistics, combined in part order on every part
                float M = xs[0];
#pragma unroll
                for (int q4 = 1; q4 < HT_PARTS; ++q4) M = fmaxf(M, xs[4 * q4]);
                float ss = 0.f, qq = 0.f;
#pragma unroll
                for (int q4 = 0; q4 < HT_PARTS; ++q4) {
                    ss += xs[4 * q4 + 1] * exp2_mufu(2.f * (xs[4 * q4] - M));
                    qq += xs[4 * q4 + 2];
                }
                const float sc = sqrtf(qq) * rsqrtf(ss) * exp2_mufu(mu - M);   // my exponentials were taken against mu
                float2 dz2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int c8 = 0; c8 < FQ / 8; ++c8) {
                    uint32_t w4[4];
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        const int i = c8 * 8 + h2 * 2;
                        w4[h2] = pack_bf16(sc * eu[i], sc * eu[i + 1]);
                        const int f = part * FQ + i;
                        const float2 zz = *reinterpret_cast<const float2 *>(zrun + f);
                        dz2[h2 & 1] = __ffma2_rn(make_float2(__uint_as_float(w4[h2] << 16),
                                                             __uint_as_float(w4[h2] & 0xffff0000u)),
                                                 zz, dz2[h2 & 1]);
                    }
                    const int f0 = part * FQ + c8 * 8;
                    *reinterpret_cast<uint4 *>(sm + Lay::PHIQ + (f0 / 64) * 16384 + sw128(r, (f0 % 64) / 8)) =
                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                den = (dz2[0].x + dz2[0].y) + (dz2[1].x + dz2[1].y);
            }
            fence_async_smem();
            mbar_arrive(&rdy_phiq);

            // ---------------- softmax pass 1: exact row maximum over my halves ---------------
            bad |= !wait(&bar_s, ph_s);
            ph_s ^= 1;
            tc_fence_after();
            // key columns of block kb this row may use: [clo, chi] (0..31); masks are row
            // ranges, so a 16-key half is often fully in or fully out for the whole warp
            auto key_range = [&](int kb, int &clo, int &chi) {
                clo = kb < P.nb ? blo - 32 * kb : 0;
                chi = kb < P.nb ? bhi - 32 * kb : nvk - 1 - 32 * (kb - P.nb);
            };
            float cmax = -INFINITY;
            for (int u = part; u < 2 * nkb; u += HT_PARTS) {
                const int kb = u >> 1, h = u & 1;
                int clo, chi;
                key_range(kb, clo, chi);
                const int lo = clo - 16 * h, hi = chi - 16 * h;   // this half's keys: [lo, hi] of 0..15
                if (__all_sync(0xffffffffu, hi < 0 || lo > 15)) continue;
                float sv[16];
                tmem_ld16(tlane + TM_S + 16 * u, sv);
                tmem_ld_wait();
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (__all_sync(0xffffffffu, lo <= 0 && hi >= 15)) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i >= lo && i <= hi) m4[i & 3] = fmaxf(m4[i & 3], sv[i]);
                }
                cmax = fmaxf(cmax, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
            }
            tmem_st1(tlane + TM_X2 + part, cmax);
            tmem_st_wait();
            tc_fence_before();
            if (sync_rows(bad)) break;
            tc_fence_after();
            {
                float c4[4];
                tmem_ld4(tlane + TM_X2, c4);
                tmem_ld_wait();
                cmax = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));   // the row maximum (all parts agree)
            }
            const float cm = cmax == -INFINITY ? 0.f : cmax * l2s;   // no softmax key: every P is 0

            // ---------------- A: mask, row sum, bf16 pairs back into TMEM ------------------
            bad = !wait(&bar_a, ph_a);
            ph_a ^= 1;
            tc_fence_after();
            if (part == HT_PARTS - 1) {
                float a[32];
                tmem_ld32(tlane + TM_A, a);
                tmem_ld_wait();
                uint32_t w[16];
                float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float x0 = (i >= llo && i <= lhi) ? a[i] : 0.f;
                    const float x1 = (i + 1 >= llo && i + 1 <= lhi) ? a[i + 1] : 0.f;
                    d4[(i / 2) & 3] += x0 + x1;
                    w[i / 2] = pack_bf16(x0, x1);
                }
                den += (d4[0] + d4[1]) + (d4[2] + d4[3]);
                tmem_st16(tlane + TM_A, w);
                tmem_st_wait();
            } else if (part == HT_PARTS - 2) {
                float a[16];
                tmem_ld16(tlane + TM_A + 32, a);
                tmem_ld_wait();
                uint32_t w[8];
                float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float x0 = i < nvx ? a[i] : 0.f;
                    const float x1 = i + 1 < nvx ? a[i + 1] : 0.f;
                    d4[(i / 2) & 3] += x0 + x1;
                    w[i / 2] = pack_bf16(x0, x1);
                }
                den += (d4[0] + d4[1]) + (d4[2] + d4[3]);
                tmem_st8(tlane + TM_A + 32, w);
                tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(&rdy_a);

            // ---------------- softmax pass 2: P (bf16 pairs) over my halves, in place -------
            // the 16 keys of half u become 8 packed columns at the start of the 16 they
            // came from; blocks below the split go to the tensor cores first
            const int split = nkb / 2;
            bool p1_sent = false;
            auto send_p1 = [&]() {
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&rdy_p1);
                p1_sent = true;
            };
            for (int u = part; u < 2 * nkb; u += HT_PARTS) {
                const int kb = u >> 1, h = u & 1;
                if (kb >= split && !p1_sent) send_p1();
                int clo, chi;
                key_range(kb, clo, chi);
                const int lo = clo - 16 * h, hi = chi - 16 * h;   // this half's keys: [lo, hi] of 0..15
                const bool skip = __all_sync(0xffffffffu, hi < 0 || lo > 15);
                const bool full = __all_sync(0xffffffffu, lo <= 0 && hi >= 15);
                uint32_t w[8];
                float d4[4] = {0.f, 0.f, 0.f, 0.f};
                if (skip) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = 0u;
                } else {
                    float sv[16];
                    tmem_ld16(tlane + TM_S + 16 * u, sv);
                    tmem_ld_wait();
                    if (full) {
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float p0 = exp2_mufu(fmaf(sv[i], l2s, -cm));
                            const float p1 = exp2_mufu(fmaf(sv[i + 1], l2s, -cm));
                            d4[(i / 2) & 3] += p0 + p1;
                            w[i / 2] = pack_bf16(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float p0 = (i >= lo && i <= hi) ? exp2_mufu(fmaf(sv[i], l2s, -cm)) : 0.f;
                            const float p1 = (i + 1 >= lo && i + 1 <= hi) ? exp2_mufu(fmaf(sv[i + 1], l2s, -cm)) : 0.f;
                            d4[(i / 2) & 3] += p0 + p1;
                            w[i / 2] = pack_bf16(p0, p1);
                        }
                    }
                }
                tmem_st8(tlane + TM_S + 16 * u, w);
                den += (d4[0] + d4[1]) + (d4[2] + d4[3]);
            }
            if (!p1_sent) send_p1();
            // my share of the denominator goes with P: the other parts read it once the
            // P V MMAs, which every row's P precedes, are complete
            tmem_st1(tlane + TM_X2 + 4 + part, den);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&rdy_p);

            // ---------------- epilogue: y = O / den (my quarter of the columns) --------------
            // the gated layer: y = (O + sigmoid(a) * O_lin) / den, the gate pre-activations of
            // my columns fetched before the wait
            uint4 gq[DQ / 8];
            if (gated) {
                const uint16_t *gp = P.gate + ((size_t)(b * dm.Hq + g * dm.G + hh) * dm.N + t) * D + part * DQ;
#pragma unroll
                for (int i = 0; i < DQ / 8; ++i)
                    gq[i] = row_ok ? __ldg(reinterpret_cast<const uint4 *>(gp) + i) : make_uint4(0, 0, 0, 0);
            }
            bad |= !wait(&bar_o, ph_o);
            ph_o ^= 1;
            tc_fence_after();
            if (gated) {
                float d4[4];
                tmem_ld4(tlane + TM_X2 + 4, d4);
                tmem_ld_wait();
                const float dtot = (d4[0] + d4[1]) + (d4[2] + d4[3]);
                const float inv = dtot != 0.f ? 1.f / dtot : 0.f;
#pragma unroll
                for (int c0 = 0; c0 < DQ; c0 += 16) {
                    float ov[16], lv[16];
                    tmem_ld16(tlane + TM_O + part * DQ + c0, ov);
                    tmem_ld16(tlane + TM_S + TM_LIN + part * DQ + c0, lv);
                    tmem_ld_wait();
#pragma unroll
                    for (int c8 = 0; c8 < 16; c8 += 8) {
                        const uint4 ga = gq[(c0 + c8) / 8];
                        const uint32_t gw[4] = {ga.x, ga.y, ga.z, ga.w};
                        float yv[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float a = __uint_as_float(i & 1 ? gw[i / 2] & 0xffff0000u : gw[i / 2] << 16);
                            const float gate = __frcp_rn(1.f + exp2_mufu(-a * LOG2E));
                            yv[i] = fmaf(gate, lv[c8 + i], ov[c8 + i]) * inv;
                        }
                        uint4 pk;
                        pk.x = pack_bf16(yv[0], yv[1]);
                        pk.y = pack_bf16(yv[2], yv[3]);
                        pk.z = pack_bf16(yv[4], yv[5]);
                        pk.w = pack_bf16(yv[6], yv[7]);
                        const int d0 = part * DQ + c0 + c8;
                        *reinterpret_cast<uint4 *>(sm + Lay::PHIQ + (d0 / 64) * 16384 + sw128(r, (d0 % 64) / 8)) = pk;
                    }
                }
            } else {
                float d4[4], ov[DQ];   // the denominator shares and my output columns in one round trip
                tmem_ld4(tlane + TM_X2 + 4, d4);
#pragma unroll
                for (int c0 = 0; c0 < DQ; c0 += 16)
                    tmem_ld16(tlane + TM_O + part * DQ + c0, *reinterpret_cast<float(*)[16]>(ov + c0));
                tmem_ld_wait();
                const float dtot = (d4[0] + d4[1]) + (d4[2] + d4[3]);
                const float inv = dtot != 0.f ? 1.f / dtot : 0.f;
#pragma unroll
                for (int c8 = 0; c8 < DQ / 8; ++c8) {
                    const float *o = ov + c8 * 8;
                    uint4 pk;
                    pk.x = pack_bf16(o[0] * inv, o[1] * inv);
                    pk.y = pack_bf16(o[2] * inv, o[3] * inv);
                    pk.z = pack_bf16(o[4] * inv, o[5] * inv);
                    pk.w = pack_bf16(o[6] * inv, o[7] * inv);
                    const int d0 = part * DQ + c8 * 8;
                    *reinterpret_cast<uint4 *>(sm + Lay::PHIQ + (d0 / 64) * 16384 + sw128(r, (d0 % 64) / 8)) = pk;
                }
            }
            // ---------------- state update: S_run += dS, z_run += dz --------------------------
            bad |= !wait(&bar_ds, ph_ds);
            ph_ds ^= 1;
            tc_fence_after();
            {
                const int f = r;
                float dzf;
                {
                    float ds[DQ];
#pragma unroll
                    for (int c0 = 0; c0 < DQ; c0 += 16)
                        tmem_ld16(tlane + TM_S + part * DQ + c0, *reinterpret_cast<float(*)[16]>(ds + c0));
                    dzf = tmem_ld1(tlane + TM_DZ);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < DQ; ++i) srun[i] += ds[i];
                }
                if (f < DF) {
#pragma unroll
                    for (int c8 = 0; c8 < DQ / 8; ++c8) {
                        const int c = part * DQ + c8 * 8;
                        uint4 pk;
                        pk.x = pack_bf16(srun[c8 * 8 + 0], srun[c8 * 8 + 1]);
                        pk.y = pack_bf16(srun[c8 * 8 + 2], srun[c8 * 8 + 3]);
                        pk.z = pack_bf16(srun[c8 * 8 + 4], srun[c8 * 8 + 5]);
                        pk.w = pack_bf16(srun[c8 * 8 + 6], srun[c8 * 8 + 7]);
                        *reinterpret_cast<uint4 *>(sm + Lay::SRUN + (c / 64) * (DF * 128) + sw128(f, (c % 64) / 8)) = pk;
                    }
                    if (part == 0) zrun[f] += dzf;
                }
            }
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&rdy_epi);
            if (bad) *(volatile int *)&s_abort = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool hybrid_tc_supported(const Dims &dm)
{
    if (dm.d != dm.df) return false;
    if (dm.G != 1 && dm.G != 2 && dm.G != 4) return false;
    if (dm.C % 32 != 0 || dm.lam > NX) return false;
    const int Wr = dm.W >= 1 ? (dm.W - 1 + 31) / 32 * 32 : 0;
    const int nb = (Wr + 32) / 32;
    if (nb > 8) return false;   // the band is one TMA box of at most 256 rows
    const int nchunks = (dm.N + dm.C - 1) / dm.C;
    const int maxg = dm.lam * min(dm.T_max, max(nchunks - 1, 0));
    return nb + (maxg + 31) / 32 <= MAX_KEY_BLOCKS;
}

size_t hybrid_tc_smem(const Dims &dm)
{
    return (dm.d == 64 ? TCLayout<64, 64>::TOTAL : TCLayout<128, 128>::TOTAL) + 1024;
}

cudaError_t launch_hybrid_tc(const Dims &dm, const SegPlan &sp, const TCBuffers &bf, const int32_t *fsel,
                             const float *dS, const float *dz, int32_t *status, cudaStream_t s)
{
    KTimer tm(bf.gate ? "hybrid_attn_gated" : "hybrid_attn", s);
    const int D = dm.d, DF = dm.df;
    const uint64_t units = (uint64_t)dm.B * dm.Hkv, heads = (uint64_t)dm.B * dm.Hq;
    const int KP = dm.T_max * dm.lam > 0 ? dm.T_max * dm.lam : 1;
    TCMaps m;
    bool ok = true;
    {
        const int nb = dm.W >= 1 ? ((dm.W - 1 + 31) / 32 * 32 + 32) / 32 : 1;
        uint64_t dq[3] = {(uint64_t)D, (uint64_t)dm.N, heads}, sq[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * dm.N};
        uint32_t boxg[3] = {64, 32, (uint32_t)dm.G};
        ok &= make_tma_map(&m.q, bf.q, 3, dq, sq, boxg, true);
        ok &= make_tma_map(&m.out, bf.out, 3, dq, sq, boxg, true);
        uint64_t dk[3] = {(uint64_t)D, (uint64_t)dm.N, units};
        uint32_t box[3] = {64, 32, 1}, boxb[3] = {64, (uint32_t)(32 * nb), 1};
        ok &= make_tma_map(&m.kband, bf.k, 3, dk, sq, boxb, true);
        ok &= make_tma_map(&m.vband, bf.v, 3, dk, sq, boxb, true);
        ok &= make_tma_map(&m.v, bf.v, 3, dk, sq, box, true);
        uint64_t df3[3] = {(uint64_t)DF, (uint64_t)dm.N, units}, sf[2] = {(uint64_t)DF * 2, (uint64_t)DF * 2 * dm.N};
        ok &= make_tma_map(&m.phik, bf.phik, 3, df3, sf, box, true);
        uint64_t dkp[3] = {(uint64_t)D, (uint64_t)KP, units}, skp[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * KP};
        uint32_t b32[3] = {64, 32, 1}, b64[3] = {64, 64, 1}, b128[3] = {64, 128, 1}, box16[3] = {64, 16, 1};
        ok &= make_tma_map(&m.kk32, bf.kk, 3, dkp, skp, b32, true);
        ok &= make_tma_map(&m.kk64, bf.kk, 3, dkp, skp, b64, true);
        ok &= make_tma_map(&m.kk128, bf.kk, 3, dkp, skp, b128, true);
        ok &= make_tma_map(&m.vk32, bf.vk, 3, dkp, skp, b32, true);
        ok &= make_tma_map(&m.vk64, bf.vk, 3, dkp, skp, b64, true);
        ok &= make_tma_map(&m.vk128, bf.vk, 3, dkp, skp, b128, true);
        ok &= make_tma_map(&m.vk16, bf.vk, 3, dkp, skp, box16, true);
        uint64_t dpk[3] = {(uint64_t)DF, (uint64_t)KP, units}, spk[2] = {(uint64_t)DF * 2, (uint64_t)DF * 2 * KP};
        ok &= make_tma_map(&m.phk16, bf.phk, 3, dpk, spk, box16, true);
        uint64_t dw[2] = {(uint64_t)D, (uint64_t)DF}, sw[1] = {(uint64_t)D * 2};
        uint32_t boxw[2] = {64, (uint32_t)DF};
        ok &= make_tma_map(&m.wft, bf.wft, 2, dw, sw, boxw, true);
    }
    if (!ok) return cudaErrorInvalidValue;
    TCParams p;
    p.dm = dm;
    p.sp = sp;
    p.Wr = dm.W >= 1 ? (dm.W - 1 + 31) / 32 * 32 : 0;
    p.nb = (p.Wr + 32) / 32;
    p.KP = KP;
    p.fsel = fsel;
    p.dS = dS;
    p.dz = dz;
    p.status = status;
    p.row_wait_limit = consumer_wait_limit();
    p.gate = bf.gate;
    dim3 grid(sp.nseg, dm.Hkv, dm.B);
    const size_t smem = hybrid_tc_smem(dm);
    cudaError_t e;
    // the warpgroups' register split draws on what the block is launched with
    auto regs_ok = [](const void *kern) {
        cudaFuncAttributes fa;
        return cudaFuncGetAttributes(&fa, kern) == cudaSuccess && fa.numRegs >= HT_LAUNCH_REGS;
    };
    auto go = [&](auto kern) -> cudaError_t {
        if (!regs_ok((const void *)kern)) return cudaErrorInvalidConfiguration;
        cudaError_t e2 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e2 != cudaSuccess) return e2;
        return launch_kernel(kern, grid, dim3(HT_THREADS), smem, s, m, p);
    };
    if (D == 64) e = p.gate ? go(hybrid_tc_kernel<64, 64, true>) : go(hybrid_tc_kernel<64, 64, false>);
    else e = p.gate ? go(hybrid_tc_kernel<128, 128, true>) : go(hybrid_tc_kernel<128, 128, false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace still
