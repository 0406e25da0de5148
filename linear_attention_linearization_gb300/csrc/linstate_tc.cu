// Key features and per-segment linear-state sums on the tensor cores.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", section "NP-Map: Norm-Preserving Feature Map" (phi) and
// section "Content-Aware Routing with Fixed Budget" (tokens that are not kept
// are accumulated into the linear-attention recurrent state).
//
// CTA s of a (sequence, kv head) walks 128-key blocks of its key range:
//   U    = K_blk Wf                          (tcgen05, TMEM)
//   phi  = ||k|| u / ||u||, u = softmax(U)   (one thread per key row)
//          -> the bf16 feature table (zero rows for slotted keys); a kept key
//             also gets its unmasked phi in the kept table (the selection
//             kernel copies its K and V rows there)
//   dS  += phi_blk^T V_blk                   (tcgen05, accumulated in TMEM)
//   dz  += phi_blk^T 1                       (tcgen05: an all-ones B operand)
// Four row threads share a key (each takes a quarter of its features and of
// its dimensions); a seventeenth warp issues the TMA copies and the MMAs: U runs
// two blocks ahead of the rows in a double-buffered TMEM U (the U of block b+2
// is issued as soon as the rows are done with block b and its K has come in),
// dS and dz as soon as a block's features are in shared memory.
// The range is [b_s - W, b_{s+1} - W) clipped to [0, N), b_s the first token
// of segment s: the keys that leave the window while segment s runs (the last
// segment also writes the features of the final W keys).  Only keys below N - W enter dS: the others never
// leave the window.  An exclusive scan over segments then gives each
// segment's starting state.
#include "sm100.cuh"
#include "tma_host.cuh"

namespace still {

using namespace sm100;

struct LinTCParams {
    Dims dm;
    SegPlan sp;
    const int32_t *kslot;   // per key: row of the kept tables, -1 when the key is in no budget slot
    uint16_t *phik, *phk;
    float *dS;
    float *dz;
    int32_t *status;
};

struct LinTCMaps {
    CUtensorMap k, v, wft, phik;   // phik: the feature table, boxes of 128 keys x 64 features
};

template <int D, int DF>
struct LinLayout {
    static constexpr int CBD = D / 64, CBF = DF / 64;
    static constexpr uint32_t WF = 0;                          // [DF rows x D]
    static constexpr uint32_t STAGE = WF + CBD * DF * 128;     // 2 x (K [128 x D] + V [128 x D])
    static constexpr uint32_t STAGE_BYTES = 2 * CBD * 16384;
    static constexpr uint32_t PHI = STAGE + 2 * STAGE_BYTES;   // [128 rows x DF], always 2 blocks
    static constexpr uint32_t ONES = PHI + 2 * 16384;          // [16 rows x 128 keys]: row 0 ones, K-major
    static constexpr uint32_t TOTAL = ONES + 2 * 2048;
};

constexpr int LS_PARTS = 4;                   // row threads per key
constexpr int LS_ROWS = 128 * LS_PARTS;       // row threads: 16 warps
constexpr int LS_THREADS = LS_ROWS + 32;      // and the issuing warp

template <int D, int DF>
__global__ void __launch_bounds__(LS_THREADS, 1) linstate_tc_kernel(const __grid_constant__ LinTCMaps maps, LinTCParams P)
{
    using Lay = LinLayout<D, DF>;
    constexpr int CBD = Lay::CBD, CBF = Lay::CBF;
    constexpr float LOG2E = 1.4426950408889634f;
    constexpr int TM_U = 0, TM_DS = 256, TM_DZ = 384;   // U double-buffered at 0 and 128
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t bar_wf, bar_full[2], bar_u[2], bar_ds, rdy_phi, phi_free;
    __shared__ float xch[LS_PARTS][128][3];   // per key row and part: max, sum of squares, ||k||^2 part
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    const Dims &dm = P.dm;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const size_t unit = (size_t)b * dm.Hkv + g;
    const int klo = max(0, P.sp.begin[s] - dm.W);
    const int fhi = P.sp.begin[s + 1] - dm.W;                              // keys folded: [klo, fhi)
    const int khi = s == P.sp.nseg - 1 ? dm.N : max(fhi, klo);            // features written: [klo, khi)
    const int nblk = khi > klo ? (khi - klo + 127) / 128 : 0;

    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_wf, 1);
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(&bar_u[0], 1);
        mbar_init(&bar_u[1], 1);
        mbar_init(&bar_ds, 1);
        mbar_init(&rdy_phi, LS_ROWS);
        mbar_init(&phi_free, 1);
        fence_barrier_init();
        s_abort = 0;
    }
    // the second feature block stays zero when d_f = 64 (it is read as padding rows of dS)
    if (CBF == 1)
        for (int i = tid; i < 16384 / 16; i += LS_THREADS) reinterpret_cast<uint4 *>(sm + Lay::PHI + 16384)[i] = make_uint4(0, 0, 0, 0);
    // the all-ones operand: row 0 of each 64-key block is ones, rows 1..15 zero
    for (int i = tid; i < 2 * 2048 / 16; i += LS_THREADS) {
        const int row = (i * 16 % 2048) / 128;
        const uint32_t one2 = 0x3f803f80u;   // two bf16 ones
        reinterpret_cast<uint4 *>(sm + Lay::ONES)[i] = row == 0 ? make_uint4(one2, one2, one2, one2) : make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    grid_dep_sync();   // the previous kernel's writes are visible from here on
    const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);

    auto load_blk = [&](int blk) {
        const int st = blk & 1;
        uint8_t *kd = sm + Lay::STAGE + st * Lay::STAGE_BYTES;
        uint8_t *vd = kd + CBD * 16384;
        const int j0 = klo + 128 * blk;
        mbar_expect_tx(&bar_full[st], 2 * CBD * 16384);
        for (int cb = 0; cb < CBD; ++cb) {
            tma_load_3d(kd + cb * 16384, &maps.k, &bar_full[st], cb * 64, j0, (int)unit);
            tma_load_3d(vd + cb * 16384, &maps.v, &bar_full[st], cb * 64, j0, (int)unit);
        }
    };
    const uint32_t id_u = idesc_bf16(128, DF, 0, 0);
    const uint32_t id_ds = idesc_bf16(128, D, 1, 1);
    const uint32_t id_dz = idesc_bf16(128, 16, 1, 0);
    uint32_t ph_ds = 0;

    if (warp == LS_ROWS / 32) {
        // ============================ the issuing warp ============================
        if (tid == LS_ROWS) {
            uint32_t ph_full[2] = {0, 0}, pe_phi = 0;
            // U of block blk = K_blk Wf into TMEM half blk & 1
            auto issue_u = [&](int blk) {
                const int st = blk & 1;
                if (!mbar_wait(&bar_full[st], ph_full[st], P.status)) s_abort = 1;
                ph_full[st] ^= 1;
                tc_fence_after();
                const uint32_t ka = sb + Lay::STAGE + st * Lay::STAGE_BYTES;
                for (int k = 0; k < D; k += 16)
                    mma_ss(tmem + TM_U + 128 * st, sdesc(ka + (k / 64) * 16384 + (k % 64) * 2, 16, 1024),
                           sdesc(sb + Lay::WF + (k / 64) * (DF * 128) + (k % 64) * 2, 16, 1024), id_u, k > 0);
                mma_commit(&bar_u[st]);
            };
            mbar_expect_tx(&bar_wf, CBD * DF * 128);
            for (int cb = 0; cb < CBD; ++cb) tma_load_2d(sm + Lay::WF + cb * DF * 128, &maps.wft, &bar_wf, cb * 64, 0);
            if (nblk > 0) load_blk(0);
            if (nblk > 1) load_blk(1);
            if (nblk > 0) {
                uint32_t ph0 = 0;
                if (!mbar_wait(&bar_wf, ph0, P.status)) s_abort = 1;
                issue_u(0);
            }
            if (nblk > 1) issue_u(1);
            for (int blk = 0; blk < nblk && !*(volatile int *)&s_abort; ++blk) {
                const int st = blk & 1;
                // the block's features are in shared memory (and the rows are done with its U and K)
                if (!mbar_wait(&rdy_phi, pe_phi, P.status)) s_abort = 1;
                pe_phi ^= 1;
                tc_fence_after();
                const uint32_t va = sb + Lay::STAGE + st * Lay::STAGE_BYTES + CBD * 16384;
                for (int kk = 0; kk < 128; kk += 16) {
                    const uint64_t a = sdesc(sb + Lay::PHI + kk * 128, 16384, 1024);
                    const uint32_t acc = (blk > 0 || kk > 0) ? 1u : 0u;
                    mma_ss(tmem + TM_DS, a, sdesc(va + kk * 128, 16384, 1024), id_ds, acc);
                    mma_ss(tmem + TM_DZ, a, sdesc(sb + Lay::ONES + (kk / 64) * 2048 + (kk % 64) * 2, 16, 1024), id_dz, acc);
                }
                mma_commit(&bar_ds);
                // a full block of table rows leaves straight from the feature buffer
                const int j0 = klo + 128 * blk;
                const bool full = min(khi, fhi) - j0 >= 128;
                if (full) {
                    for (int cb = 0; cb < CBF; ++cb)
                        tma_store_3d(&maps.phik, sm + Lay::PHI + cb * 16384, cb * 64, j0, (int)unit);
                    tma_store_commit();
                }
                // this stage is free once dS has read its V: block blk + 2 comes in; the
                // feature buffer is free once dS, dz and the store have read it
                if (!mbar_wait(&bar_ds, ph_ds, P.status)) s_abort = 1;
                ph_ds ^= 1;
                if (blk + 2 < nblk) load_blk(blk + 2);
                if (full) tma_store_wait_read();
                mbar_arrive(&phi_free);
                // U of block blk + 2 into the TMEM half the rows are done with (block blk's):
                // it is ready long before the rows get there
                if (blk + 2 < nblk) issue_u(blk + 2);
            }
            tma_store_wait_all();
        }
        __syncwarp();
    } else {
        // ============================== the row warps ==============================
        constexpr int DFH = DF / LS_PARTS, CH8 = CBD * 8 / LS_PARTS;   // features per part; 16-byte K chunks per part
        uint32_t ph_u[2] = {0, 0}, ph_kf[2] = {0, 0}, ph_pf = 0;
        const int r = tid & 127, part = tid >> 7;   // key row of the block; which part of it
        // kept-slot index of this thread's key, one block ahead
        auto slot_of = [&](int blk) {
            const int jj = klo + 128 * blk + r;
            return blk < nblk && jj < khi ? __ldg(P.kslot + unit * dm.N + jj) : -1;
        };
        int kslot_next = slot_of(0);
        for (int blk = 0; blk < nblk; ++blk) {
            const int st = blk & 1;
            const int j = klo + 128 * blk + r;
            uint8_t *kd = sm + Lay::STAGE + st * Lay::STAGE_BYTES;
            const bool in_range = j < khi;
            const int kslot = kslot_next;
            kslot_next = slot_of(blk + 1);
            // ||k||^2 over my part of the dimensions, once the block's K has arrived
            bool bad = !mbar_wait(&bar_full[st], ph_kf[st], P.status);
            ph_kf[st] ^= 1;
            float kn2 = 0.f;
#pragma unroll
            for (int q = 0; q < CH8; ++q) {
                const int c = part * CH8 + q;   // 16-byte chunk of the row, 8 per 64-column block
                const uint4 pk = *reinterpret_cast<const uint4 *>(kd + (c / 8) * 16384 + sw128(r, c % 8));
                const uint32_t w4[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                for (int h2 = 0; h2 < 4; ++h2) {
                    const float a0 = __uint_as_float(w4[h2] << 16), a1 = __uint_as_float(w4[h2] & 0xffff0000u);
                    kn2 = fmaf(a0, a0, fmaf(a1, a1, kn2));
                }
            }
            bad |= !mbar_wait(&bar_u[st], ph_u[st], P.status);
            ph_u[st] ^= 1;
            tc_fence_after();
            // my part of the features: exponentials against my part's maximum, in registers
            float u[DFH];
#pragma unroll
            for (int c0 = 0; c0 < DFH; c0 += 16)
                tmem_ld16(tlane + TM_U + 128 * st + part * DFH + c0, *reinterpret_cast<float(*)[16]>(u + c0));
            tmem_ld_wait();
            float mu = -INFINITY, s2 = 0.f;
#pragma unroll
            for (int i = 0; i < DFH; ++i) mu = fmaxf(mu, u[i] * LOG2E);
#pragma unroll
            for (int i = 0; i < DFH; ++i) {
                u[i] = exp2_mufu(fmaf(u[i], LOG2E, -mu));
                s2 = fmaf(u[i], u[i], s2);
            }
            xch[part][r][0] = mu;
            xch[part][r][1] = s2;
            xch[part][r][2] = kn2;
            tc_fence_before();
            if (named_sync_or(1, LS_ROWS, bad || *(volatile int *)&s_abort)) break;
            float sc;
            {
                // the parts' statistics, combined in part order on every part
                float M = xch[0][r][0];
#pragma unroll
                for (int p = 1; p < LS_PARTS; ++p) M = fmaxf(M, xch[p][r][0]);
                float ss = 0.f, kk = 0.f;
#pragma unroll
                for (int p = 0; p < LS_PARTS; ++p) {
                    ss += xch[p][r][1] * exp2_mufu(2.f * (xch[p][r][0] - M));
                    kk += xch[p][r][2];
                }
                sc = sqrtf(kk) * rsqrtf(ss) * exp2_mufu(mu - M);
            }
            // the previous block's dS / dz MMAs and table store are done with the feature buffer
            if (blk > 0) {
                bad = !mbar_wait(&phi_free, ph_pf, P.status);
                ph_pf ^= 1;
            }
            const bool slotted = kslot >= 0;
            const int KP = dm.T_max * dm.lam;
            uint16_t *krow = slotted ? P.phk + (unit * KP + kslot) * DF : nullptr;
            const bool folded = j < fhi && !slotted;
            // keys that stay in the window to the end (the last segment's tail) go to the
            // table from here; every other row of the table is copied from the block below
            const bool tail = in_range && j >= fhi;
            uint16_t *grow = P.phik + (unit * dm.N + (in_range ? j : 0)) * DF;
#pragma unroll
            for (int q = 0; q < DFH; q += 8) {
                const int f0 = part * DFH + q;
                uint32_t w4[4];
#pragma unroll
                for (int h2 = 0; h2 < 4; ++h2) w4[h2] = pack_bf16(sc * u[q + 2 * h2], sc * u[q + 2 * h2 + 1]);
                const uint4 val = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                const uint4 zero = make_uint4(0, 0, 0, 0);
                if (tail) *reinterpret_cast<uint4 *>(grow + f0) = slotted ? zero : val;
                if (slotted) *reinterpret_cast<uint4 *>(krow + f0) = val;   // kept: unmasked features
                *reinterpret_cast<uint4 *>(sm + Lay::PHI + (f0 / 64) * 16384 + sw128(r, (f0 % 64) / 8)) = folded ? val : zero;
            }
            fence_async_smem();
            mbar_arrive(&rdy_phi);
            if (bad) *(volatile int *)&s_abort = 1;
            const int j0 = klo + 128 * blk;
            const int nrow = max(0, min(128, min(khi, fhi) - j0));
            if (nrow > 0 && nrow < 128) {
                // a partial block: rows below fhi hold exactly the table's values (phi, or zero
                // for slotted keys); each warp stores two 256-byte rows per instruction
                if (named_sync_or(1, LS_ROWS, *(volatile int *)&s_abort)) break;
                constexpr int CH = DF / 8;   // 16-byte chunks per row
                uint16_t *gbase = P.phik + (unit * dm.N + j0) * DF;
                for (int e = tid; e < nrow * CH; e += LS_ROWS) {
                    const int row = e / CH, ch = e % CH;
                    const uint4 x = *reinterpret_cast<const uint4 *>(sm + Lay::PHI + (ch / 8) * 16384 + sw128(row, ch % 8));
                    *reinterpret_cast<uint4 *>(gbase + (size_t)row * DF + ch * 8) = x;
                }
                named_sync_or(1, LS_ROWS, false);   // the copy's reads end before the buffer is rewritten
            }
        }
        // dS / dz of this segment: row r, my part of the columns (the last block's MMAs)
        if (nblk > 0 && !*(volatile int *)&s_abort) {
            if (!mbar_wait(&bar_ds, (uint32_t)((nblk - 1) & 1), P.status)) s_abort = 1;
            tc_fence_after();
        }
        float *out = P.dS + (unit * (P.sp.nseg + 1) + s) * (size_t)(DF * D);
        for (int c0 = part * (D / LS_PARTS); c0 < (part + 1) * (D / LS_PARTS); c0 += 16) {
            float v[16];
            tmem_ld16(tlane + TM_DS + c0, v);
            tmem_ld_wait();
            if (r < DF) {
#pragma unroll
                for (int i = 0; i < 16; i += 4)
                    *reinterpret_cast<float4 *>(out + (size_t)r * D + c0 + i) =
                        nblk > 0 ? make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        const float zacc = tmem_ld1(tlane + TM_DZ);
        tmem_ld_wait();
        if (r < DF && part == 0) P.dz[(unit * (P.sp.nseg + 1) + s) * DF + r] = nblk > 0 ? zacc : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t launch_linstate_tc(const Dims &dm, const SegPlan &sp, const uint16_t *k, const uint16_t *v,
                               const uint16_t *wft, const int32_t *kslot, uint16_t *phik, uint16_t *phk, float *dS,
                               float *dz, int32_t *status, cudaStream_t s)
{
    KTimer tm("features_linstate", s);
    LinTCMaps m;
    const int D = dm.d, DF = dm.df;
    const uint64_t units = (uint64_t)dm.B * dm.Hkv;
    uint64_t dk[3] = {(uint64_t)D, (uint64_t)dm.N, units}, sk[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * dm.N};
    uint32_t box[3] = {64, 128, 1};
    bool ok = make_tma_map(&m.k, k, 3, dk, sk, box, true) && make_tma_map(&m.v, v, 3, dk, sk, box, true);
    uint64_t dw[2] = {(uint64_t)D, (uint64_t)DF}, sw[1] = {(uint64_t)D * 2};
    uint32_t boxw[2] = {64, (uint32_t)DF};
    ok = ok && make_tma_map(&m.wft, wft, 2, dw, sw, boxw, true);
    uint64_t dp[3] = {(uint64_t)DF, (uint64_t)dm.N, units}, sp2[2] = {(uint64_t)DF * 2, (uint64_t)DF * 2 * dm.N};
    ok = ok && make_tma_map(&m.phik, phik, 3, dp, sp2, box, true);
    if (!ok) return cudaErrorInvalidValue;
    LinTCParams p{dm, sp, kslot, phik, phk, dS, dz, status};
    dim3 grid(sp.nseg, dm.Hkv, dm.B);
    cudaError_t e;
#define STILL_LIN(DD, FF)                                                                                     \
    {                                                                                                         \
        const size_t smem = LinLayout<DD, FF>::TOTAL + 1024;                                                  \
        e = cudaFuncSetAttribute(linstate_tc_kernel<DD, FF>, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                                 (int)smem);                                                                  \
        if (e != cudaSuccess) return e;                                                                       \
        e = launch_kernel(linstate_tc_kernel<DD, FF>, grid, dim3(LS_THREADS), smem, s, m, p);              \
        if (e != cudaSuccess) return e;                                                                    \
    }
    if (D == 64 && DF == 64) STILL_LIN(64, 64)
    else if (D == 64) STILL_LIN(64, 128)
    else if (DF == 64) STILL_LIN(128, 64)
    else STILL_LIN(128, 128)
#undef STILL_LIN
    return cudaGetLastError();
}

}  // namespace still
