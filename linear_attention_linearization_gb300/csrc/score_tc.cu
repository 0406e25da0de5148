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
// band of keys [t0 - Wr, t0 + 32) that holds every window of the tile.  The
// logits stay in TMEM; 8 warps (two per TMEM lane quarter, each owning half of
// the band columns) reduce each row to (max, off-diagonal mass, self mass).
// Tiles are pipelined over up to four shared-memory / TMEM stages: while the
// row warps reduce tile i, the MMA of tile i+1 runs and the loads of the
// following tiles are in flight.
#include "sm100.cuh"
#include "tma_host.cuh"

namespace still {

using namespace sm100;

namespace {
constexpr int SC_MAX_NB = 8;         // band blocks of 32 keys (W <= 225)
constexpr int SC_MAX_STAGES = 4;     // tiles in flight
constexpr size_t SC_SMEM_CAP = 227 * 1024 - 4096;   // dynamic share of the 227 KB per-block limit
}

struct ScoreTCParams {
    Dims dm;
    int Wr, nb;        // band [t0 - Wr, t0 + 32), nb blocks of 32 keys
    int tiles_per_unit, total_tiles;
    int stages;        // tiles in flight (shared-memory and TMEM stages)
    uint32_t stage_bytes, tmem_stride;
    float *scores;
};

struct ScoreTCMaps {
    CUtensorMap q, k;
};

template <int D>
__global__ void __launch_bounds__(256, 1) score_tc_kernel(const __grid_constant__ ScoreTCMaps maps, ScoreTCParams P)
{
    constexpr int CBD = D / 64;
    constexpr uint32_t QB = CBD * 16384;          // Q tile bytes
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t bar_full[SC_MAX_STAGES], bar_mma[SC_MAX_STAGES];
    __shared__ uint32_t tmem_base;
    __shared__ float xch[2][128][3];
    __shared__ float hsc[4][32];
    __shared__ int s_abort;

    const Dims &dm = P.dm;
    const int NS = P.stages;
    const uint32_t STB = P.stage_bytes, KBB = P.nb * 4096;   // bytes of a stage, of one K column block
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane, hh = r / 32, tt = r % 32;
    const int ncols = P.nb * 32, hcols = ncols / 2;
    const int W = dm.W;
    const float l2s = 1.4426950408889634f * rsqrtf((float)D);   // log2(e) / sqrt(d)

    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) { mbar_init(&bar_full[i], 1); mbar_init(&bar_mma[i], 1); }
        fence_barrier_init();
        s_abort = 0;
    }
    // padding rows of absent heads: zero in every stage buffer, never written again
    for (int st = 0; st < NS; ++st)
        for (int i = tid; i < (int)(QB / 16); i += 256) {
            const int row = (i * 16 % 16384) / 128;
            if (row >= dm.G * 32) reinterpret_cast<uint4 *>(sm + st * STB)[i] = make_uint4(0, 0, 0, 0);
        }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16);

    const int first = blockIdx.x, step = gridDim.x;
    const int my_tiles = first < P.total_tiles ? (P.total_tiles - first + step - 1) / step : 0;
    const uint32_t idesc = idesc_bf16(128, ncols, 0, 0);
    const uint64_t d0 = sdesc(sb, 16, 1024);

    auto tile_coords = [&](int i, int &unit, int &t0) {
        const int tile = first + i * step;
        unit = tile / P.tiles_per_unit;
        t0 = (tile % P.tiles_per_unit) * 32;
    };
    auto issue_load = [&](int i) {
        int unit, t0;
        tile_coords(i, unit, t0);
        const int st = i % NS;
        uint8_t *qd = sm + st * STB;
        uint8_t *kd = qd + QB;
        const int b = unit / dm.Hkv, g = unit % dm.Hkv;
        mbar_expect_tx(&bar_full[st], dm.G * CBD * 4096 + P.nb * CBD * 4096);
        for (int h = 0; h < dm.G; ++h)
            for (int cb = 0; cb < CBD; ++cb)
                tma_load_3d(qd + cb * 16384 + h * 4096, &maps.q, &bar_full[st], cb * 64, t0, b * dm.Hq + g * dm.G + h);
        for (int kb = 0; kb < P.nb; ++kb)
            for (int cb = 0; cb < CBD; ++cb)
                tma_load_3d(kd + cb * KBB + kb * 4096, &maps.k, &bar_full[st], cb * 64, t0 - P.Wr + 32 * kb, unit);
    };
    uint32_t ph_full = 0, ph_mma = 0;   // one parity bit per stage
    auto issue_mma = [&](int i) {
        const int st = i % NS;
        if (!mbar_wait(&bar_full[st], (ph_full >> st) & 1u, nullptr)) { s_abort = 1; return; }
        ph_full ^= 1u << st;
        tc_fence_after();
        const uint64_t qa = d0 + ((st * STB) >> 4), ka = qa + (QB >> 4);
#pragma unroll
        for (int k = 0; k < D; k += 16)
            mma_ss(tmem + st * P.tmem_stride, qa + (((k / 64) * 16384 + (k % 64) * 2) >> 4),
                   ka + (((k / 64) * KBB + (k % 64) * 2) >> 4), idesc, k > 0);
        mma_commit(&bar_mma[st]);
    };

    if (tid == 0) {
        for (int i = 0; i < NS && i < my_tiles; ++i) issue_load(i);
        if (my_tiles > 0) issue_mma(0);
    }
    for (int i = 0; i < my_tiles; ++i) {
        const int st = i % NS;
        int unit, t0;
        tile_coords(i, unit, t0);
        if (tid == 0 && i + 1 < my_tiles && !s_abort) issue_mma(i + 1);
        if (!mbar_wait(&bar_mma[st], (ph_mma >> st) & 1u, nullptr)) s_abort = 1;
        ph_mma ^= 1u << st;
        tc_fence_after();

        // row statistics over this thread's half of the band columns
        const int t = t0 + tt;
        const int band_lo = t0 - P.Wr;
        const int lo = max(max(t - W + 1, 0) - band_lo, 0), hi = t - band_lo;   // window columns [lo, hi]
        const int self_c = t - band_lo;
        const int c_beg = half * hcols;
        float m = -INFINITY, oth = 0.f, slf = 0.f;
        for (int c0 = 0; c0 < hcols; c0 += 16) {
            float v[16];
            tmem_ld16(tlane + st * P.tmem_stride + c_beg + c0, v);
            tmem_ld_wait();
            float bm = -INFINITY;
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int c = c_beg + c0 + x;
                v[x] = (c >= lo && c <= hi) ? v[x] * l2s : -INFINITY;
                bm = fmaxf(bm, v[x]);
            }
            if (bm > m) {
                const float sc = exp2f(m - bm);
                oth *= sc;
                slf *= sc;
                m = bm;
            }
            if (m != -INFINITY) {
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float e = exp2_mufu(v[x] - m);
                    if (c_beg + c0 + x == self_c) slf += e;
                    else oth += e;
                }
            }
        }
        xch[half][r][0] = m;
        xch[half][r][1] = oth;
        xch[half][r][2] = slf;
        tc_fence_before();
        __syncthreads();
        if (s_abort) break;
        if (half == 0) {
            const float m1 = xch[1][r][0];
            const float M = fmaxf(m, m1);
            float o = 0.f, sl = 0.f;
            if (M != -INFINITY) {
                const float f0 = m == -INFINITY ? 0.f : exp2f(m - M), f1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
                o = oth * f0 + xch[1][r][1] * f1;
                sl = slf * f0 + xch[1][r][2] * f1;
            }
            hsc[hh][tt] = (hh < dm.G && t < dm.N) ? saliency_from_stats(o, sl) : 0.f;
        }
        __syncthreads();
        if (tid < 32 && t0 + tid < dm.N) {
            float a = 0.f;
            for (int h = 0; h < dm.G; ++h) a += hsc[h][tid];
            P.scores[(size_t)unit * dm.N + t0 + tid] = a / dm.G;
        }
        // stage st is free again: load tile i + NS into it
        if (tid == 0 && i + NS < my_tiles && !s_abort) issue_load(i + NS);
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

cudaError_t launch_score_tc(const Dims &dm, const uint16_t *q, const uint16_t *k, float *scores, cudaStream_t s)
{
    KTimer tm("score", s);
    ScoreTCMaps m;
    const int D = dm.d;
    uint64_t dq[3] = {(uint64_t)D, (uint64_t)dm.N, (uint64_t)dm.B * dm.Hq};
    uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * dm.N};
    uint32_t box[3] = {64, 32, 1};
    bool ok = make_tma_map(&m.q, q, 3, dq, sq, box, true);
    uint64_t dk[3] = {(uint64_t)D, (uint64_t)dm.N, (uint64_t)dm.B * dm.Hkv};
    ok = ok && make_tma_map(&m.k, k, 3, dk, sq, box, true);
    if (!ok) return cudaErrorInvalidValue;
    ScoreTCParams p;
    p.dm = dm;
    p.Wr = (dm.W - 1 + 31) / 32 * 32;
    p.nb = (p.Wr + 32) / 32;
    p.tiles_per_unit = (dm.N + 31) / 32;
    p.total_tiles = p.tiles_per_unit * dm.B * dm.Hkv;
    p.scores = scores;
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
    cudaError_t e;
    if (D == 64) {
        e = cudaFuncSetAttribute(score_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        score_tc_kernel<64><<<grid, 256, smem, s>>>(m, p);
    } else {
        e = cudaFuncSetAttribute(score_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        score_tc_kernel<128><<<grid, 256, smem, s>>>(m, p);
    }
    return cudaGetLastError();
}

}  // namespace still
