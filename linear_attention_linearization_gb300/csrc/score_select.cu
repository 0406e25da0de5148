// Self-Saliency score, top-lambda chunk selection and the standalone NP-Map.
//
// Score: "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", section "Self-Saliency Score: Predicting Future Utility from
// Local Context" -- the KL sensitivity between the window distribution with
// the token's own key (a^diag) and without it (a^nodiag), in the closed form
// -log(1 - p_t + 1e-6).  Selection: section "Delayed Chunk-Level Selection for
// Unified Training-Inference Parallelism" -- each completed chunk keeps its
// top-lambda tokens.  NP-Map: section "NP-Map: Norm-Preserving Feature Map".
#include "common.cuh"

namespace still {

// ---------------------------------------------------------------------------
// Score.  One CTA = 64 tokens of one (sequence, kv head); each warp owns 8
// tokens and walks the G query heads of the group so that the group mean needs
// no atomics.  Lane i of the warp scores keys t - i, t - i - 32, ... and keeps
// an online (max, off-diagonal mass, self mass) triple that the warp merges.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) score_kernel(const uint16_t *__restrict__ q,
                                                    const uint16_t *__restrict__ k, Dims dm,
                                                    float *__restrict__ scores, int diag)
{
    grid_dep_sync();
    const int g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float qs[8][D];
    const float inv = rsqrtf((float)D);
    const uint16_t *kb = k + (size_t)(b * dm.Hkv + g) * dm.N * D;
    for (int tt = warp; tt < 64; tt += 8) {
        const int t = blockIdx.x * 64 + tt;
        if (t >= dm.N) break;
        const int n = min(t + 1, dm.W);
        float acc = 0.f;
        for (int hh = 0; hh < dm.G; ++hh) {
            const int h = g * dm.G + hh;
            const uint16_t *qr = q + ((size_t)(b * dm.Hq + h) * dm.N + t) * D;
            __syncwarp();
            for (int e = lane; e < D; e += 32) qs[warp][e] = bf2f(qr[e]) * inv;
            __syncwarp();
            float ml = -INFINITY, tl = 0.f, sl = 0.f;
            for (int i = lane; i < n; i += 32) {
                const float s = dot_bf16_row<D>(kb + (size_t)(t - i) * D, qs[warp]);
                if (s > ml) {
                    const float c = expf(ml - s);
                    tl *= c;
                    sl *= c;
                    ml = s;
                }
                const float w = expf(s - ml);
                if (i == 0) sl += w;
                else tl += w;
            }
            const float M = warp_max(ml);
            const float f = (ml == -INFINITY) ? 0.f : expf(ml - M);
            const float oth = warp_sum(tl * f);
            const float self = warp_sum(sl * f);
            acc += diag ? self / (oth + self) : saliency_from_stats(oth, self);
        }
        if (lane == 0) scores[(size_t)(b * dm.Hkv + g) * dm.N + t] = acc / dm.G;
    }
}

cudaError_t launch_score(const Dims &dm, const uint16_t *q, const uint16_t *k, float *scores, cudaStream_t s, int diag)
{
    KTimer tm("score", s);
    dim3 grid((dm.N + 63) / 64, dm.Hkv, dm.B);
    const cudaError_t e = launch_kernel(dm.d == 64 ? score_kernel<64> : score_kernel<128>, grid, dim3(256), 0, s, q, k,
                                        dm, scores, diag);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Select.  One warp per (sequence, kv head, chunk c < T_max).  lambda rounds of
// a warp-wide arg-max under outranks(); winners are then written in ascending
// position by a ballot compaction.  The unfinished tail chunk (when < T_max)
// is ranked too: its current top-lambda goes to `fsel` (the internal table of
// tokens kept out of the linear state) but not to the public sel_idx.  `kslot`
// maps each such token to its row c*lambda + r of that table, and the token's
// K and V rows are copied to the same row of the kept tables.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) select_kernel(const float *__restrict__ scores, Dims dm,
                                                    int32_t *__restrict__ sel_idx, int32_t *__restrict__ fsel,
                                                    int32_t *__restrict__ kslot, const uint16_t *__restrict__ k,
                                                    const uint16_t *__restrict__ v, uint16_t *__restrict__ kk,
                                                    uint16_t *__restrict__ vk)
{
    grid_dep_sync();
    extern __shared__ float sel_smem[];
    float *sc = sel_smem;
    int *kidx = reinterpret_cast<int *>(sc + dm.C);            // chunk offsets of the kept tokens, in order
    uint8_t *taken = reinterpret_cast<uint8_t *>(kidx + dm.lam);
    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x;
    const size_t row = ((size_t)(b * dm.Hkv + g) * dm.T_max + c) * dm.lam;
    const int base = c * dm.C;
    const int cnt = min(dm.C, dm.N - base);
    const bool complete = cnt == dm.C;
    if (cnt <= 0) {
        for (int r = lane; r < dm.lam; r += 32) {
            if (sel_idx) sel_idx[row + r] = -1;
            if (fsel) fsel[row + r] = -1;
        }
        return;
    }
    const float *sg = scores + (size_t)(b * dm.Hkv + g) * dm.N + base;
    for (int i = lane; i < cnt; i += 32) {
        sc[i] = sg[i];
        taken[i] = 0;
    }
    __syncwarp();
    const int keep = min(dm.lam, cnt);
    for (int r = 0; r < keep; ++r) {
        int bi = -1;
        float bs = 0.f;
        for (int i = lane; i < cnt; i += 32) {
            if (taken[i]) continue;
            if (bi < 0 || outranks(i, sc[i], bi, bs)) {
                bi = i;
                bs = sc[i];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            if (oi >= 0 && (bi < 0 || outranks(oi, os, bi, bs))) {
                bi = oi;
                bs = os;
            }
        }
        if (lane == 0) taken[bi] = 1;
        __syncwarp();
    }
    int outn = 0;
    for (int i0 = 0; i0 < cnt; i0 += 32) {
        const int i = i0 + lane;
        const bool f = i < cnt && taken[i];
        const unsigned mask = __ballot_sync(0xffffffffu, f);
        if (f) {
            const int p = outn + __popc(mask & ((1u << lane) - 1u));
            kidx[p] = i;
            if (fsel) fsel[row + p] = base + i;
            if (sel_idx) sel_idx[row + p] = complete ? base + i : -1;
            if (kslot) kslot[(size_t)(b * dm.Hkv + g) * dm.N + base + i] = c * dm.lam + p;
        }
        outn += __popc(mask);
    }
    for (int r = outn + lane; r < dm.lam; r += 32) {
        if (fsel) fsel[row + r] = -1;
        if (sel_idx) sel_idx[row + r] = -1;
    }
    if (!complete && sel_idx)
        for (int r = lane; r < outn; r += 32) sel_idx[row + r] = -1;
    // K and V rows of the kept tokens into the kept tables (row c*lambda + r):
    // (token, 16-byte word) pairs spread over the lanes, every load issued
    // before the stores
    if (kk) {
        __syncwarp();
        const size_t ug = (size_t)b * dm.Hkv + g;
        const int words = dm.d / 8;   // 16-byte words per row
        const int total = outn * words;
        for (int e0 = 0; e0 < total; e0 += 128) {
            uint4 kv[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * 32 + lane;
                if (e < total) {
                    const size_t j = (size_t)(base + kidx[e / words]);
                    kv[u][0] = reinterpret_cast<const uint4 *>(k + (ug * dm.N + j) * dm.d)[e % words];
                    kv[u][1] = reinterpret_cast<const uint4 *>(v + (ug * dm.N + j) * dm.d)[e % words];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u * 32 + lane;
                if (e < total) {
                    const size_t dst = (row + (size_t)(e / words)) * dm.d;
                    reinterpret_cast<uint4 *>(kk + dst)[e % words] = kv[u][0];
                    reinterpret_cast<uint4 *>(vk + dst)[e % words] = kv[u][1];
                }
            }
        }
    }
}

cudaError_t launch_select(const Dims &dm, const float *scores, int32_t *sel_idx, int32_t *fsel, int32_t *kslot,
                          cudaStream_t s, const uint16_t *k, const uint16_t *v, uint16_t *kk, uint16_t *vk)
{
    if (dm.lam <= 0) return cudaSuccess;
    KTimer tm("select", s);
    const size_t smem = (size_t)dm.C * (sizeof(float) + 1) + sizeof(int) * dm.lam;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(dm.T_max, dm.Hkv, dm.B);
    const cudaError_t e = launch_kernel(select_kernel, grid, dim3(32), smem, s, scores, dm, sel_idx, fsel, kslot, k, v, kk, vk);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Standalone NP-Map: one warp per row.
// ---------------------------------------------------------------------------
template <int D, int DF>
__global__ void __launch_bounds__(256) npmap_kernel(const uint16_t *__restrict__ x, long long rows,
                                                    const float *__restrict__ Wf, float *__restrict__ phi)
{
    grid_dep_sync();
    __shared__ float xs[8][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (long long r = (long long)blockIdx.x * 8 + warp; r < rows; r += (long long)gridDim.x * 8) {
        __syncwarp();
        for (int e = lane; e < D; e += 32) xs[warp][e] = bf2f(x[r * D + e]);
        __syncwarp();
        warp_npmap<D, DF>(xs[warp], Wf, phi + r * DF, lane);
    }
}

cudaError_t launch_npmap(const uint16_t *x, long long rows, int d, const float *Wf, int df, float *phi,
                         cudaStream_t s)
{
    KTimer tm("npmap", s);
    long long blocks = (rows + 7) / 8;
    int grid = (int)(blocks < 152 * 16 ? blocks : 152 * 16);
    auto kern = d == 64 ? (df == 64 ? npmap_kernel<64, 64> : npmap_kernel<64, 128>)
                        : (df == 64 ? npmap_kernel<128, 64> : npmap_kernel<128, 128>);
    const cudaError_t e = launch_kernel(kern, grid, dim3(256), 0, s, x, rows, Wf, phi);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace still
