// Routing metrics other than the Self-Saliency Score.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", section "Ablation Studies" (routing metric comparison): the
// fixed-budget chunk selection is run with other per-token scores in place of
// the Self-Saliency Score -- diagonal attention, the q.k dot product, the key
// norm, uniform and random selection.  Each metric gives one fp32 score per
// (sequence, kv head, token); the delayed top-lambda selection is unchanged.
//   diagonal  mean over the G query heads of p_t, the token's own weight in its
//             causal window of W keys (the score kernels, with `diag` set)
//   q.k       mean over the G query heads of q_t . k_t / sqrt(d)
//   key norm  ||k_t||
//   uniform   1 at the lambda evenly spaced offsets floor((r + 1/2) C / lambda)
//             of each chunk, 0 elsewhere
//   random    SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
//             number generators") as a counter-based generator: output number
//             i + 1 of the stream started at `seed`, i = (b Hkv + g) N + t, top
//             24 bits scaled to [0, 1)
#include "common.cuh"

namespace still {

namespace {

__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t i)
{
    uint64_t z = seed + (i + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// 1 when offset i of a chunk of C tokens is one of floor((2r + 1) C / (2 lambda)),
// r < lambda: the smallest r with (2r + 1) C >= 2 lambda i is the only candidate
__device__ __forceinline__ float uniform_pick(int i, int C, int lam)
{
    if (lam >= C) return 1.f;
    if (lam <= 0) return 0.f;
    const long long a = 2ll * lam * i - C;   // need (2r + 1) C >= 2 lambda i, i.e. 2 r C >= a
    long long r = a <= 0 ? 0 : (a + 2ll * C - 1) / (2ll * C);
    return (r < lam && (2 * r + 1) * (long long)C < 2ll * lam * (i + 1)) ? 1.f : 0.f;
}

}  // namespace

// Dot-product metrics: L = D / 8 lanes per token row (16-byte loads), 32 / L
// tokens per row group and U groups per warp pass, every load of a pass issued
// before its arithmetic; 8 warps per CTA walk the rows of one (sequence, kv head).
template <int D>
__global__ void __launch_bounds__(256) metric_dot_kernel(const uint16_t *__restrict__ q,
                                                         const uint16_t *__restrict__ k, Dims dm, int metric,
                                                         float *__restrict__ scores)
{
    grid_dep_sync();
    constexpr int L = D / 8, TPW = 32 / L, U = 4;
    const int g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / L, e8 = lane % L;
    const size_t unit = (size_t)b * dm.Hkv + g;
    const float inv = rsqrtf((float)D);
    const bool norm = metric == STILL_METRIC_KEY_NORM;
    auto dot4 = [](const uint4 &x, const uint4 &y, float acc) {
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc = fmaf(__uint_as_float(xs[j] << 16), __uint_as_float(ys[j] << 16), acc);
            acc = fmaf(__uint_as_float(xs[j] & 0xffff0000u), __uint_as_float(ys[j] & 0xffff0000u), acc);
        }
        return acc;
    };
    for (int t0 = (blockIdx.x * 8 + warp) * TPW * U; t0 < dm.N; t0 += gridDim.x * 8 * TPW * U) {
        uint4 kw[U];
        float acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + u * TPW + sub;
            kw[u] = t < dm.N ? reinterpret_cast<const uint4 *>(k + (unit * dm.N + t) * D)[e8] : make_uint4(0, 0, 0, 0);
            acc[u] = 0.f;
        }
        if (norm) {
#pragma unroll
            for (int u = 0; u < U; ++u) acc[u] = dot4(kw[u], kw[u], 0.f);
        } else {
            for (int h0 = 0; h0 < dm.G; h0 += 2) {
                uint4 qw[U][2];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int t = t0 + u * TPW + sub;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const size_t row = ((size_t)b * dm.Hq + (size_t)g * dm.G + h0 + j) * dm.N + t;
                        qw[u][j] = (t < dm.N && h0 + j < dm.G) ? reinterpret_cast<const uint4 *>(q + row * D)[e8]
                                                                : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) acc[u] = dot4(qw[u][1], kw[u], dot4(qw[u][0], kw[u], acc[u]));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int o = L / 2; o > 0; o >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
            const int t = t0 + u * TPW + sub;
            if (e8 == 0 && t < dm.N) scores[unit * dm.N + t] = norm ? sqrtf(acc[u]) : acc[u] * inv / dm.G;
        }
    }
}

// Position-only metrics: one thread per token.
__global__ void __launch_bounds__(256) metric_pos_kernel(Dims dm, int metric, unsigned long long seed,
                                                         float *__restrict__ scores)
{
    grid_dep_sync();
    const size_t total = (size_t)dm.B * dm.Hkv * dm.N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i % dm.N);
        scores[i] = metric == STILL_METRIC_UNIFORM ? uniform_pick(t % dm.C, dm.C, dm.lam)
                                                   : (float)(splitmix64_at(seed, i) >> 40) * 0x1p-24f;
    }
}

cudaError_t launch_metric(const Dims &dm, int metric, unsigned long long seed, const uint16_t *q, const uint16_t *k,
                          float *scores, cudaStream_t s)
{
    if (metric == STILL_METRIC_SELF_SALIENCY || metric == STILL_METRIC_DIAGONAL) {
        const int diag = metric == STILL_METRIC_DIAGONAL;
        if (score_tc_supported(dm)) return launch_score_tc(dm, q, k, scores, s, nullptr, diag);
        return launch_score(dm, q, k, scores, s, diag);
    }
    KTimer tm("routing_metric", s);
    cudaError_t e;
    if (metric == STILL_METRIC_QK || metric == STILL_METRIC_KEY_NORM) {
        const int tpc = 8 * 4 * (32 / (dm.d / 8));   // tokens per CTA pass
        int bx = (dm.N + tpc - 1) / tpc;
        const int cap = (152 * 8 + dm.B * dm.Hkv - 1) / (dm.B * dm.Hkv);   // about 8 CTAs per SM in all
        if (bx > cap) bx = cap;
        if (bx < 1) bx = 1;
        dim3 grid(bx, dm.Hkv, dm.B);
        e = launch_kernel(dm.d == 64 ? metric_dot_kernel<64> : metric_dot_kernel<128>, grid, dim3(256), 0, s, q, k, dm,
                          metric, scores);
    } else {
        const size_t total = (size_t)dm.B * dm.Hkv * dm.N;
        size_t blocks = (total + 255) / 256;
        if (blocks > 152 * 8) blocks = 152 * 8;
        e = launch_kernel(metric_pos_kernel, dim3((unsigned)blocks), dim3(256), 0, s, dm, metric, seed, scores);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace still
