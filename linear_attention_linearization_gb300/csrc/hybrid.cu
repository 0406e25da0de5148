// Fused hybrid attention of the prefill: softmax over the window and the kept
// tokens, the linear branch through the running state, one normalisation.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", sections "Content-Aware Routing with Fixed Budget" and
// "Delayed Chunk-Level Selection for Unified Training-Inference Parallelism":
//   SA(t) = {t-W < j <= t} U {j kept by chunk(j) < chunk(t), j <= t-W}
//   LA(t) = {j <= t-W} minus SA(t)
//   y_t   = (sum_SA e^{s-c} v + sum_LA (phi(q).phi(k)) v) /
//           (sum_SA e^{s-c} + sum_LA phi(q).phi(k)),   c = max_SA s.
//
// General-shape kernel on CUDA cores: it serves the shapes outside the
// tensor-core kernel's envelope (see hybrid_tc.cu).  One CTA walks the query
// tiles of one segment of one (sequence, kv head) in order.  Its running state
// S_run, z_run holds every key j < t0 - W that sits in no budget slot (t0 =
// first token of the tile).  For a query t of the tile the linear keys are
//   S_run  +  unslotted keys e0 <= j <= t-W                     (e0 = t0 - W)
//          +  slotted keys of t's own chunk with j <= t-W,
// because a kept token is a softmax key only for queries of later chunks.
// The feature table has zero rows for slotted keys, so the second term needs
// no test; the third reads the unmasked features of the kept table.
#include "common.cuh"

namespace still {

template <int D, int DF>
__global__ void __launch_bounds__(256) hybrid_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
                                                     const uint16_t *__restrict__ v, const float *__restrict__ Wf,
                                                     const uint16_t *__restrict__ phik, const uint16_t *__restrict__ phkept,
                                                     const int32_t *__restrict__ fsel, const float *__restrict__ dS,
                                                     const float *__restrict__ dz, Dims dm, SegPlan sp,
                                                     uint16_t *__restrict__ out, int32_t *status,
                                                     const uint16_t *__restrict__ gate)
{
    grid_dep_sync();
    constexpr int PD = D / 32;          // output dims per lane
    constexpr int PER = DF * D / 256;   // state elements per thread
    constexpr int RSTEP = 256 / D;
    extern __shared__ float sm[];
    float *Srun = sm;
    float *zrun = Srun + DF * D;
    float *qs = zrun + DF;
    float *pq = qs + 8 * D;
    float *fph = pq + 8 * DF;
    float *fv = fph + sp.T * DF;

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t ug = (size_t)b * dm.Hkv + g;
    const uint16_t *kg = k + ug * dm.N * D;
    const uint16_t *vg = v + ug * dm.N * D;
    const uint16_t *phg = phik + ug * dm.N * DF;
    const uint16_t *phkg = phkept + ug * dm.T_max * dm.lam * DF;
    const int32_t *fs = fsel + ug * dm.T_max * dm.lam;
    const float inv = rsqrtf((float)D);
    const int col = tid % D, row0 = tid / D;

    {
        const float *S0 = dS + (ug * (sp.nseg + 1) + s) * (size_t)(DF * D);
        for (int e = tid; e < DF * D; e += 256) Srun[e] = S0[e];
        const float *z0 = dz + (ug * (sp.nseg + 1) + s) * DF;
        for (int e = tid; e < DF; e += 256) zrun[e] = z0[e];
    }
    __syncthreads();

    const int tbeg = sp.begin[s], tend = sp.begin[s + 1];
    for (int t0 = tbeg; t0 < tend; t0 += sp.T) {
        const int nt = min(sp.T, tend - t0);
        const int e0 = t0 - dm.W;
        for (int rr = warp; rr < nt * dm.G; rr += 8) {
            const int hh = rr / nt, t = t0 + rr % nt, h = g * dm.G + hh;
            const int ct = t / dm.C;
            float *xq = qs + warp * D;
            float *fq = pq + warp * DF;
            const uint16_t *qr = q + ((size_t)(b * dm.Hq + h) * dm.N + t) * D;
            __syncwarp();
            for (int e = lane; e < D; e += 32) xq[e] = bf2f(qr[e]);
            __syncwarp();
            warp_npmap<D, DF>(xq, Wf, fq, lane);
            __syncwarp();

            // softmax keys: window (newest first), then the kept tokens of
            // earlier finished chunks that already left the window
            const int nw = min(t + 1, dm.W);
            const int ng = min(ct, dm.T_max) * dm.lam;
            float M = -INFINITY, l = 0.f, acc[PD];
#pragma unroll
            for (int r = 0; r < PD; ++r) acc[r] = 0.f;
            for (int p0 = 0; p0 < nw + ng; p0 += 32) {
                const int p = p0 + lane;
                int j = -1;
                if (p < nw) {
                    j = t - p;
                } else if (p < nw + ng) {
                    j = fs[p - nw];
                    if (j > t - dm.W) j = -1;
                    if (j >= dm.N) { set_status(status, STILL_ERR_BOUNDS); j = -1; }
                }
                const float sv = j >= 0 ? dot_bf16_row<D>(kg + (size_t)j * D, xq) * inv : -INFINITY;
                const float bm = warp_max(sv);
                const float Mn = fmaxf(M, bm);
                if (Mn == -INFINITY) continue;
                const float sc = expf(M - Mn);
                l *= sc;
#pragma unroll
                for (int r = 0; r < PD; ++r) acc[r] *= sc;
                M = Mn;
                const float pw = j >= 0 ? expf(sv - M) : 0.f;
                l += warp_sum(pw);
                for (int jj = 0; jj < 32; ++jj) {
                    const float pj = __shfl_sync(0xffffffffu, pw, jj);
                    const int jp = __shfl_sync(0xffffffffu, j, jj);
                    if (pj == 0.f) continue;
                    const uint16_t *vr = vg + (size_t)jp * D;
#pragma unroll
                    for (int r = 0; r < PD; ++r) acc[r] = fmaf(pj, bf2f(vr[lane + 32 * r]), acc[r]);
                }
            }

            // linear keys: running state, then the lagged keys of this tile
            // and the slotted keys of t's own chunk
            float la[PD];
#pragma unroll
            for (int r = 0; r < PD; ++r) la[r] = 0.f;
            for (int i = 0; i < DF; ++i) {
                const float f = fq[i];
#pragma unroll
                for (int r = 0; r < PD; ++r) la[r] = fmaf(f, Srun[i * D + lane + 32 * r], la[r]);
            }
            float dl = 0.f;
            for (int i = lane; i < DF; i += 32) dl = fmaf(fq[i], zrun[i], dl);
            dl = warp_sum(dl);
            const int ilo = max(0, e0);
            const int ni = max(0, t - dm.W - ilo + 1);
            const int nx = ct < dm.T_max ? dm.lam : 0;
            for (int p0 = 0; p0 < ni + nx; p0 += 32) {
                const int p = p0 + lane;
                int j = -1;
                const uint16_t *pr = nullptr;
                if (p < ni) {
                    j = ilo + p;
                    pr = phg + (size_t)j * DF;
                } else if (p < ni + nx) {
                    j = fs[ct * dm.lam + (p - ni)];
                    if (j > t - dm.W) j = -1;
                    pr = phkg + (size_t)(ct * dm.lam + (p - ni)) * DF;
                }
                float a = 0.f;
                if (j >= 0)
                    for (int i = 0; i < DF; ++i) a = fmaf(fq[i], bf2f(pr[i]), a);
                dl += warp_sum(a);
                for (int jj = 0; jj < 32; ++jj) {
                    const float aj = __shfl_sync(0xffffffffu, a, jj);
                    const int jp = __shfl_sync(0xffffffffu, j, jj);
                    if (jp < 0) continue;
                    const uint16_t *vr = vg + (size_t)jp * D;
#pragma unroll
                    for (int r = 0; r < PD; ++r) la[r] = fmaf(aj, bf2f(vr[lane + 32 * r]), la[r]);
                }
            }
            const float den = l + dl;
            uint16_t *orow = out + ((size_t)(b * dm.Hq + h) * dm.N + t) * D;
            // the gated layer: sigmoid(gate) on the linear numerator, channel by channel
            const uint16_t *grow = gate ? gate + ((size_t)(b * dm.Hq + h) * dm.N + t) * D : nullptr;
#pragma unroll
            for (int r = 0; r < PD; ++r) {
                const float gch = grow ? 1.f / (1.f + expf(-bf2f(grow[lane + 32 * r]))) : 1.f;
                orow[lane + 32 * r] = f2bf(den != 0.f ? fmaf(gch, la[r], acc[r]) / den : 0.f);
            }
        }
        __syncthreads();

        // keys [e0, t0 + nt - W) leave the window before the next tile
        const int flo = max(0, e0), fhi = t0 + nt - dm.W;
        if (fhi > flo) {
            const int nf = fhi - flo;
            for (int e = tid; e < nf * DF; e += 256) fph[e] = bf2f(phg[(size_t)flo * DF + e]);
            for (int e = tid; e < nf * D; e += 256) fv[e] = bf2f(vg[(size_t)flo * D + e]);
            __syncthreads();
#pragma unroll 4
            for (int r = 0; r < PER; ++r) {
                const int i = row0 + RSTEP * r;
                float a = Srun[i * D + col];
                for (int kk = 0; kk < nf; ++kk) a = fmaf(fph[kk * DF + i], fv[kk * D + col], a);
                Srun[i * D + col] = a;
            }
            if (tid < DF) {
                float a = zrun[tid];
                for (int kk = 0; kk < nf; ++kk) a += fph[kk * DF + tid];
                zrun[tid] = a;
            }
            __syncthreads();
        }
    }
}

template <int D, int DF>
static cudaError_t launch_hybrid_t(const Dims &dm, const SegPlan &sp, const uint16_t *q, const uint16_t *k,
                                   const uint16_t *v, const float *Wf, const uint16_t *phik,
                                   const uint16_t *phkept, const int32_t *fsel, const float *dS, const float *dz,
                                   uint16_t *out, int32_t *status, cudaStream_t s, const uint16_t *gate)
{
    const size_t smem = sizeof(float) * ((size_t)DF * D + DF + 8 * D + 8 * DF + (size_t)sp.T * (DF + D));
    cudaError_t e = cudaFuncSetAttribute(hybrid_kernel<D, DF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(sp.nseg, dm.Hkv, dm.B);
    e = launch_kernel(hybrid_kernel<D, DF>, grid, dim3(256), smem, s, q, k, v, Wf, phik, phkept, fsel, dS, dz, dm, sp,
                      out, status, gate);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_hybrid_general(const Dims &dm, const SegPlan &sp, const uint16_t *q, const uint16_t *k,
                                  const uint16_t *v, const float *Wf, const uint16_t *phik, const uint16_t *phkept,
                                  const int32_t *fsel, const float *dS, const float *dz, uint16_t *out,
                                  int32_t *status, cudaStream_t s, const uint16_t *gate)
{
    KTimer tm(gate ? "hybrid_attn_general_gated" : "hybrid_attn_general", s);
    if (dm.d == 64 && dm.df == 64)
        return launch_hybrid_t<64, 64>(dm, sp, q, k, v, Wf, phik, phkept, fsel, dS, dz, out, status, s, gate);
    if (dm.d == 64)
        return launch_hybrid_t<64, 128>(dm, sp, q, k, v, Wf, phik, phkept, fsel, dS, dz, out, status, s, gate);
    if (dm.df == 64)
        return launch_hybrid_t<128, 64>(dm, sp, q, k, v, Wf, phik, phkept, fsel, dS, dz, out, status, s, gate);
    return launch_hybrid_t<128, 128>(dm, sp, q, k, v, Wf, phik, phkept, fsel, dS, dz, out, status, s, gate);
}

}  // namespace still
