// Chunked linear-attention state of the prefill.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", section "Content-Aware Routing with Fixed Budget": tokens
// that are not kept are accumulated into the linear-attention recurrent state.
//
// Segment s of a (sequence, kv head) owns the keys that leave the window
// while its query tiles run: [s*L - W, (s+1)*L - W) clipped to [0, N - W).
// This kernel forms, per segment, dS_s = sum phi(k_j) v_j^T and dz_s =
// sum phi(k_j) over those keys from the feature table (whose rows of slotted
// keys are zero).  An exclusive scan over segments then gives the state each
// segment starts from, and slot nseg the state after all N tokens.
#include "common.cuh"

namespace still {

template <int D, int DF>
__global__ void __launch_bounds__(256) linstate_kernel(const uint16_t *__restrict__ phik,
                                                       const uint16_t *__restrict__ v, Dims dm, SegPlan sp,
                                                       float *__restrict__ dS, float *__restrict__ dz)
{
    constexpr int PER = DF * D / 256;   // state elements per thread
    constexpr int RSTEP = 256 / D;      // state rows between a thread's elements
    __shared__ float ph[32][DF];
    __shared__ float vs[32][D];
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const size_t ug = (size_t)b * dm.Hkv + g;
    const int lo = max(0, s * sp.L - dm.W);
    const int hi = min((s + 1) * sp.L, dm.N) - dm.W;
    const int col = tid % D, row0 = tid / D;
    float acc[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) acc[r] = 0.f;
    float zacc = 0.f;
    for (int kb = lo; kb < hi; kb += 32) {
        const int nk = min(32, hi - kb);
        for (int e = tid; e < nk * DF; e += 256) ph[e / DF][e % DF] = bf2f(phik[(ug * dm.N + kb) * DF + e]);
        for (int e = tid; e < nk * D; e += 256) vs[e / D][e % D] = bf2f(v[(ug * dm.N + kb) * D + e]);
        __syncthreads();
        for (int kk = 0; kk < nk; ++kk) {
            const float vv = vs[kk][col];
#pragma unroll
            for (int r = 0; r < PER; ++r) acc[r] = fmaf(ph[kk][row0 + RSTEP * r], vv, acc[r]);
            if (tid < DF) zacc += ph[kk][tid];
        }
        __syncthreads();
    }
    float *out = dS + (ug * (sp.nseg + 1) + s) * (size_t)(DF * D);
#pragma unroll
    for (int r = 0; r < PER; ++r) out[(size_t)(row0 + RSTEP * r) * D + col] = acc[r];
    if (tid < DF) dz[(ug * (sp.nseg + 1) + s) * DF + tid] = zacc;
}

// Exclusive scan of dS / dz over the segments of each (sequence, kv head);
// slot nseg receives the total.
__global__ void scan_kernel(float *__restrict__ dS, float *__restrict__ dz, int nseg, int nel_s, int nel_z)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    const size_t ug = blockIdx.y;
    float *p;
    size_t stride;
    if (e < nel_s) {
        p = dS + ug * (nseg + 1) * (size_t)nel_s + e;
        stride = nel_s;
    } else if (e < nel_s + nel_z) {
        p = dz + ug * (nseg + 1) * (size_t)nel_z + (e - nel_s);
        stride = nel_z;
    } else {
        return;
    }
    float run = 0.f;
    for (int s = 0; s < nseg; ++s) {
        const float x = p[s * stride];
        p[s * stride] = run;
        run += x;
    }
    p[nseg * stride] = run;
}

cudaError_t launch_linstate(const Dims &dm, const SegPlan &sp, const uint16_t *phik, const uint16_t *v, float *dS,
                            float *dz, cudaStream_t s)
{
    {
        KTimer tm("linstate", s);
        dim3 grid(sp.nseg, dm.Hkv, dm.B);
        if (dm.d == 64 && dm.df == 64) linstate_kernel<64, 64><<<grid, 256, 0, s>>>(phik, v, dm, sp, dS, dz);
        else if (dm.d == 64) linstate_kernel<64, 128><<<grid, 256, 0, s>>>(phik, v, dm, sp, dS, dz);
        else if (dm.df == 64) linstate_kernel<128, 64><<<grid, 256, 0, s>>>(phik, v, dm, sp, dS, dz);
        else linstate_kernel<128, 128><<<grid, 256, 0, s>>>(phik, v, dm, sp, dS, dz);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    KTimer tm("scan", s);
    const int nel_s = dm.df * dm.d, nel_z = dm.df;
    dim3 grid((nel_s + nel_z + 255) / 256, dm.B * dm.Hkv);
    scan_kernel<<<grid, 256, 0, s>>>(dS, dz, sp.nseg, nel_s, nel_z);
    return cudaGetLastError();
}

}  // namespace still
