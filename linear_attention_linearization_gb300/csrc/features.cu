// Kept-token tables of the prefill and the bf16 copy of Wf^T.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", section "Content-Aware Routing with Fixed Budget" (kept
// tokens stay out of the linear state) and section "NP-Map: Norm-Preserving
// Feature Map" (phi).
//
//   kept tables, row c*lambda + r for the r-th kept token of chunk c (the
//   order of the selection table): K, V and the unmasked phi of that token,
//   zero rows where the selection has no token.  The kept tokens of all
//   chunks before chunk c are the contiguous prefix [0, c*lambda).
//   wft      = bf16(Wf^T), [d_f, d]: the B operand of the tensor-core NP-Map.
#include "common.cuh"

namespace still {

template <int D, int DF>
__global__ void __launch_bounds__(256) kept_kernel(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                                                   const float *__restrict__ Wf, const int32_t *__restrict__ fsel,
                                                   Dims dm, uint16_t *__restrict__ kk, uint16_t *__restrict__ vk,
                                                   uint16_t *__restrict__ phk)
{
    __shared__ float xs[8][D];
    __shared__ float ph[8][DF];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t ug = blockIdx.y;
    const int KP = dm.T_max * dm.lam;
    for (int e = blockIdx.x * 8 + warp; e < KP; e += gridDim.x * 8) {
        const int j = fsel[ug * KP + e];
        uint16_t *kd = kk + (ug * KP + e) * D;
        uint16_t *vd = vk + (ug * KP + e) * D;
        uint16_t *pd = phk + (ug * KP + e) * DF;
        if (j < 0) {
            for (int x = lane; x < D; x += 32) { kd[x] = 0; vd[x] = 0; }
            for (int x = lane; x < DF; x += 32) pd[x] = 0;
            continue;
        }
        const uint16_t *kr = k + (ug * dm.N + j) * D;
        const uint16_t *vr = v + (ug * dm.N + j) * D;
        __syncwarp();
        for (int x = lane; x < D; x += 32) {
            kd[x] = kr[x];
            vd[x] = vr[x];
            xs[warp][x] = bf2f(kr[x]);
        }
        __syncwarp();
        warp_npmap<D, DF>(xs[warp], Wf, ph[warp], lane);
        __syncwarp();
        for (int x = lane; x < DF; x += 32) pd[x] = f2bf(ph[warp][x]);
    }
}

__global__ void wft_kernel(const float *__restrict__ Wf, int d, int df, uint16_t *__restrict__ wft)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d * df; i += gridDim.x * blockDim.x) {
        const int f = i / d, e = i % d;
        wft[i] = f2bf(Wf[e * df + f]);
    }
}

cudaError_t launch_kept(const Dims &dm, const uint16_t *k, const uint16_t *v, const float *Wf, const int32_t *fsel,
                        uint16_t *kk, uint16_t *vk, uint16_t *phk, uint16_t *wft, cudaStream_t s)
{
    const int units = dm.B * dm.Hkv;
    if (dm.lam > 0) {
        KTimer tm("kept_tables", s);
        const int KP = dm.T_max * dm.lam;
        dim3 grid((KP + 7) / 8 < 64 ? (KP + 7) / 8 : 64, units);
#define STILL_KEPT(DD, FF) kept_kernel<DD, FF><<<grid, 256, 0, s>>>(k, v, Wf, fsel, dm, kk, vk, phk)
        if (dm.d == 64 && dm.df == 64) STILL_KEPT(64, 64);
        else if (dm.d == 64) STILL_KEPT(64, 128);
        else if (dm.df == 64) STILL_KEPT(128, 64);
        else STILL_KEPT(128, 128);
#undef STILL_KEPT
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    KTimer tm("wf_transpose", s);
    wft_kernel<<<16, 256, 0, s>>>(Wf, dm.d, dm.df, wft);
    return cudaGetLastError();
}

}  // namespace still
