// bf16 copy of Wf^T, [d_f, d]: the B operand of the tensor-core NP-Map
// ("STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", section "NP-Map: Norm-Preserving Feature Map").
#include "common.cuh"

namespace still {

__global__ void wft_kernel(const float *__restrict__ Wf, int d, int df, uint16_t *__restrict__ wft)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d * df; i += gridDim.x * blockDim.x) {
        const int f = i / d, e = i % d;
        wft[i] = f2bf(Wf[e * df + f]);
    }
}

cudaError_t launch_wft(const Dims &dm, const float *Wf, uint16_t *wft, cudaStream_t s)
{
    KTimer tm("wf_transpose", s);
    wft_kernel<<<16, 256, 0, s>>>(Wf, dm.d, dm.df, wft);
    return cudaGetLastError();
}

}  // namespace still
