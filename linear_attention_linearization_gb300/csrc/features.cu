// Set-up pass of the prefill: the bf16 copy of Wf^T, [d_f, d] (the B operand
// of the tensor-core NP-Map, "STILL: Content-Aware Intra-Layer Hybrid
// Attention for Efficient LLM Linearization", section "NP-Map:
// Norm-Preserving Feature Map"), and the workspace pieces that must start
// empty: the status word, the per-key slot map (-1: in no budget slot) and the
// kept-token tables (zero rows stand for slots not yet filled).
#include "common.cuh"

namespace still {

__global__ void __launch_bounds__(256) prep_kernel(const float *__restrict__ Wf, int d, int df,
                                                   uint16_t *__restrict__ wft, int32_t *status, int32_t *kslot,
                                                   size_t nkslot, uint4 *kept, size_t nkept16)
{
    grid_dep_sync();
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, nt = (size_t)gridDim.x * blockDim.x;
    if (tid == 0) *status = 0;
    for (size_t i = tid; i < nkslot / 4; i += nt) reinterpret_cast<int4 *>(kslot)[i] = make_int4(-1, -1, -1, -1);
    for (size_t i = nkslot / 4 * 4 + tid; i < nkslot; i += nt) kslot[i] = -1;
    for (size_t i = tid; i < nkept16; i += nt) kept[i] = make_uint4(0, 0, 0, 0);
    for (size_t i = tid; i < (size_t)d * df; i += nt) {
        const int f = (int)(i / d), e = (int)(i % d);
        wft[i] = f2bf(Wf[(size_t)e * df + f]);
    }
}

cudaError_t launch_prep(const Dims &dm, const float *Wf, uint16_t *wft, int32_t *status, int32_t *kslot, void *kept,
                        size_t kept_bytes, cudaStream_t s)
{
    KTimer tm("prep", s);
    return launch_kernel(prep_kernel, dim3(152), dim3(256), 0, s, Wf, dm.d, dm.df, wft, status, kslot,
                         (size_t)dm.B * dm.Hkv * dm.N, reinterpret_cast<uint4 *>(kept), kept_bytes / 16);
}

}  // namespace still
