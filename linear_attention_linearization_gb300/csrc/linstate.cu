// Exclusive scan of the per-segment linear-state sums (linstate_tc.cu): the
// state each segment of the chunk-parallel prefill starts from, and slot nseg
// the state after all N tokens ("STILL: Content-Aware Intra-Layer Hybrid
// Attention for Efficient LLM Linearization", section "Content-Aware Routing
// with Fixed Budget": unkept tokens accumulate into the recurrent state).
#include "common.cuh"

namespace still {

// Exclusive scan of dS / dz over the segments of each (sequence, kv head);
// slot nseg receives the total.
__global__ void scan_kernel(float *__restrict__ dS, float *__restrict__ dz, int nseg, int nel_s, int nel_z)
{
    grid_dep_sync();
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
    for (int s0 = 0; s0 < nseg; s0 += 32) {
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = s0 + i < nseg ? p[(size_t)(s0 + i) * stride] : 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if (s0 + i < nseg) p[(size_t)(s0 + i) * stride] = run;
            run += x[i];
        }
    }
    p[nseg * stride] = run;
}

cudaError_t launch_scan(const Dims &dm, const SegPlan &sp, float *dS, float *dz, cudaStream_t s)
{
    KTimer tm("scan", s);
    const int nel_s = dm.df * dm.d, nel_z = dm.df;
    dim3 grid((nel_s + nel_z + 255) / 256, dm.B * dm.Hkv);
    const cudaError_t e = launch_kernel(scan_kernel, grid, dim3(256), 0, s, dS, dz, sp.nseg, nel_s, nel_z);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace still
