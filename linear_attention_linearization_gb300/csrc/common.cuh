// Shared device helpers and the internal launch interface of libstill.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "still.h"

namespace still {

// Sizes and routing parameters of one call, resolved on the host.
struct Dims {
    int B, Hq, Hkv, N, d, df, G;
    int W, C, m, T_max, lam;
    int n_full;   // completed chunks: N / C
    int n_sel;    // chunks that run a selection: min(T_max, ceil(N / C))
    int tail;     // the unfinished last chunk when it is < T_max, else -1
};

// Segment plan of the chunk-parallel prefill: CTA s of a (sequence, kv head)
// walks the query tiles of [begin[s], begin[s+1]) in order, starting from the
// linear state of the keys that left the window before its first tile.
// Segments are cut so that their attention work (not their token counts) is
// even: tiles late in the sequence see more kept keys.
constexpr int MAX_SEGMENTS = 152;
struct SegPlan {
    int T;      // query tokens per tile
    int nseg;   // segments per (sequence, kv head)
    int begin[MAX_SEGMENTS + 1];   // first token of each segment (multiples of T); begin[nseg] = N
};

// ---- programmatic dependent launch ---------------------------------------------
// Every kernel of the library is launched so that it may be scheduled while
// the previous kernel on the stream is still finishing; before it touches
// global memory it waits for that kernel's completion (and the visibility of
// its writes), then lets the next kernel be scheduled in turn.
__device__ __forceinline__ void grid_dep_sync()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---- bf16 ------------------------------------------------------------------
__device__ __forceinline__ float bf2f(uint16_t x) { return __uint_as_float(((uint32_t)x) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// ---- warp reductions ---------------------------------------------------------
__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Ranking of the top-lambda selection: higher score first, exact ties to the
// lower position.
__device__ __forceinline__ bool outranks(long long i, float si, long long j, float sj)
{
    return si > sj || (si == sj && i < j);
}

__device__ __forceinline__ void set_status(int32_t *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// Bounded device-side waits: clock cycles a wait may spin before it gives up
// (about 2 s at the GB300's 2.07 GHz), setting STILL_ERR_TIMEOUT.
constexpr long long WAIT_LIMIT_CYCLES = 4000000000LL;

// Limit of the consumer-side waits (row warps waiting for a copy or an MMA) of
// the tensor-core prefill kernels: WAIT_LIMIT_CYCLES unless a test lowered it
// with still_debug_set_wait_limit (api.cu).
long long consumer_wait_limit();

// Self-Saliency score from the window's softmax statistics: oth = sum of
// e^{s-M} over the window without the token itself, self = e^{s_tt - M}.
// -log(1 - p + eps) is taken through log1p while p is small, so that small
// scores keep full relative precision, and through the off-diagonal mass
// otherwise, so that 1 - p never comes from a cancelling difference.
__device__ __forceinline__ float saliency_from_stats(float oth, float self)
{
    const float tot = oth + self;
    const float p = self / tot;
    if (p < 0.5f) return -log1pf(1e-6f - p);
    return -logf(oth / tot + 1e-6f);
}

// ---- 2^x on the MUFU unit: the PTX ex2.approx instruction, results below
// 2^-126 flushed to zero (the weights it forms are rounded to bf16 or summed
// in fp32, where such values do not count)
__device__ __forceinline__ float exp2_mufu(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- NP-Map of one row, by one warp -------------------------------------------
// x: the row in shared memory (fp32, D values); Wf: global fp32 [D, DF].
// Writes phi (DF values) to `phi` (shared or global).
template <int D, int DF>
__device__ __forceinline__ void warp_npmap(const float *x, const float *__restrict__ Wf, float *phi, int lane)
{
    constexpr int PJ = DF / 32;
    float l[PJ];
#pragma unroll
    for (int r = 0; r < PJ; ++r) l[r] = 0.f;
    for (int i = 0; i < D; ++i) {
        float xi = x[i];
#pragma unroll
        for (int r = 0; r < PJ; ++r) l[r] = fmaf(xi, __ldg(Wf + i * DF + lane + 32 * r), l[r]);
    }
    float nx = 0.f;
    for (int e = lane; e < D; e += 32) nx = fmaf(x[e], x[e], nx);
    nx = sqrtf(warp_sum(nx));
    float mx = l[0];
#pragma unroll
    for (int r = 1; r < PJ; ++r) mx = fmaxf(mx, l[r]);
    mx = warp_max(mx);
    float su = 0.f;
#pragma unroll
    for (int r = 0; r < PJ; ++r) { l[r] = expf(l[r] - mx); su += l[r]; }
    su = warp_sum(su);
    float nu = 0.f;
#pragma unroll
    for (int r = 0; r < PJ; ++r) { l[r] /= su; nu = fmaf(l[r], l[r], nu); }
    nu = sqrtf(warp_sum(nu));
    float sc = nx / nu;
#pragma unroll
    for (int r = 0; r < PJ; ++r) phi[lane + 32 * r] = sc * l[r];
}

// Dot product of a bf16 global row with an fp32 shared row, by one thread.
template <int D>
__device__ __forceinline__ float dot_bf16_row(const uint16_t *__restrict__ row, const float *x)
{
    float s = 0.f;
#pragma unroll 4
    for (int e = 0; e < D; e += 8) {
        uint4 pk = __ldg(reinterpret_cast<const uint4 *>(row + e));
        uint32_t w[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            s = fmaf(__uint_as_float(w[h] << 16), x[e + 2 * h], s);
            s = fmaf(__uint_as_float(w[h] & 0xffff0000u), x[e + 2 * h + 1], s);
        }
    }
    return s;
}

// ---- timing hooks (implemented in api.cu) -----------------------------------
void timing_begin(const char *name, cudaStream_t s);
void timing_end(cudaStream_t s);

struct KTimer {
    cudaStream_t s;
    KTimer(const char *name, cudaStream_t st) : s(st) { timing_begin(name, st); }
    ~KTimer() { timing_end(s); }
};

// The status still_prefill returns for these sizes and routing parameters
// before it looks at any pointer (STILL_OK when they are valid).
still_status check_prefill_sizes(const still_shape *shape, int W, int C, int m, int T_max);

// ---- launchers (one per kernel family) ----------------------------------------
// diag = 1: the mean self probability p_t (the diagonal-attention routing metric)
cudaError_t launch_score(const Dims &dm, const uint16_t *q, const uint16_t *k, float *scores, cudaStream_t s,
                         int diag = 0);
bool score_tc_supported(const Dims &dm);
// The prefill's set-up pass (see prep_kernel), folded into the score kernel.
struct PrepArgs {
    const float *Wf;
    uint16_t *wft;
    int32_t *status, *kslot;
    void *kept;
    size_t kept_bytes;
};
cudaError_t launch_score_tc(const Dims &dm, const uint16_t *q, const uint16_t *k, float *scores, cudaStream_t s,
                            const PrepArgs *prep = nullptr, int diag = 0);
// Routing metrics (routing.cu); metric is a still_metric value.
cudaError_t launch_metric(const Dims &dm, int metric, unsigned long long seed, const uint16_t *q, const uint16_t *k,
                          float *scores, cudaStream_t s);
cudaError_t launch_select(const Dims &dm, const float *scores, int32_t *sel_idx, int32_t *fsel, int32_t *kslot,
                          cudaStream_t s, const uint16_t *k = nullptr, const uint16_t *v = nullptr,
                          uint16_t *kk = nullptr, uint16_t *vk = nullptr);
cudaError_t launch_npmap(const uint16_t *x, long long rows, int d, const float *Wf, int df, float *phi,
                         cudaStream_t s);
cudaError_t launch_prep(const Dims &dm, const float *Wf, uint16_t *wft, int32_t *status, int32_t *kslot, void *kept,
                        size_t kept_bytes, cudaStream_t s);
cudaError_t launch_linstate_tc(const Dims &dm, const SegPlan &sp, const uint16_t *k, const uint16_t *v,
                               const uint16_t *wft, const int32_t *kslot, uint16_t *phik, uint16_t *phk, float *dS,
                               float *dz, int32_t *status, cudaStream_t s);
cudaError_t launch_scan(const Dims &dm, const SegPlan &sp, float *dS, float *dz, cudaStream_t s);
cudaError_t launch_hybrid_general(const Dims &dm, const SegPlan &sp, const uint16_t *q, const uint16_t *k,
                                  const uint16_t *v, const float *Wf, const uint16_t *phik, const uint16_t *phkept,
                                  const int32_t *fsel, const float *dS, const float *dz, uint16_t *out,
                                  int32_t *status, cudaStream_t s, const uint16_t *gate = nullptr);
struct TCBuffers {
    const uint16_t *q, *k, *v, *kk, *vk, *phik, *phk, *wft;
    uint16_t *out;
    const uint16_t *gate;   // nullable: pre-activations of the linear branch's gate, [B, Hq, N, d]
};
bool hybrid_tc_supported(const Dims &dm);
cudaError_t launch_hybrid_tc(const Dims &dm, const SegPlan &sp, const TCBuffers &bf, const int32_t *fsel,
                             const float *dS, const float *dz, int32_t *status, cudaStream_t s);
cudaError_t launch_export(const Dims &dm, const SegPlan &sp, const uint16_t *k, const uint16_t *v,
                          const float *scores, const int32_t *fsel, const float *dS, const float *dz,
                          const still_decode_state &st, cudaStream_t s);
// gate_t (nullable): the gated layer's pre-activations [B, Hq, d] of this step
cudaError_t launch_decode(const Dims &dm, const still_decode_state &st, const uint16_t *q_t,
                          const uint16_t *k_t, const uint16_t *v_t, const float *Wf, uint16_t *out_t,
                          cudaStream_t s, const uint16_t *gate_t = nullptr);
// the decode step runs its staged kernel (the one the gated layer needs) for this state
bool decode_staged(const Dims &dm, const still_decode_state &st);


// ---- backward pass (backward.cu) ----------------------------------------------
struct BwdInputs {
    const uint16_t *q, *k, *v, *dy;
    const float *Wf;
    const int32_t *sel;
    float *dq, *dk, *dv, *dWf;
    int32_t *cidx;   // nullable
    cudaStream_t stream;
};
// byte offsets of the backward pass's workspace pieces
struct BwdLayout {
    size_t kslot, phkk, phkk32, phk, Sp, zp, Rs, rs, g, phq, phq32, phk32, dlq, dlk, rc, rinv, rdelta, rds, rjs, total;
};
BwdLayout bwd_layout(const Dims &dm);
bool backward_supported(const Dims &dm);
cudaError_t launch_backward(const Dims &dm, const BwdInputs &in, void *ws);

}  // namespace still
