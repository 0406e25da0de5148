// still_prefill_noalloc: the prefill with its scratch memory in a fixed,
// library-owned device array instead of caller-provided or call-allocated
// workspace.
//
// Who needs this: callers that may not allocate device memory while they
// run -- a plug-in inside an inference engine whose execution step must not
// allocate (the engine plans all memory up front), code that must not risk
// the implicit synchronisation or out-of-memory failure of an allocation in a
// latency-critical path, or a host program without access to an allocator.
// They still pass their own inputs and outputs; only the scratch is fixed.
//
// The array is STILL_NOALLOC_SCRATCH_BYTES (16 MiB).  Every GPU on which the
// library's device code is loaded holds it until the process exits, and every
// call on that GPU shares it.
#include <cstdio>
#include <mutex>

#include "common.cuh"

#define STILL_NOALLOC_SCRATCH_BYTES (16u << 20)

static __device__ __align__(256) unsigned char still_noalloc_scratch[STILL_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device

// Device address of the scratch array on the current device, looked up once
// per device (the host-side name of the array is not a device address).
still_status scratch_on_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return STILL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, still_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            fprintf(stderr, "libstill: cudaGetSymbolAddress of the scratch array failed: %s\n",
                    cudaGetErrorString(e));
            return STILL_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return STILL_OK;
}
}  // namespace

extern "C" {

size_t still_prefill_noalloc_max_bytes(void) { return STILL_NOALLOC_SCRATCH_BYTES; }

still_status still_prefill_noalloc(const still_shape *shape, const still_bf16 *q, const still_bf16 *k,
                                   const still_bf16 *v, const float *Wf, int W, int C, int m, int T_max,
                                   still_bf16 *out, int32_t *sel_idx, const still_decode_state *export_state,
                                   still_stream_t stream)
{
    // sizes or a budget still_prefill refuses are refused with the same status
    const still_status chk = still::check_prefill_sizes(shape, W, C, m, T_max);
    if (chk != STILL_OK) return chk;
    const size_t need = still_prefill_workspace_size(shape, W, C, m, T_max);
    if (need > STILL_NOALLOC_SCRATCH_BYTES) {
        fprintf(stderr,
                "libstill: still_prefill_noalloc needs %zu bytes of scratch for this size, more than its fixed "
                "%u-byte array; use still_prefill with a workspace instead\n",
                need, STILL_NOALLOC_SCRATCH_BYTES);
        return STILL_ERR_WORKSPACE;
    }
    void *scratch = nullptr;
    still_status st = scratch_on_current_device(&scratch);
    if (st != STILL_OK) return st;
    // still_prefill clears the parts of its workspace that must start at zero
    // (status word, slot flags, kept-token tables) on the stream before use,
    // so whatever an earlier call left in the array does not matter.
    return still_prefill(shape, q, k, v, Wf, W, C, m, T_max, out, sel_idx, scratch, STILL_NOALLOC_SCRATCH_BYTES,
                         export_state, stream);
}

}  // extern "C"
