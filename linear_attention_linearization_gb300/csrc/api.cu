// C ABI of libstill: argument checks, workspace plan, launch order, timing.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace still {

// ---------------------------------------------------------------------------
// kernel timing (host-side record of CUDA event pairs)
// ---------------------------------------------------------------------------
namespace {
struct TimedLaunch {
    std::string name;
    cudaEvent_t a, b;
};
std::mutex g_tm_mu;
bool g_tm_on = false;
std::vector<TimedLaunch> g_tm_open;   // one per stream nesting level
std::vector<TimedLaunch> g_tm_done;
std::vector<cudaEvent_t> g_tm_pool;

cudaEvent_t pool_event()
{
    if (!g_tm_pool.empty()) {
        cudaEvent_t e = g_tm_pool.back();
        g_tm_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

void timing_begin(const char *name, cudaStream_t s)
{
    std::lock_guard<std::mutex> lk(g_tm_mu);
    if (!g_tm_on) return;
    TimedLaunch t{name, pool_event(), pool_event()};
    cudaEventRecord(t.a, s);
    g_tm_open.push_back(t);
}

void timing_end(cudaStream_t s)
{
    std::lock_guard<std::mutex> lk(g_tm_mu);
    if (!g_tm_on || g_tm_open.empty()) return;
    TimedLaunch t = g_tm_open.back();
    g_tm_open.pop_back();
    cudaEventRecord(t.b, s);
    g_tm_done.push_back(t);
}

size_t decode_smem_bytes(const Dims &dm);

namespace {
std::atomic<long long> g_consumer_wait_limit{0};   // 0: WAIT_LIMIT_CYCLES
}

long long consumer_wait_limit()
{
    const long long v = g_consumer_wait_limit.load();
    return v > 0 ? v : WAIT_LIMIT_CYCLES;
}

}  // namespace still

using namespace still;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

still_status check_shape(const still_shape *sh, bool need_n)
{
    if (!sh) return STILL_ERR_INVALID_ARG;
    if (sh->B < 1 || sh->Hq < 1 || sh->Hkv < 1 || (need_n && sh->N < 0)) return STILL_ERR_INVALID_ARG;
    if (sh->Hq % sh->Hkv) return STILL_ERR_INVALID_ARG;
    if (!((sh->d == 64 || sh->d == 128) && (sh->d_f == 64 || sh->d_f == 128))) return STILL_ERR_UNSUPPORTED;
    return STILL_OK;
}

still_status make_dims(const still_shape *sh, int W, int C, int m, int T_max, Dims *dm)
{
    still_status st = check_shape(sh, true);
    if (st != STILL_OK) return st;
    if (W < 0 || C < 1 || T_max < 1 || m < W) return STILL_ERR_INVALID_ARG;
    const int lam = (m - W) / T_max;
    if (W < 1 && lam > 0) return STILL_ERR_INVALID_ARG;
    if (C > 16384) return STILL_ERR_UNSUPPORTED;
    dm->B = sh->B; dm->Hq = sh->Hq; dm->Hkv = sh->Hkv; dm->N = sh->N; dm->d = sh->d; dm->df = sh->d_f;
    dm->G = sh->Hq / sh->Hkv;
    dm->W = W; dm->C = C; dm->m = m; dm->T_max = T_max; dm->lam = lam;
    dm->n_full = sh->N / C;
    const int nch = (sh->N + C - 1) / C;
    dm->n_sel = nch < T_max ? nch : T_max;
    dm->tail = (sh->N % C != 0 && sh->N / C < T_max && lam > 0) ? sh->N / C : -1;
    return STILL_OK;
}

// One CTA per segment of 32-token tiles; segments are sized so that all
// (sequence, kv head, segment) CTAs fit one wave of one CTA per SM.
SegPlan plan_segments(const Dims &dm)
{
    SegPlan sp;
    sp.T = 32;
    const int ntile = (dm.N + sp.T - 1) / sp.T;
    const int units = dm.B * dm.Hkv;
    int target = MAX_SEGMENTS / (units > 0 ? units : 1);
    if (target < 1) target = 1;
    if (target > ntile) target = ntile;
    if (ntile == 0) {
        sp.nseg = 1;
        sp.begin[0] = 0;
        sp.begin[1] = dm.N;
        return sp;
    }
    // work of a tile: a fixed part (NP-Map, epilogues, state update) worth about
    // 600 keys (fitted to measured segment times), plus the softmax keys it
    // attends (window and kept tokens)
    auto cost = [&](int tile) {
        const int ct = tile * sp.T / dm.C;
        return 600.0 + dm.W + (double)(ct < dm.T_max ? ct : dm.T_max) * dm.lam;
    };
    double total = 0.0;
    for (int i = 0; i < ntile; ++i) total += cost(i);
    sp.nseg = target;
    sp.begin[0] = 0;
    double acc = 0.0;
    int s = 1, i = 0;
    for (; i < ntile && s < target; ++i) {
        acc += cost(i);
        // cut after tile i once this segment has its share, leaving a tile for each later one
        if (acc >= total * s / target || ntile - (i + 1) == target - s) sp.begin[s++] = (i + 1) * sp.T;
    }
    sp.nseg = s;
    sp.begin[s] = dm.N;
    return sp;
}

struct WsLayout {
    size_t status, scores, fsel, kslot, phik, kk, vk, phk, wft, dS, dz, total;
    size_t kept_bytes;
};

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(const Dims &dm, const SegPlan &sp)
{
    WsLayout L;
    size_t o = 0;
    const size_t units = (size_t)dm.B * dm.Hkv;
    const size_t KP = (size_t)dm.T_max * dm.lam > 0 ? (size_t)dm.T_max * dm.lam : 1;
    L.status = o; o += al(256);
    L.scores = o; o += al(units * dm.N * 4);
    L.fsel = o; o += al(units * KP * 4);
    L.kslot = o; o += al(units * dm.N * 4);
    L.phik = o; o += al(units * dm.N * (size_t)dm.df * 2);
    L.kk = o; o += al(units * KP * dm.d * 2);
    L.vk = o; o += al(units * KP * dm.d * 2);
    L.phk = o; o += al(units * KP * dm.df * 2);
    L.kept_bytes = o - L.kk;
    L.wft = o; o += al((size_t)dm.df * dm.d * 2);
    L.dS = o; o += al(units * (size_t)(sp.nseg + 1) * dm.df * dm.d * 4);
    L.dz = o; o += al(units * (size_t)(sp.nseg + 1) * dm.df * 4);
    L.total = o;
    return L;
}

still_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return STILL_OK;
    fprintf(stderr, "libstill: CUDA error %s\n", cudaGetErrorString(e));
    return STILL_ERR_CUDA;
}

// With m == 0 (no softmax budget at all) the slot arrays are empty and may be null.
bool state_ok(const still_decode_state *s, int m)
{
    if (!s || !s->S || !s->z || !s->score_ring || !s->t || !s->status || !aligned16(s->S)) return false;
    if (m == 0) return true;
    return s->K && s->V && s->slot_pos && s->slot_cnt && s->slot_score && aligned16(s->K) && aligned16(s->V);
}

}  // namespace

extern "C" {

const char *still_status_string(still_status s)
{
    switch (s) {
    case STILL_OK: return "ok";
    case STILL_ERR_INVALID_ARG: return "invalid argument";
    case STILL_ERR_UNSUPPORTED: return "unsupported shape";
    case STILL_ERR_CUDA: return "CUDA error";
    case STILL_ERR_TIMEOUT: return "device wait timed out";
    case STILL_ERR_BOUNDS: return "index out of bounds";
    case STILL_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

int still_lambda(int W, int m, int T_max)
{
    if (T_max < 1 || W < 0 || m < W) return -1;
    return (m - W) / T_max;
}

still_status still_score(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, int W, float *scores,
                         still_stream_t stream)
{
    still_status st = check_shape(shape, true);
    if (st != STILL_OK) return st;
    if (W < 1) return STILL_ERR_INVALID_ARG;
    if (!q || !k || !scores || !aligned16(q) || !aligned16(k) || !aligned16(scores)) return STILL_ERR_INVALID_ARG;
    if (shape->N == 0) return STILL_OK;
    Dims dm;
    st = make_dims(shape, W, 1, W, 1, &dm);
    if (st != STILL_OK) return st;
    if (score_tc_supported(dm)) return cuda_status(launch_score_tc(dm, q, k, scores, (cudaStream_t)stream));
    return cuda_status(launch_score(dm, q, k, scores, (cudaStream_t)stream));
}

still_status still_select(const still_shape *shape, const float *scores, int W, int C, int m, int T_max,
                          int32_t *sel_idx, still_stream_t stream)
{
    Dims dm;
    still_status st = make_dims(shape, W, C, m, T_max, &dm);
    if (st != STILL_OK) return st;
    if (!scores || !sel_idx || !aligned16(scores) || !aligned16(sel_idx)) return STILL_ERR_INVALID_ARG;
    if (dm.lam == 0) return STILL_OK;
    if (dm.N == 0)
        return cuda_status(cudaMemsetAsync(sel_idx, 0xff, (size_t)dm.B * dm.Hkv * dm.T_max * dm.lam * 4,
                                           (cudaStream_t)stream));
    return cuda_status(launch_select(dm, scores, sel_idx, nullptr, nullptr, (cudaStream_t)stream));
}

still_status still_npmap(const still_bf16 *x, long long rows, int d, const float *Wf, int d_f, float *phi,
                         still_stream_t stream)
{
    if (rows < 0 || !x || !Wf || !phi || !aligned16(x) || !aligned16(Wf) || !aligned16(phi))
        return STILL_ERR_INVALID_ARG;
    if (!((d == 64 || d == 128) && (d_f == 64 || d_f == 128))) return STILL_ERR_UNSUPPORTED;
    if (rows == 0) return STILL_OK;
    return cuda_status(launch_npmap(x, rows, d, Wf, d_f, phi, (cudaStream_t)stream));
}

}  // extern "C"

namespace still {
still_status check_prefill_sizes(const still_shape *shape, int W, int C, int m, int T_max)
{
    Dims dm;
    return make_dims(shape, W, C, m, T_max, &dm);
}
}  // namespace still

extern "C" {

size_t still_prefill_workspace_size(const still_shape *shape, int W, int C, int m, int T_max)
{
    Dims dm;
    if (make_dims(shape, W, C, m, T_max, &dm) != STILL_OK) return 0;
    return ws_layout(dm, plan_segments(dm)).total;
}

}  // extern "C"

namespace {

// The prefill, its chunks ranked by `metric`.  The Self-Saliency path runs the
// set-up pass inside the tensor-core score kernel; other metrics run it as a
// kernel of its own before their scores.
still_status prefill_impl(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, const still_bf16 *v,
                          const float *Wf, int W, int C, int m, int T_max, int metric, unsigned long long seed,
                          still_bf16 *out, int32_t *sel_idx, void *workspace, size_t workspace_bytes,
                          const still_decode_state *export_state, still_stream_t stream,
                          const still_bf16 *gate = nullptr)
{
    Dims dm;
    still_status st = make_dims(shape, W, C, m, T_max, &dm);
    if (st != STILL_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (sel_idx && !aligned16(sel_idx)) return STILL_ERR_INVALID_ARG;
    if (dm.N == 0) {
        // nothing to attend; the selection table is all "no token"
        if (sel_idx && dm.lam > 0)
            return cuda_status(cudaMemsetAsync(sel_idx, 0xff, (size_t)dm.B * dm.Hkv * dm.T_max * dm.lam * 4, s));
        return STILL_OK;
    }
    if (!q || !k || !v || !Wf || !out) return STILL_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(Wf) || !aligned16(out) ||
        (workspace && !aligned16(workspace)))
        return STILL_ERR_INVALID_ARG;
    if (export_state && !state_ok(export_state, dm.m)) return STILL_ERR_INVALID_ARG;
    const SegPlan sp = plan_segments(dm);
    const WsLayout L = ws_layout(dm, sp);
    if (workspace && workspace_bytes < L.total) return STILL_ERR_WORKSPACE;
    void *ws = workspace;
    if (!ws) {
        cudaError_t e = cudaMallocAsync(&ws, L.total, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    char *base = (char *)ws;
    int32_t *status = (int32_t *)(base + L.status);
    float *scores = (float *)(base + L.scores);
    int32_t *fsel = (int32_t *)(base + L.fsel);
    int32_t *kslot = (int32_t *)(base + L.kslot);
    uint16_t *phik = (uint16_t *)(base + L.phik);
    uint16_t *kk = (uint16_t *)(base + L.kk);
    uint16_t *vk = (uint16_t *)(base + L.vk);
    uint16_t *phk = (uint16_t *)(base + L.phk);
    uint16_t *wft = (uint16_t *)(base + L.wft);
    float *dS = (float *)(base + L.dS);
    float *dz = (float *)(base + L.dz);
    // the status word starts at zero before any kernel of this call can write it
    cudaError_t e0 = cudaMemsetAsync(status, 0, 4, s);
    if (e0 != cudaSuccess) {
        if (!workspace) cudaFreeAsync(ws, s);
        return cuda_status(e0);
    }
    const bool tc = hybrid_tc_supported(dm);
    // the set-up pass rides on the tensor-core score kernel when that one runs
    const bool fused_prep = dm.lam > 0 && score_tc_supported(dm) && metric == STILL_METRIC_SELF_SALIENCY;
    cudaError_t e = cudaSuccess;
    if (fused_prep) {
        const PrepArgs pa{Wf, wft, status, kslot, kk, L.kept_bytes};
        e = launch_score_tc(dm, q, k, scores, s, &pa);
    } else {
        e = launch_prep(dm, Wf, wft, status, kslot, kk, L.kept_bytes, s);
        if (e == cudaSuccess && dm.lam > 0) e = launch_metric(dm, metric, seed, q, k, scores, s);
    }
    if (e == cudaSuccess && dm.lam > 0) e = launch_select(dm, scores, sel_idx, fsel, kslot, s, k, v, kk, vk);
    if (e == cudaSuccess) e = launch_linstate_tc(dm, sp, k, v, wft, kslot, phik, phk, dS, dz, status, s);
    if (e == cudaSuccess) e = launch_scan(dm, sp, dS, dz, s);
    if (e == cudaSuccess) {
        if (tc) {
            TCBuffers bf{q, k, v, kk, vk, phik, phk, wft, out, gate};
            e = launch_hybrid_tc(dm, sp, bf, fsel, dS, dz, status, s);
        } else {
            e = launch_hybrid_general(dm, sp, q, k, v, Wf, phik, phk, fsel, dS, dz, out, status, s, gate);
        }
    }
    if (e == cudaSuccess && export_state) e = launch_export(dm, sp, k, v, scores, fsel, dS, dz, *export_state, s);
    if (!workspace) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    return cuda_status(e);
}

bool metric_ok(int metric) { return metric >= STILL_METRIC_SELF_SALIENCY && metric <= STILL_METRIC_RANDOM; }

}  // namespace

extern "C" {

still_status still_prefill(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, const still_bf16 *v,
                           const float *Wf, int W, int C, int m, int T_max, still_bf16 *out, int32_t *sel_idx,
                           void *workspace, size_t workspace_bytes, const still_decode_state *export_state,
                           still_stream_t stream)
{
    return prefill_impl(shape, q, k, v, Wf, W, C, m, T_max, STILL_METRIC_SELF_SALIENCY, 0, out, sel_idx, workspace,
                        workspace_bytes, export_state, stream);
}

still_status still_prefill_routed(const still_shape *shape, const still_bf16 *q, const still_bf16 *k,
                                  const still_bf16 *v, const float *Wf, int W, int C, int m, int T_max,
                                  still_metric metric, uint64_t seed, still_bf16 *out, int32_t *sel_idx,
                                  void *workspace, size_t workspace_bytes, still_stream_t stream)
{
    if (!metric_ok(metric)) return STILL_ERR_INVALID_ARG;
    return prefill_impl(shape, q, k, v, Wf, W, C, m, T_max, metric, seed, out, sel_idx, workspace, workspace_bytes,
                        nullptr, stream);
}

still_status still_prefill_gated(const still_shape *shape, const still_bf16 *q, const still_bf16 *k,
                                 const still_bf16 *v, const still_bf16 *gate, const float *Wf, int W, int C, int m,
                                 int T_max, still_bf16 *out, int32_t *sel_idx, void *workspace,
                                 size_t workspace_bytes, const still_decode_state *export_state,
                                 still_stream_t stream)
{
    if (shape && shape->N > 0 && (!gate || !aligned16(gate))) return STILL_ERR_INVALID_ARG;
    return prefill_impl(shape, q, k, v, Wf, W, C, m, T_max, STILL_METRIC_SELF_SALIENCY, 0, out, sel_idx, workspace,
                        workspace_bytes, export_state, stream, gate);
}

size_t still_backward_workspace_size(const still_shape *shape, int W, int C, int m, int T_max)
{
    Dims dm;
    if (make_dims(shape, W, C, m, T_max, &dm) != STILL_OK) return 0;
    return bwd_layout(dm).total;
}

still_status still_backward(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, const still_bf16 *v,
                            const float *Wf, int W, int C, int m, int T_max, const int32_t *sel_idx,
                            const still_bf16 *dout, float *dq, float *dk, float *dv, float *dWf, int32_t *cmax_idx,
                            void *workspace, size_t workspace_bytes, still_stream_t stream)
{
    Dims dm;
    still_status st = make_dims(shape, W, C, m, T_max, &dm);
    if (st != STILL_OK) return st;
    if (!backward_supported(dm)) return STILL_ERR_UNSUPPORTED;
    if (!dWf || !aligned16(dWf) || !Wf || !aligned16(Wf)) return STILL_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (dm.N == 0) return cuda_status(cudaMemsetAsync(dWf, 0, (size_t)dm.d * dm.df * 4, s));
    const void *ptrs[] = {q, k, v, dout, dq, dk, dv};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return STILL_ERR_INVALID_ARG;
    if ((dm.lam > 0 && (!sel_idx || !aligned16(sel_idx))) || (cmax_idx && !aligned16(cmax_idx)) ||
        (workspace && !aligned16(workspace)))
        return STILL_ERR_INVALID_ARG;
    const BwdLayout L = bwd_layout(dm);
    if (workspace && workspace_bytes < L.total) return STILL_ERR_WORKSPACE;
    void *ws = workspace;
    if (!ws) {
        cudaError_t e = cudaMallocAsync(&ws, L.total, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    BwdInputs in{(const uint16_t *)q, (const uint16_t *)k, (const uint16_t *)v, (const uint16_t *)dout, Wf, sel_idx,
                 dq, dk, dv, dWf, cmax_idx, s};
    cudaError_t e = launch_backward(dm, in, ws);
    if (!workspace) {
        const cudaError_t ef = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = ef;
    }
    return cuda_status(e);
}

still_status still_score_metric(const still_shape *shape, const still_bf16 *q, const still_bf16 *k, int W, int C,
                                int m, int T_max, still_metric metric, uint64_t seed, float *scores,
                                still_stream_t stream)
{
    if (!metric_ok(metric)) return STILL_ERR_INVALID_ARG;
    const bool windowed = metric == STILL_METRIC_SELF_SALIENCY || metric == STILL_METRIC_DIAGONAL;
    const bool needs_q = windowed || metric == STILL_METRIC_QK;
    const bool needs_k = needs_q || metric == STILL_METRIC_KEY_NORM;
    Dims dm;
    const still_status st = make_dims(shape, W, C, m, T_max, &dm);   // the routing parameters, as still_select
    if (st != STILL_OK) return st;
    if (windowed && W < 1) return STILL_ERR_INVALID_ARG;
    if (!scores || !aligned16(scores)) return STILL_ERR_INVALID_ARG;
    if ((needs_q && (!q || !aligned16(q))) || (needs_k && (!k || !aligned16(k)))) return STILL_ERR_INVALID_ARG;
    if (dm.N == 0) return STILL_OK;
    return cuda_status(launch_metric(dm, metric, seed, q, k, scores, (cudaStream_t)stream));
}

still_status still_decode_state_init(const still_shape *shape, const still_decode_state *state, int W, int C, int m,
                                     int T_max, still_stream_t stream)
{
    still_shape sh = *shape;
    sh.N = 0;
    Dims dm;
    still_status st = make_dims(&sh, W, C, m, T_max, &dm);
    if (st != STILL_OK) return st;
    if (!state_ok(state, dm.m)) return STILL_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t units = (size_t)dm.B * dm.Hkv;
    cudaError_t e = cudaMemsetAsync(state->K, 0, units * m * dm.d * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->V, 0, units * m * dm.d * 2, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->slot_pos, 0xff, units * m * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->slot_cnt, 0, units * m * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->slot_score, 0, units * m * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->S, 0, units * dm.df * dm.d * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->z, 0, units * dm.df * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->score_ring, 0, units * C * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->t, 0, units * 8, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(state->status, 0, 4, s);
    return cuda_status(e);
}

still_status still_decode_step(const still_shape *shape, const still_decode_state *state, const still_bf16 *q_t,
                               const still_bf16 *k_t, const still_bf16 *v_t, const float *Wf, int W, int C, int m,
                               int T_max, still_bf16 *out_t, still_stream_t stream)
{
    still_shape sh = *shape;
    sh.N = 0;
    Dims dm;
    still_status st = make_dims(&sh, W, C, m, T_max, &dm);
    if (st != STILL_OK) return st;
    if (!state_ok(state, dm.m) || !q_t || !k_t || !v_t || !Wf || !out_t) return STILL_ERR_INVALID_ARG;
    if (!aligned16(q_t) || !aligned16(k_t) || !aligned16(v_t) || !aligned16(Wf) || !aligned16(out_t))
        return STILL_ERR_INVALID_ARG;
    if (dm.G > 8) return STILL_ERR_UNSUPPORTED;
    if (decode_smem_bytes(dm) > 200 * 1024) return STILL_ERR_UNSUPPORTED;
    return cuda_status(launch_decode(dm, *state, q_t, k_t, v_t, Wf, out_t, (cudaStream_t)stream));
}

still_status still_decode_step_gated(const still_shape *shape, const still_decode_state *state, const still_bf16 *q_t,
                                     const still_bf16 *k_t, const still_bf16 *v_t, const still_bf16 *gate_t,
                                     const float *Wf, int W, int C, int m, int T_max, still_bf16 *out_t,
                                     still_stream_t stream)
{
    if (!shape) return STILL_ERR_INVALID_ARG;
    still_shape sh = *shape;
    sh.N = 0;
    Dims dm;
    still_status st = make_dims(&sh, W, C, m, T_max, &dm);
    if (st != STILL_OK) return st;
    if (!gate_t || !aligned16(gate_t)) return STILL_ERR_INVALID_ARG;
    if (!state_ok(state, dm.m) || !q_t || !k_t || !v_t || !Wf || !out_t) return STILL_ERR_INVALID_ARG;
    if (!aligned16(q_t) || !aligned16(k_t) || !aligned16(v_t) || !aligned16(Wf) || !aligned16(out_t))
        return STILL_ERR_INVALID_ARG;
    if (dm.G > 8 || !decode_staged(dm, *state)) return STILL_ERR_UNSUPPORTED;
    return cuda_status(launch_decode(dm, *state, q_t, k_t, v_t, Wf, out_t, (cudaStream_t)stream, gate_t));
}

still_status still_read_status(const int32_t *status_word, still_stream_t stream, int32_t *host_value)
{
    if (!status_word || !host_value) return STILL_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(host_value, status_word, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    return cuda_status(e);
}

void still_debug_set_wait_limit(long long cycles) { g_consumer_wait_limit.store(cycles > 0 ? cycles : 0); }

void still_timing_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_tm_mu);
    g_tm_on = on != 0;
}

int still_timing_read(still_kernel_time *out, int max)
{
    std::lock_guard<std::mutex> lk(g_tm_mu);
    std::vector<still_kernel_time> agg;
    for (auto &t : g_tm_done) {
        cudaEventSynchronize(t.b);
        float ms = 0.f;
        cudaEventElapsedTime(&ms, t.a, t.b);
        still_kernel_time *hit = nullptr;
        for (auto &a : agg)
            if (t.name == a.name) hit = &a;
        if (!hit) {
            still_kernel_time k{};
            strncpy(k.name, t.name.c_str(), sizeof(k.name) - 1);
            agg.push_back(k);
            hit = &agg.back();
        }
        hit->launches += 1;
        hit->ms += ms;
        g_tm_pool.push_back(t.a);
        g_tm_pool.push_back(t.b);
    }
    g_tm_done.clear();
    int n = (int)agg.size();
    for (int i = 0; i < n && i < max; ++i) out[i] = agg[i];
    return n;
}

}  // extern "C"
