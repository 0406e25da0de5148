// Decode step against the m-slot softmax cache plus the linear state (S, z),
// and the export of that state at the end of a prefill.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", sections "Content-Aware Routing with Fixed Budget" (W
// window slots, m - W slots for kept tokens, no re-scoring or eviction, the
// rest accumulated into the recurrent state) and "Delayed Chunk-Level
// Selection for Unified Training-Inference Parallelism" (decode shares the
// prefill's routing rules and memory updates).  roboind.com write-up,
// "Efficiency": decode memory stays almost constant in the context length.
//
// Step at token t of one (sequence, kv head), tokens 0..t-1 absorbed:
//  1. score t over its window [t-W+1, t];
//  2. current-chunk candidates now outranked by lambda tokens fold into (S,z);
//  3. token e = t-W leaves the window: kept by its finished chunk -> already
//     in its slot; current chunk and still in the running top-lambda -> a
//     candidate slot; otherwise -> folded into (S, z);
//  4. t enters the window ring;
//  5. attend: softmax over the window and the kept tokens of finished chunks
//     that left the window, linear over (S, z) and the candidates;
//  6. when t completes its chunk, the chunk's top-lambda are kept for good
//     (the in-window ones are copied into their slots now).
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "sm100.cuh"
#include "tma_host.cuh"

namespace still {

namespace {
constexpr int FB = 8;   // folded keys staged per pass over S
constexpr int CB = 8;   // candidates handled per batch
constexpr int GMAX = 8; // query heads per kv head
}

struct DecodeGeneralSmem {
    int G, D, DF, nslot, lam, C;
    size_t off_qs, off_pq, off_kt, off_vt, off_hsc, off_w, off_sa, off_cand, off_fph, off_fv, off_fold, off_cph,
        off_ac, off_red, off_rs, off_win, total;
};

static DecodeGeneralSmem decode_general_smem(const Dims &dm)
{
    DecodeGeneralSmem L;
    L.G = dm.G; L.D = dm.d; L.DF = dm.df; L.nslot = dm.W + dm.lam * dm.T_max; L.lam = dm.lam; L.C = dm.C;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o += (bytes + 15) & ~size_t(15); return r; };
    L.off_qs = take(4ull * dm.G * dm.d);
    L.off_pq = take(4ull * dm.G * dm.df);
    L.off_kt = take(4ull * dm.d);
    L.off_vt = take(4ull * dm.d);
    L.off_hsc = take(4ull * GMAX + 64);
    L.off_w = take(4ull * dm.G * (L.nslot > 0 ? L.nslot : 1));
    L.off_sa = take(4ull * (L.nslot > 0 ? L.nslot : 1));
    L.off_cand = take(4ull * (dm.lam + 1));
    L.off_fph = take(4ull * FB * dm.df);
    L.off_fv = take(4ull * FB * dm.d);
    L.off_fold = take(4ull * (dm.lam + 2));
    L.off_cph = take(4ull * CB * dm.df);
    L.off_ac = take(4ull * GMAX * CB);
    L.off_red = take(4ull * (256 / dm.d) * dm.G * dm.d);
    L.off_rs = take(dm.C <= 4096 ? 4ull * dm.C : 16);
    L.off_win = take(4ull * (dm.lam + 1));
    L.total = o;
    return L;
}

template <int D, int DF>
__global__ void __launch_bounds__(256) decode_general_kernel(still_decode_state st, const uint16_t *__restrict__ q_t,
                                                     const uint16_t *__restrict__ k_t,
                                                     const uint16_t *__restrict__ v_t, const float *__restrict__ Wf,
                                                     Dims dm, DecodeGeneralSmem L, uint16_t *__restrict__ out_t)
{
    grid_dep_sync();
    constexpr int PARTS = 256 / D;
    extern __shared__ __align__(16) unsigned char dsm[];
    float *qs = reinterpret_cast<float *>(dsm + L.off_qs);
    float *pq = reinterpret_cast<float *>(dsm + L.off_pq);
    float *kt = reinterpret_cast<float *>(dsm + L.off_kt);
    float *vt = reinterpret_cast<float *>(dsm + L.off_vt);
    float *hsc = reinterpret_cast<float *>(dsm + L.off_hsc);
    float *wsa = reinterpret_cast<float *>(dsm + L.off_w);
    int *sa_idx = reinterpret_cast<int *>(dsm + L.off_sa);
    int *cand_idx = reinterpret_cast<int *>(dsm + L.off_cand);
    float *fph = reinterpret_cast<float *>(dsm + L.off_fph);
    float *fv = reinterpret_cast<float *>(dsm + L.off_fv);
    int *fold = reinterpret_cast<int *>(dsm + L.off_fold);
    float *cph = reinterpret_cast<float *>(dsm + L.off_cph);
    float *ac = reinterpret_cast<float *>(dsm + L.off_ac);
    float *red = reinterpret_cast<float *>(dsm + L.off_red);
    float *rs = reinterpret_cast<float *>(dsm + L.off_rs);
    int *win = reinterpret_cast<int *>(dsm + L.off_win);
    __shared__ float s_score, s_den[GMAX];
    __shared__ int s_count, s_nfold, s_cand_slot, s_cand_count, s_nsa, s_ncand, s_nwin;

    const int g = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = dm.G, W = dm.W, C = dm.C, lam = dm.lam, m = dm.m;
    const size_t ug = (size_t)b * dm.Hkv + g;
    uint16_t *K = st.K + ug * m * D;
    uint16_t *V = st.V + ug * m * D;
    int32_t *pos = st.slot_pos + ug * m;
    int32_t *cnt = st.slot_cnt + ug * m;
    float *ssc = st.slot_score + ug * m;
    float *S = st.S + ug * DF * D;
    float *z = st.z + ug * DF;
    float *ring = st.score_ring + ug * C;
    const long long t = st.t[ug];
    const long long ct = t / C;
    const bool selecting = lam > 0 && ct < dm.T_max;
    const int nslot = W + lam * dm.T_max;
    const long long e = t - W;
    const float inv = rsqrtf((float)D);

    for (int i = tid; i < G * D; i += 256) qs[i] = bf2f(q_t[((size_t)b * dm.Hq + (size_t)g * G) * D + i]);
    for (int i = tid; i < D; i += 256) {
        kt[i] = bf2f(k_t[ug * D + i]);
        vt[i] = bf2f(v_t[ug * D + i]);
    }
    if (tid < GMAX) s_den[tid] = 0.f;
    if (tid == 0) { s_count = 0; s_nsa = 0; s_ncand = 0; s_nwin = 0; }
    __syncthreads();

    // NP-Map of the query rows, and the score of token t
    for (int hh = warp; hh < G; hh += 8) {
        warp_npmap<D, DF>(qs + hh * D, Wf, pq + hh * DF, lane);
        if (selecting) {
            const int n = (int)(t + 1 < (long long)W ? t + 1 : (long long)W);
            float ml = -INFINITY, tl = 0.f, sl = 0.f;
            for (int i = lane; i < n; i += 32) {
                float s;
                if (i == 0) {
                    s = 0.f;
                    for (int x = 0; x < D; ++x) s = fmaf(kt[x], qs[hh * D + x], s);
                } else {
                    s = dot_bf16_row<D>(K + (size_t)((t - i) % W) * D, qs + hh * D);
                }
                s *= inv;
                if (s > ml) {
                    const float c = expf(ml - s);
                    tl *= c;
                    sl *= c;
                    ml = s;
                }
                const float w = expf(s - ml);
                if (i == 0) sl += w;
                else tl += w;
            }
            const float M = warp_max(ml);
            const float f = ml == -INFINITY ? 0.f : expf(ml - M);
            const float oth = warp_sum(tl * f), self = warp_sum(sl * f);
            if (lane == 0) hsc[hh] = saliency_from_stats(oth, self);
        }
    }
    __syncthreads();
    if (tid == 0 && selecting) {
        float a = 0.f;
        for (int hh = 0; hh < G; ++hh) a += hsc[hh];
        s_score = a / G;
        ring[t % C] = s_score;
    }
    __syncthreads();

    // how many tokens of the current chunk outrank the token leaving the window
    const bool e_current = e >= 0 && selecting && e / C == ct;
    if (e_current) {
        const float se = ring[e % C];
        int local = 0;
        for (long long i = ct * C + tid; i <= t; i += 256)
            if (i != e && outranks(i, ring[i % C], e, se)) ++local;
        if (local) atomicAdd(&s_count, local);
    }
    __syncthreads();

    // routing decisions (one thread; at most lambda + 1 slots are touched)
    if (tid == 0) {
        int nf = 0;
        s_cand_slot = -1;
        if (selecting) {
            for (int r = 0; r < lam; ++r) {
                const int sl = W + (int)ct * lam + r;
                const int p = pos[sl];
                if (p >= 0 && outranks(t, s_score, p, ssc[sl])) {
                    const int c = cnt[sl] + 1;
                    cnt[sl] = c;
                    if (c >= lam) {
                        fold[nf++] = sl;
                        pos[sl] = -1;
                        cnt[sl] = 0;
                    }
                }
            }
        }
        if (e >= 0) {
            const int esrc = W > 0 ? (int)(e % W) : -1;
            const long long ce = e / C;
            if (lam == 0 || ce >= dm.T_max) {
                fold[nf++] = esrc;
            } else if (ce < ct) {
                bool kept = false;
                for (int r = 0; r < lam; ++r) kept |= pos[W + ce * lam + r] == e;
                if (!kept) fold[nf++] = esrc;
            } else if (s_count < lam) {
                int target = -1;
                for (int r = 0; r < lam && target < 0; ++r)
                    if (pos[W + ct * lam + r] < 0) target = W + (int)ct * lam + r;
                if (target < 0) {
                    set_status(st.status, STILL_ERR_BOUNDS);
                    fold[nf++] = esrc;
                } else {
                    s_cand_slot = target;
                    s_cand_count = s_count;
                }
            } else {
                fold[nf++] = esrc;
            }
        }
        s_nfold = nf;
    }
    __syncthreads();
    const int nfold = s_nfold;

    // stage the folded keys: phi(k) and v in fp32 (batches of FB)
    int nbatch = (nfold + FB - 1) / FB;
    for (int bt = 0; bt < nbatch; ++bt) {
        const int f0 = bt * FB, nb = min(FB, nfold - f0);
        for (int ff = warp; ff < nb; ff += 8) {
            const int src = fold[f0 + ff];
            float *xk = fph + ff * DF;   // first the raw key, then phi in place
            __shared__ float kraw[8][D];
            __syncwarp();
            for (int x = lane; x < D; x += 32) {
                kraw[warp][x] = src >= 0 ? bf2f(K[(size_t)src * D + x]) : kt[x];
                fv[ff * D + x] = src >= 0 ? bf2f(V[(size_t)src * D + x]) : vt[x];
            }
            __syncwarp();
            warp_npmap<D, DF>(kraw[warp], Wf, xk, lane);
        }
        __syncthreads();
        if (bt + 1 < nbatch) {
            // all but the last batch: update S, z only
            for (int i = tid / D; i < DF; i += PARTS) {
                const int c = tid % D;
                float a = S[(size_t)i * D + c];
                for (int ff = 0; ff < nb; ++ff) a = fmaf(fph[ff * DF + i], fv[ff * D + c], a);
                S[(size_t)i * D + c] = a;
            }
            if (tid < DF) {
                float a = z[tid];
                for (int ff = 0; ff < nb; ++ff) a += fph[ff * DF + tid];
                z[tid] = a;
            }
            __syncthreads();
        } else {
            // keep nb for the fused pass below
            if (tid == 0) s_nfold = nb;
            __syncthreads();
        }
    }
    const int nlast = nbatch > 0 ? s_nfold : 0;

    // token e becomes a candidate (before the ring slot is reused by t)
    if (s_cand_slot >= 0) {
        const int sl = s_cand_slot, src = (int)(e % W);
        for (int x = tid; x < D; x += 256) {
            K[(size_t)sl * D + x] = K[(size_t)src * D + x];
            V[(size_t)sl * D + x] = V[(size_t)src * D + x];
        }
        if (tid == 0) {
            pos[sl] = (int32_t)e;
            cnt[sl] = s_cand_count;
            ssc[sl] = ring[e % C];
        }
    }
    __syncthreads();
    if (W > 0) {
        const int sl = (int)(t % W);
        for (int x = tid; x < D; x += 256) {
            K[(size_t)sl * D + x] = k_t[ug * D + x];
            V[(size_t)sl * D + x] = v_t[ug * D + x];
        }
        if (tid == 0) pos[sl] = (int32_t)t;
    }
    __syncthreads();

    // softmax keys and candidates
    for (int s = tid; s < nslot; s += 256) {
        const int p = pos[s];
        bool sa, cd = false;
        if (s < W) {
            sa = p >= 0;
        } else {
            sa = p >= 0 && p / C < ct && p <= t - W;
            cd = p >= 0 && p / C == ct;
        }
        if (sa) sa_idx[atomicAdd(&s_nsa, 1)] = s;
        if (cd) cand_idx[atomicAdd(&s_ncand, 1)] = s;
    }
    __syncthreads();
    const int nsa = s_nsa, ncand = s_ncand;

    // logits: one warp per key, coalesced row loads
    for (int kk = warp; kk < nsa; kk += 8) {
        const uint16_t *kr = K + (size_t)sa_idx[kk] * D;
        float part[GMAX];
#pragma unroll
        for (int hh = 0; hh < GMAX; ++hh) part[hh] = 0.f;
        for (int x = lane; x < D; x += 32) {
            const float kv = bf2f(kr[x]);
#pragma unroll
            for (int hh = 0; hh < GMAX; ++hh)
                if (hh < G) part[hh] = fmaf(kv, qs[hh * D + x], part[hh]);
        }
#pragma unroll
        for (int hh = 0; hh < GMAX; ++hh) {
            if (hh >= G) break;
            const float sv = warp_sum(part[hh]);
            if (lane == 0) wsa[hh * nslot + kk] = sv * inv;
        }
    }
    __syncthreads();
    for (int hh = warp; hh < G; hh += 8) {
        float mx = -INFINITY;
        for (int kk = lane; kk < nsa; kk += 32) mx = fmaxf(mx, wsa[hh * nslot + kk]);
        mx = warp_max(mx);
        float su = 0.f;
        for (int kk = lane; kk < nsa; kk += 32) {
            const float w = expf(wsa[hh * nslot + kk] - mx);
            wsa[hh * nslot + kk] = w;
            su += w;
        }
        su = warp_sum(su);
        if (lane == 0) s_den[hh] += su;
    }
    __syncthreads();

    const int col = tid % D, part = tid / D;
    float acc[GMAX];
#pragma unroll
    for (int hh = 0; hh < GMAX; ++hh) acc[hh] = 0.f;
    for (int kk = part; kk < nsa; kk += PARTS) {
        const float vv = bf2f(V[(size_t)sa_idx[kk] * D + col]);
#pragma unroll
        for (int hh = 0; hh < GMAX; ++hh)
            if (hh < G) acc[hh] = fmaf(wsa[hh * nslot + kk], vv, acc[hh]);
    }
    // linear state (with the last batch of folded keys added on the way)
    for (int i = part; i < DF; i += PARTS) {
        float sv = S[(size_t)i * D + col];
        if (nlast) {
            for (int ff = 0; ff < nlast; ++ff) sv = fmaf(fph[ff * DF + i], fv[ff * D + col], sv);
            S[(size_t)i * D + col] = sv;
        }
#pragma unroll
        for (int hh = 0; hh < GMAX; ++hh)
            if (hh < G) acc[hh] = fmaf(pq[hh * DF + i], sv, acc[hh]);
    }
#pragma unroll
    for (int hh = 0; hh < GMAX; ++hh)
        if (hh < G) red[(part * G + hh) * D + col] = acc[hh];
    if (warp == 0) {
        float dz[GMAX];
#pragma unroll
        for (int hh = 0; hh < GMAX; ++hh) dz[hh] = 0.f;
        for (int i = lane; i < DF; i += 32) {
            float zv = z[i];
            if (nlast) {
                for (int ff = 0; ff < nlast; ++ff) zv += fph[ff * DF + i];
                z[i] = zv;
            }
#pragma unroll
            for (int hh = 0; hh < GMAX; ++hh)
                if (hh < G) dz[hh] = fmaf(pq[hh * DF + i], zv, dz[hh]);
        }
#pragma unroll
        for (int hh = 0; hh < GMAX; ++hh) {
            if (hh >= G) break;
            const float a = warp_sum(dz[hh]);
            if (lane == 0) s_den[hh] += a;
        }
    }
    __syncthreads();

    // candidates of the current chunk are linear keys with explicit phi(k)
    for (int c0 = 0; c0 < ncand; c0 += CB) {
        const int nb = min(CB, ncand - c0);
        for (int cc = warp; cc < nb; cc += 8) {
            __shared__ float craw[8][D];
            const int sl = cand_idx[c0 + cc];
            __syncwarp();
            for (int x = lane; x < D; x += 32) craw[warp][x] = bf2f(K[(size_t)sl * D + x]);
            __syncwarp();
            warp_npmap<D, DF>(craw[warp], Wf, cph + cc * DF, lane);
            __syncwarp();
            for (int hh = 0; hh < G; ++hh) {
                float a = 0.f;
                for (int i = lane; i < DF; i += 32) a = fmaf(pq[hh * DF + i], cph[cc * DF + i], a);
                a = warp_sum(a);
                if (lane == 0) ac[hh * CB + cc] = a;
            }
        }
        __syncthreads();
        if (part == 0) {
            for (int cc = 0; cc < nb; ++cc) {
                const float vv = bf2f(V[(size_t)cand_idx[c0 + cc] * D + col]);
                for (int hh = 0; hh < G; ++hh) red[hh * D + col] = fmaf(ac[hh * CB + cc], vv, red[hh * D + col]);
            }
        }
        if (tid < G)
            for (int cc = 0; cc < nb; ++cc) s_den[tid] += ac[tid * CB + cc];
        __syncthreads();
    }

    for (int i = tid; i < G * D; i += 256) {
        const int hh = i / D, c = i % D;
        float num = 0.f;
        for (int p = 0; p < PARTS; ++p) num += red[(p * G + hh) * D + c];
        const float den = s_den[hh];
        out_t[((size_t)b * dm.Hq + (size_t)g * G + hh) * D + c] = f2bf(den != 0.f ? num / den : 0.f);
    }

    // the chunk of t is complete: keep its top-lambda for good
    if (selecting && (t + 1) % C == 0) {
        const long long base = ct * C;
        const bool staged = C <= 4096;
        if (staged)
            for (int i = tid; i < C; i += 256) rs[i] = ring[i];
        __syncthreads();
        const float *src = staged ? rs : ring;
        for (int i = tid; i < C; i += 256) {
            const float si = src[i];
            int rank = 0;
            for (int j = 0; j < C && rank < lam; ++j)
                if (j != i && outranks(base + j, src[j], base + i, si)) ++rank;
            if (rank < lam) win[atomicAdd(&s_nwin, 1)] = i;
        }
        __syncthreads();
        if (warp == 0) {
            const int nw = s_nwin;
            for (int r = 0; r < nw; ++r) {
                const long long w = base + win[r];
                if (w <= t - W) {
                    bool found = false;
                    for (int x = 0; x < lam; ++x) found |= pos[W + ct * lam + x] == w;
                    if (!found && lane == 0) set_status(st.status, STILL_ERR_BOUNDS);
                    continue;
                }
                int target = -1;
                for (int x = 0; x < lam && target < 0; ++x)
                    if (pos[W + ct * lam + x] < 0) target = W + (int)ct * lam + x;
                if (target < 0) {
                    if (lane == 0) set_status(st.status, STILL_ERR_BOUNDS);
                    continue;
                }
                const int srcs = (int)(w % W);
                for (int x = lane; x < D; x += 32) {
                    K[(size_t)target * D + x] = K[(size_t)srcs * D + x];
                    V[(size_t)target * D + x] = V[(size_t)srcs * D + x];
                }
                __syncwarp();
                if (lane == 0) {
                    pos[target] = (int32_t)w;
                    ssc[target] = src[win[r]];
                }
                __syncwarp();
            }
            for (int x = lane; x < lam; x += 32) cnt[W + ct * lam + x] = 0;
        }
    }
    if (tid == 0) st.t[ug] = t + 1;
}

// ---------------------------------------------------------------------------
// Staged decode step: the slot cache of one (sequence, kv head) passes
// through one 128-byte-swizzled shared buffer, K first and then V, each
// brought in by TMA, so that two steps share an SM and one's loads overlap
// the other's arithmetic.  Folded keys and candidates are linear keys with an
// explicit weight phi(q).phi(k): the output reads the linear state before the
// fold plus those keys, and the fold itself is written to (S, z) once V is in.
// ---------------------------------------------------------------------------
namespace {
constexpr int DS_THREADS = 256;
constexpr int DS_BOX_ROWS = 64;    // rows per TMA box (64 bf16 columns x 64 rows = 8 KB)
constexpr int DS_NP_ROWS = 8;      // rows per pass of the block-wide NP-Map
}

struct DecodeSmem {
    int nslot;      // W + lambda * T_max slots in use
    int R;          // slot rows held in the buffer (nslot rounded up to DS_BOX_ROWS)
    int xrows;      // feature rows: G query heads + at most lambda + 1 linear keys
    size_t off_buf, off_x, off_phi, off_np, off_w, off_pos, off_kv, off_lin, off_small, off_qb, total;
};

static DecodeSmem decode_smem(const Dims &dm)
{
    DecodeSmem L;
    L.nslot = dm.W + dm.lam * dm.T_max;
    L.R = (L.nslot + DS_BOX_ROWS - 1) / DS_BOX_ROWS * DS_BOX_ROWS;
    L.xrows = dm.G + dm.lam + 1;
    const int rg = DS_THREADS / (dm.d / 4);
    size_t o = 0;
    auto take = [&](size_t bytes, size_t align) {
        o = (o + align - 1) / align * align;
        const size_t r = o;
        o += bytes;
        return r;
    };
    size_t buf = (size_t)L.R * dm.d * 2;
    const size_t parts = (size_t)rg + 8 / (dm.d / 16);                                    // + the MMA's slot splits
    buf = buf > 4ull * parts * dm.G * dm.d ? buf : 4ull * parts * dm.G * dm.d;           // partial outputs
    const size_t fin = (dm.C <= 4096 ? 4ull * dm.C : 0) + 4ull * (dm.lam + 1) + 16;      // chunk completion
    buf = buf > fin ? buf : fin;
    L.off_buf = take(buf, 1024);
    L.off_x = take(4ull * L.xrows * dm.d, 16);
    L.off_phi = take(4ull * L.xrows * dm.df, 16);
    // NP-Map partial sums, then (from the logits on) the softmax weights
    const size_t np = 4ull * (1024 / dm.df) * DS_NP_ROWS * dm.df, w = 4ull * dm.G * (L.nslot > 0 ? L.nslot : 1);
    L.off_np = take(np > w ? np : w, 16);
    L.off_w = L.off_np;
    L.off_pos = take(4ull * (L.nslot > 0 ? L.nslot : 1), 16);
    L.off_kv = take(8ull * dm.d, 16);
    L.off_lin = take(4ull * (dm.lam + 1) * (dm.G + 1), 16);
    L.off_small = take(16ull * (dm.lam + 2), 16);
    L.off_qb = take(2ull * 8 * dm.d, 16);   // bf16 query rows, 8 heads (zero past G): the MMA's B operand
    L.total = o + 1024;   // room to align the base to 1024 bytes
    return L;
}

// Warp-level bf16 MMA (m16n8k16, fp32 accumulation) and the 8x8 shared-memory
// matrix loads that feed it.  The decode step's two contractions (q K^T over
// the slots, and V^T P^T) are too small for the asynchronous tensor-core
// path; these replace long per-thread dot-product loops.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of element (row, col) in the staged buffer: 64-column blocks of
// R rows x 128 B, 16-byte chunks XOR-swizzled with the row (the layout TMA
// writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint32_t ds_off(int R, int row, int col)
{
    return (uint32_t)(col >> 6) * (uint32_t)R * 128u + sm100::sw128((uint32_t)row, (uint32_t)((col >> 3) & 7)) +
           (uint32_t)(col & 7) * 2u;
}

// NP-Map of `nrows` fp32 rows x (shared, [nrows][D]) into phi ([nrows][DF]).
// x Wf is split over 1024/DF slices of the D inputs, one float4 of columns
// per thread; warp r then finishes row r (softmax over DF, norms).
template <int D, int DF>
__device__ void block_npmap(const float *x, int nrows, const float *__restrict__ Wf, float *phi, float *part)
{
    constexpr int C4 = DF / 4, NS = DS_THREADS / C4, IS = D / NS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c4 = tid % C4, sl = tid / C4;
    for (int r0 = 0; r0 < nrows; r0 += DS_NP_ROWS) {
        const int nr = min(DS_NP_ROWS, nrows - r0);
        float4 acc[DS_NP_ROWS];
#pragma unroll
        for (int r = 0; r < DS_NP_ROWS; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int i = 0; i < IS; ++i) {
            const float4 w = __ldg(reinterpret_cast<const float4 *>(Wf + (size_t)(sl * IS + i) * DF) + c4);
#pragma unroll
            for (int r = 0; r < DS_NP_ROWS; ++r) {
                if (r < nr) {
                    const float xv = x[(r0 + r) * D + sl * IS + i];
                    const float2 lo = __ffma2_rn(make_float2(xv, xv), make_float2(w.x, w.y), make_float2(acc[r].x, acc[r].y));
                    const float2 hi = __ffma2_rn(make_float2(xv, xv), make_float2(w.z, w.w), make_float2(acc[r].z, acc[r].w));
                    acc[r] = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < DS_NP_ROWS; ++r)
            if (r < nr) reinterpret_cast<float4 *>(part + ((size_t)sl * DS_NP_ROWS + r) * DF)[c4] = acc[r];
        __syncthreads();
        if (warp < nr) {
            const int r = warp;
            constexpr int PJ = DF / 32;
            float u[PJ];
#pragma unroll
            for (int k = 0; k < PJ; ++k) {
                float a = 0.f;
                for (int s2 = 0; s2 < NS; ++s2) a += part[((size_t)s2 * DS_NP_ROWS + r) * DF + lane + 32 * k];
                u[k] = a;
            }
            float mx = u[0];
#pragma unroll
            for (int k = 1; k < PJ; ++k) mx = fmaxf(mx, u[k]);
            mx = warp_max(mx);
            float s2e = 0.f;
#pragma unroll
            for (int k = 0; k < PJ; ++k) {
                u[k] = expf(u[k] - mx);
                s2e = fmaf(u[k], u[k], s2e);
            }
            s2e = warp_sum(s2e);
            float nx = 0.f;
            for (int i = lane; i < D; i += 32) nx = fmaf(x[(r0 + r) * D + i], x[(r0 + r) * D + i], nx);
            nx = warp_sum(nx);
            // phi = ||x|| u / ||u||, u = e / sum(e): the softmax sum cancels
            const float sc = sqrtf(nx) * rsqrtf(s2e);
#pragma unroll
            for (int k = 0; k < PJ; ++k) phi[(r0 + r) * DF + lane + 32 * k] = sc * u[k];
        }
        __syncthreads();
    }
}

template <int D, int DF, int G>
__global__ void __launch_bounds__(DS_THREADS, 2)
    decode_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                  still_decode_state st, const uint16_t *__restrict__ q_t, const uint16_t *__restrict__ k_t,
                  const uint16_t *__restrict__ v_t, const float *__restrict__ Wf, Dims dm, DecodeSmem L,
                  uint16_t *__restrict__ out_t, const uint16_t *__restrict__ gate_t)
{
    grid_dep_sync();
    using namespace sm100;
    constexpr int C4 = D / 4;              // 4-column groups of an output row
    constexpr int RG = DS_THREADS / C4;    // thread rows: S rows / slots handled in parallel
    constexpr int SR = DF / RG;            // S rows held per thread
    extern __shared__ __align__(16) unsigned char dsm_raw[];
    unsigned char *dsm = (unsigned char *)(((uintptr_t)dsm_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *buf = dsm + L.off_buf;
    float *xs = reinterpret_cast<float *>(dsm + L.off_x);       // q heads, then linear keys (fp32)
    float *phs = reinterpret_cast<float *>(dsm + L.off_phi);
    float *npart = reinterpret_cast<float *>(dsm + L.off_np);
    float *wsa = reinterpret_cast<float *>(dsm + L.off_w);
    int *spos = reinterpret_cast<int *>(dsm + L.off_pos);
    float *ktf = reinterpret_cast<float *>(dsm + L.off_kv), *vtf = ktf + D;
    float *alin = reinterpret_cast<float *>(dsm + L.off_lin);   // [lin][G] weights phi(q).phi(k)
    int *lsrc = reinterpret_cast<int *>(dsm + L.off_small);     // source slot of each linear key (-1: k_t)
    int *scnt = lsrc + (dm.lam + 2);
    float *sssc = reinterpret_cast<float *>(scnt + (dm.lam + 2));
    int *lcand = scnt + 2 * (dm.lam + 2);                        // candidates, before they follow the folds
    __shared__ uint64_t bar_kv;
    __shared__ float s_score, s_den[G], s_hsc[G];
    __shared__ int s_count, s_nfold, s_nlin, s_cand_slot, s_cand_count, s_nwin;

    const int g = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int W = dm.W, C = dm.C, lam = dm.lam, m = dm.m;
    const int nslot = L.nslot, R = L.R;
    const size_t ug = (size_t)b * dm.Hkv + g;
    uint16_t *K = st.K + ug * m * D;
    uint16_t *V = st.V + ug * m * D;
    int32_t *pos = st.slot_pos + ug * m;
    int32_t *cnt = st.slot_cnt + ug * m;
    float *ssc = st.slot_score + ug * m;
    float *S = st.S + ug * DF * D;
    float *z = st.z + ug * DF;
    float *ring = st.score_ring + ug * C;
    const long long t = st.t[ug];
    const long long ct = t / C;
    const bool selecting = lam > 0 && ct < dm.T_max;
    const long long e = t - W;
    const float inv = rsqrtf((float)D);
    const int tslot = W > 0 ? (int)(t % W) : -1;
    const uint32_t buf_bytes = (uint32_t)R * D * 2;

    // ---- K of every slot into the buffer; S, z and the small rows meanwhile ----
    if (tid == 0) {
        mbar_init(&bar_kv, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && nslot > 0) {
        mbar_expect_tx(&bar_kv, buf_bytes);
        for (int j = 0; j < R / DS_BOX_ROWS; ++j)
            for (int cb = 0; cb < D / 64; ++cb)
                tma_load_2d(buf + (size_t)cb * R * 128 + (size_t)j * DS_BOX_ROWS * 128, &mapK, &bar_kv, cb * 64,
                            (int)(ug * m) + j * DS_BOX_ROWS);
    }
    const int c4 = tid % C4, part = tid / C4;
    const float zo = tid < DF ? z[tid] : 0.f;
    for (int i = tid; i < G * D; i += DS_THREADS) xs[i] = bf2f(q_t[((size_t)b * dm.Hq + (size_t)g * G) * D + i]);
    uint16_t *qb = reinterpret_cast<uint16_t *>(dsm + L.off_qb);
    for (int i = tid; i < 8 * D; i += DS_THREADS) qb[i] = i < G * D ? q_t[((size_t)b * dm.Hq + (size_t)g * G) * D + i] : (uint16_t)0;
    for (int i = tid; i < D; i += DS_THREADS) {
        ktf[i] = bf2f(k_t[ug * D + i]);
        vtf[i] = bf2f(v_t[ug * D + i]);
    }
    for (int i = tid; i < nslot; i += DS_THREADS) spos[i] = pos[i];
    if (selecting && tid < lam) {
        scnt[tid] = cnt[W + ct * lam + tid];
        sssc[tid] = ssc[W + ct * lam + tid];
    }
    if (tid < G) s_den[tid] = 0.f;
    if (tid == 0) { s_count = 0; s_nwin = 0; s_cand_slot = -1; }
    if (nslot > 0) mbar_wait_sleep(&bar_kv, 0, st.status);
    __syncthreads();

    // ---- (1) score of token t over its window [t-W+1, t] --------------------------
    if (selecting) {
        for (int hh = warp; hh < G; hh += DS_THREADS / 32) {
            const int n = (int)(t + 1 < (long long)W ? t + 1 : (long long)W);
            const float *qh = xs + hh * D;
            float ml = -INFINITY, ol = 0.f, sl = 0.f;
            for (int i = lane; i < n; i += 32) {
                float sv = 0.f;
                if (i == 0) {
                    for (int x = 0; x < D; ++x) sv = fmaf(ktf[x], qh[x], sv);
                } else {
                    const int row = (int)((t - i) % W);
#pragma unroll 4
                    for (int c = 0; c < D / 8; ++c) {
                        const uint4 pk = *reinterpret_cast<const uint4 *>(buf + ds_off(R, row, 8 * c));
                        const uint32_t w4[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                        for (int h2 = 0; h2 < 4; ++h2) {
                            sv = fmaf(__uint_as_float(w4[h2] << 16), qh[8 * c + 2 * h2], sv);
                            sv = fmaf(__uint_as_float(w4[h2] & 0xffff0000u), qh[8 * c + 2 * h2 + 1], sv);
                        }
                    }
                }
                sv *= inv;
                if (sv > ml) {
                    const float cf = expf(ml - sv);
                    ol *= cf;
                    sl *= cf;
                    ml = sv;
                }
                const float w = expf(sv - ml);
                if (i == 0) sl += w;
                else ol += w;
            }
            const float M = warp_max(ml);
            const float f = ml == -INFINITY ? 0.f : expf(ml - M);
            const float oth = warp_sum(ol * f), self = warp_sum(sl * f);
            if (lane == 0) s_hsc[hh] = saliency_from_stats(oth, self);
        }
        __syncthreads();
        if (tid == 0) {
            float a = 0.f;
            for (int hh = 0; hh < G; ++hh) a += s_hsc[hh];
            s_score = a / G;
            ring[t % C] = s_score;
        }
        __syncthreads();
    }

    // ---- (2)-(3) routing --------------------------------------------------------------
    const bool e_current = e >= 0 && selecting && e / C == ct;
    if (e_current) {
        const float se = ring[e % C];
        int local = 0;
        for (long long i = ct * C + tid; i <= t; i += DS_THREADS)
            if (i != e && outranks(i, ring[i % C], e, se)) ++local;
        if (local) atomicAdd(&s_count, local);
    }
    __syncthreads();
    if (tid == 0) {
        // linear keys of this step: folded keys first (lsrc[0..nf)), then the
        // candidates of the current chunk, which stay in their slots
        int nf = 0, nc = 0;
        if (selecting) {
            for (int r = 0; r < lam; ++r) {
                const int sl = W + (int)ct * lam + r;
                if (spos[sl] < 0) continue;
                bool folded = false;
                if (outranks(t, s_score, spos[sl], sssc[r])) {
                    const int c = scnt[r] + 1;
                    cnt[sl] = c;
                    if (c >= lam) {
                        lsrc[nf++] = sl;
                        pos[sl] = -1;
                        cnt[sl] = 0;
                        folded = true;
                    }
                }
                if (!folded) lcand[nc++] = sl;
            }
        }
        if (e >= 0) {
            const long long ce = e / C;
            bool fold = false;
            if (lam == 0 || ce >= dm.T_max) {
                fold = true;
            } else if (ce < ct) {
                bool kept = false;
                for (int r = 0; r < lam; ++r) kept |= spos[W + ce * lam + r] == e;
                fold = !kept;
            } else if (s_count < lam) {
                int target = -1;
                for (int r = 0; r < lam && target < 0; ++r)
                    if (pos[W + ct * lam + r] < 0) target = W + (int)ct * lam + r;
                if (target < 0) {
                    set_status(st.status, STILL_ERR_BOUNDS);
                    fold = true;
                } else {
                    s_cand_slot = target;
                    s_cand_count = s_count;
                    lcand[nc++] = tslot;   // its K/V still sit in the window slot of the buffer
                }
            } else {
                fold = true;
            }
            if (fold) lsrc[nf++] = tslot;   // -1 when W = 0: the token t itself
        }
        for (int c = 0; c < nc; ++c) lsrc[nf + c] = lcand[c];
        s_nfold = nf;
        s_nlin = nf + nc;
    }
    __syncthreads();
    const int nfold = s_nfold, nlin = s_nlin;

    // ---- NP-Map of the query heads and the linear keys -----------------------------
    for (int i = tid; i < nlin * D; i += DS_THREADS) {
        const int l = i / D, x = i % D, src = lsrc[l];
        xs[(G + l) * D + x] = src >= 0 ? bf2f(*reinterpret_cast<const uint16_t *>(buf + ds_off(R, src, x))) : ktf[x];
    }
    __syncthreads();
    // every read of the staged K before this step is done: the window slot of t
    // takes k_t, so that every slot is a plain row for the logits (the NP-Map's
    // barriers order these writes before them)
    if (nslot > 0 && tslot >= 0)
        for (int x = tid; x < D; x += DS_THREADS) *reinterpret_cast<uint16_t *>(buf + ds_off(R, tslot, x)) = k_t[ug * D + x];
    block_npmap<D, DF>(xs, G + nlin, Wf, phs, npart);

    // the linear state S (fp32) into registers; the loads complete behind the logits
    float4 Sreg[SR];
#pragma unroll
    for (int k = 0; k < SR; ++k) Sreg[k] = *reinterpret_cast<const float4 *>(S + (size_t)(part + RG * k) * D + 4 * c4);

    // ---- (4)-(5) softmax logits: window (slot t % W now holds t) and kept slots ----
    // [16 slots x 8 heads] += K[16 slots x 16 dims] q^T[16 dims x 8 heads] per MMA,
    // one group of 16 slots per warp at a time; heads past G are zero columns
    {
        const int g8 = lane >> 2, t4 = lane & 3, mi = lane >> 3;
        uint32_t qf[D / 16][2];
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qf[ks][0] = *reinterpret_cast<const uint32_t *>(qb + g8 * D + ks * 16 + 2 * t4);
            qf[ks][1] = *reinterpret_cast<const uint32_t *>(qb + g8 * D + ks * 16 + 2 * t4 + 8);
        }
        const uint32_t bufa = smem_u32(buf);
        for (int grp = warp; grp * 16 < nslot; grp += DS_THREADS / 32) {
            // this lane's row address: 8x8 matrix mi holds slots +8 (mi & 1), dims +8 (mi >> 1)
            const uint32_t row = (uint32_t)(grp * 16 + (mi & 1) * 8 + (lane & 7));
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t j = (uint32_t)(2 * ks + (mi >> 1));   // 16-byte chunk of the row
                uint32_t a[4];
                ldsm_x4(bufa + (j >> 3) * (uint32_t)R * 128u + sw128(row, j & 7u), a);
                mma_16816(c, a, qf[ks][0], qf[ks][1]);
            }
            // c[2 hf + e]: slot grp*16 + g8 + 8 hf, head 2 t4 + e
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int sl = grp * 16 + g8 + 8 * hf;
                if (sl >= nslot) continue;
                const int p = spos[sl];
                bool sa;
                if (sl < W) sa = sl == tslot || p >= 0;
                else sa = p >= 0 && p / C < ct && p <= t - W;
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int hh = 2 * t4 + e2;
                    if (hh < G) wsa[hh * nslot + sl] = sa ? c[2 * hf + e2] * inv : -INFINITY;
                }
            }
        }
    }
    __syncthreads();
    // every read of K in the buffer is done: V takes its place
    if (tid == 0 && nslot > 0) {
        fence_async_smem();
        mbar_expect_tx(&bar_kv, buf_bytes);
        for (int j = 0; j < R / DS_BOX_ROWS; ++j)
            for (int cb = 0; cb < D / 64; ++cb)
                tma_load_2d(buf + (size_t)cb * R * 128 + (size_t)j * DS_BOX_ROWS * 128, &mapV, &bar_kv, cb * 64,
                            (int)(ug * m) + j * DS_BOX_ROWS);
    }
    // softmax weights, one warp per head
    for (int hh = warp; hh < G; hh += DS_THREADS / 32) {
        float mx = -INFINITY;
        for (int sl = lane; sl < nslot; sl += 32) mx = fmaxf(mx, wsa[hh * nslot + sl]);
        mx = warp_max(mx);
        float su = 0.f;
        for (int sl = lane; sl < nslot; sl += 32) {
            const float x = wsa[hh * nslot + sl];
            const float w = x == -INFINITY ? 0.f : expf(x - mx);
            wsa[hh * nslot + sl] = w;
            su += w;
        }
        su = warp_sum(su);
        if (lane == 0) atomicAdd(&s_den[hh], su);
    }
    // linear keys: weight phi(q_h).phi(k), one warp per key
    for (int l = warp; l < nlin; l += DS_THREADS / 32) {
        const float *pk = phs + (G + l) * DF;
        for (int hh = 0; hh < G; ++hh) {
            float a = 0.f;
            for (int i = lane; i < DF; i += 32) a = fmaf(phs[hh * DF + i], pk[i], a);
            a = warp_sum(a);
            if (lane == 0) alin[l * G + hh] = a;
        }
    }
    // readout of the linear state before this step's fold
    float2 acc[G][2];   // output columns 4*c4 .. 4*c4+3 of each head, in pairs
#pragma unroll
    for (int hh = 0; hh < G; ++hh) acc[hh][0] = acc[hh][1] = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < SR; ++k) {
        const int i = part + RG * k;
        const float4 sv = Sreg[k];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float a = phs[hh * DF + i];
            acc[hh][0] = __ffma2_rn(make_float2(a, a), make_float2(sv.x, sv.y), acc[hh][0]);
            acc[hh][1] = __ffma2_rn(make_float2(a, a), make_float2(sv.z, sv.w), acc[hh][1]);
        }
    }
    if (tid < DF) {
        float zn = zo;
        for (int f = 0; f < nfold; ++f) zn += phs[(G + f) * DF + tid];
        if (nfold > 0) z[tid] = zn;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float a = warp_sum(phs[hh * DF + tid] * zo);
            if (lane == 0) atomicAdd(&s_den[hh], a);
        }
    }
    __syncthreads();
    if (tid < G) {
        float a = 0.f;
        for (int l = 0; l < nlin; ++l) a += alin[l * G + tid];
        s_den[tid] += a;
    }

    // ---- V: softmax keys and linear keys; the fold into S ----------------------------
    if (nslot > 0) mbar_wait_sleep(&bar_kv, 1, st.status);
    // V row `src` of the buffer, columns 4*c4 .. 4*c4+3, as two pairs
    auto vbuf4 = [&](uint32_t off, float2 &v01, float2 &v23) {
        const uint2 pk = *reinterpret_cast<const uint2 *>(buf + off);
        v01 = make_float2(__uint_as_float(pk.x << 16), __uint_as_float(pk.x & 0xffff0000u));
        v23 = make_float2(__uint_as_float(pk.y << 16), __uint_as_float(pk.y & 0xffff0000u));
    };
    // linear keys: a slot of the buffer as it was before this step (the window
    // slot of t still holds the token leaving the window), or v_t when W = 0
    auto vlin4 = [&](int src, float2 &v01, float2 &v23) {
        if (src >= 0) {
            vbuf4(ds_off(R, src, 4 * c4), v01, v23);
        } else {
            v01 = make_float2(vtf[4 * c4], vtf[4 * c4 + 1]);
            v23 = make_float2(vtf[4 * c4 + 2], vtf[4 * c4 + 3]);
        }
    };
    for (int l = part; l < nlin; l += RG) {
        float2 v01, v23;
        vlin4(lsrc[l], v01, v23);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float a = alin[l * G + hh];
            acc[hh][0] = __ffma2_rn(make_float2(a, a), v01, acc[hh][0]);
            acc[hh][1] = __ffma2_rn(make_float2(a, a), v23, acc[hh][1]);
        }
    }
    if (nfold > 0) {
        for (int f = 0; f < nfold; ++f) {
            float2 v01, v23;
            vlin4(lsrc[f], v01, v23);
#pragma unroll
            for (int k = 0; k < SR; ++k) {
                const float a = phs[(G + f) * DF + part + RG * k];
                const float2 lo = __ffma2_rn(make_float2(a, a), v01, make_float2(Sreg[k].x, Sreg[k].y));
                const float2 hi = __ffma2_rn(make_float2(a, a), v23, make_float2(Sreg[k].z, Sreg[k].w));
                Sreg[k] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
#pragma unroll
        for (int k = 0; k < SR; ++k) *reinterpret_cast<float4 *>(S + (size_t)(part + RG * k) * D + 4 * c4) = Sreg[k];
    }
    // ---- softmax keys: V^T P^T on the tensor cores ----------------------------------
    // The window slot of t takes v_t (the linear keys above have read the token
    // that left it).  Warp w: output dims [16 (w % MT), +16) over every KSPLIT-th
    // group of 16 slots; V^T comes from the slot rows by transposing 8x8 loads,
    // P^T as bf16 pairs of consecutive slots of one head.
    constexpr int MT = D / 16, KSPLIT = (DS_THREADS / 32) / MT;
    __syncthreads();
    if (nslot > 0 && tslot >= 0)
        for (int x = tid; x < D; x += DS_THREADS) *reinterpret_cast<uint16_t *>(buf + ds_off(R, tslot, x)) = v_t[ug * D + x];
    __syncthreads();
    const int mt = warp % MT, kp = warp / MT;
    float pv[4] = {0.f, 0.f, 0.f, 0.f};
    {
        const int g8 = lane >> 2, t4 = lane & 3, mi = lane >> 3;
        const uint32_t bufa = smem_u32(buf);
        const uint32_t j = (uint32_t)(2 * mt + (mi & 1));   // 16-byte chunk of the slot row
        for (int ks = kp; ks * 16 < nslot; ks += KSPLIT) {
            const int k0 = ks * 16;
            const uint32_t row = (uint32_t)(k0 + (mi >> 1) * 8 + (lane & 7));
            uint32_t a[4];
            ldsm_x4_trans(bufa + (j >> 3) * (uint32_t)R * 128u + sw128(row, j & 7u), a);
            uint32_t bb[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int s0 = k0 + 2 * t4 + 8 * hf;
                const float w0 = (g8 < G && s0 < nslot) ? wsa[g8 * nslot + s0] : 0.f;
                const float w1 = (g8 < G && s0 + 1 < nslot) ? wsa[g8 * nslot + s0 + 1] : 0.f;
                bb[hf] = pack_bf16(w0, w1);
            }
            mma_16816(pv, a, bb[0], bb[1]);
        }
    }
    __syncthreads();   // all reads of V in the buffer are done: partial outputs take its place
    float *red = reinterpret_cast<float *>(buf);
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
        *reinterpret_cast<float4 *>(red + ((size_t)part * G + hh) * D + 4 * c4) =
            make_float4(acc[hh][0].x, acc[hh][0].y, acc[hh][1].x, acc[hh][1].y);
    {
        // pv[2 hf + e]: dim 16 mt + g8 + 8 hf, head 2 t4 + e
        const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int hh = 2 * t4 + e2;
                if (hh < G) red[((size_t)(RG + kp) * G + hh) * D + 16 * mt + g8 + 8 * hf] = pv[2 * hf + e2];
            }
    }
    __syncthreads();
    // the parts below RG hold the linear numerator (state readout and linear keys), the
    // others the softmax one; the gated layer scales the linear numerator by sigmoid(gate)
    for (int i = tid; i < G * D; i += DS_THREADS) {
        const int hh = i / D, c = i % D;
        const size_t oi = ((size_t)b * dm.Hq + (size_t)g * G + hh) * D + c;
        float lin = 0.f, sm = 0.f;
        for (int p2 = 0; p2 < RG; ++p2) lin += red[((size_t)p2 * G + hh) * D + c];
        for (int p2 = RG; p2 < RG + KSPLIT; ++p2) sm += red[((size_t)p2 * G + hh) * D + c];
        const float gch = gate_t ? 1.f / (1.f + expf(-bf2f(gate_t[oi]))) : 1.f;
        const float num = fmaf(gch, lin, sm);
        const float den = s_den[hh];
        out_t[oi] = f2bf(den != 0.f ? num / den : 0.f);
    }

    // ---- state: the new candidate's slot, then t into the window ring --------------
    if (s_cand_slot >= 0) {
        const int sl = s_cand_slot;
        for (int x = tid; x < D; x += DS_THREADS) {
            K[(size_t)sl * D + x] = K[(size_t)tslot * D + x];
            V[(size_t)sl * D + x] = V[(size_t)tslot * D + x];
        }
        if (tid == 0) {
            pos[sl] = (int32_t)e;
            cnt[sl] = s_cand_count;
            ssc[sl] = ring[e % C];
        }
    }
    __syncthreads();
    if (W > 0) {
        for (int x = tid; x < D; x += DS_THREADS) {
            K[(size_t)tslot * D + x] = k_t[ug * D + x];
            V[(size_t)tslot * D + x] = v_t[ug * D + x];
        }
        if (tid == 0) pos[tslot] = (int32_t)t;
    }
    __syncthreads();

    // ---- (6) the chunk of t is complete: keep its top-lambda for good ----------------
    if (selecting && (t + 1) % C == 0) {
        const long long base = ct * C;
        const bool staged = C <= 4096;
        float *rs = reinterpret_cast<float *>(buf);
        int *win = reinterpret_cast<int *>(buf) + (staged ? C : 0);
        if (staged)
            for (int i = tid; i < C; i += DS_THREADS) rs[i] = ring[i];
        __syncthreads();
        const float *src = staged ? rs : ring;
        for (int i = tid; i < C; i += DS_THREADS) {
            const float si = src[i];
            int rank = 0;
            for (int j = 0; j < C && rank < lam; ++j)
                if (j != i && outranks(base + j, src[j], base + i, si)) ++rank;
            if (rank < lam) win[atomicAdd(&s_nwin, 1)] = i;
        }
        __syncthreads();
        if (warp == 0) {
            const int nw = s_nwin;
            for (int r = 0; r < nw; ++r) {
                const long long w = base + win[r];
                if (w <= t - W) {
                    bool found = false;
                    for (int x = 0; x < lam; ++x) found |= pos[W + ct * lam + x] == w;
                    if (!found && lane == 0) set_status(st.status, STILL_ERR_BOUNDS);
                    continue;
                }
                int target = -1;
                for (int x = 0; x < lam && target < 0; ++x)
                    if (pos[W + ct * lam + x] < 0) target = W + (int)ct * lam + x;
                if (target < 0) {
                    if (lane == 0) set_status(st.status, STILL_ERR_BOUNDS);
                    continue;
                }
                const int srcs = (int)(w % W);
                for (int x = lane; x < D; x += 32) {
                    K[(size_t)target * D + x] = K[(size_t)srcs * D + x];
                    V[(size_t)target * D + x] = V[(size_t)srcs * D + x];
                }
                __syncwarp();
                if (lane == 0) {
                    pos[target] = (int32_t)w;
                    ssc[target] = src[win[r]];
                }
                __syncwarp();
            }
            for (int x = lane; x < lam; x += 32) cnt[W + ct * lam + x] = 0;
        }
    }
    if (tid == 0) st.t[ug] = t + 1;
}

namespace {
// Tensor maps over the decode state's K and V ([B*Hkv*m, d] bf16), reused
// while the state's buffers stay the same.
struct DecodeMaps {
    const void *K = nullptr, *V = nullptr;
    uint64_t rows = 0;
    int d = 0;
    CUtensorMap mk, mv;
};
std::mutex g_map_mu;
DecodeMaps g_maps[8];
int g_map_next = 0;

bool decode_maps(const Dims &dm, const still_decode_state &st, CUtensorMap &mk, CUtensorMap &mv)
{
    const uint64_t rows = (uint64_t)dm.B * dm.Hkv * dm.m;
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (auto &c : g_maps)
        if (c.K == st.K && c.V == st.V && c.rows == rows && c.d == dm.d) {
            mk = c.mk;
            mv = c.mv;
            return true;
        }
    DecodeMaps n;
    n.K = st.K;
    n.V = st.V;
    n.rows = rows;
    n.d = dm.d;
    const uint64_t dims[2] = {(uint64_t)dm.d, rows};
    const uint64_t strides[1] = {(uint64_t)dm.d * 2};
    const uint32_t box[2] = {64, (uint32_t)DS_BOX_ROWS};
    if (!make_tma_map(&n.mk, st.K, 2, dims, strides, box, true)) return false;
    if (!make_tma_map(&n.mv, st.V, 2, dims, strides, box, true)) return false;
    g_maps[g_map_next] = n;
    g_map_next = (g_map_next + 1) % 8;
    mk = n.mk;
    mv = n.mv;
    return true;
}

constexpr size_t DS_SMEM_LIMIT = 200 * 1024;

bool staged_ok(const Dims &dm, const still_decode_state &st)
{
    const DecodeSmem L = decode_smem(dm);
    if (L.total > DS_SMEM_LIMIT || (dm.G != 1 && dm.G != 2 && dm.G != 4 && dm.G != 8)) return false;
    if (L.nslot == 0) return true;
    return (reinterpret_cast<uintptr_t>(st.K) & 15) == 0 && (reinterpret_cast<uintptr_t>(st.V) & 15) == 0 &&
           (uint64_t)dm.B * dm.Hkv * dm.m < (1ull << 31);
}
}  // namespace

cudaError_t launch_decode(const Dims &dm, const still_decode_state &st, const uint16_t *q_t, const uint16_t *k_t,
                          const uint16_t *v_t, const float *Wf, uint16_t *out_t, cudaStream_t s, const uint16_t *gate_t)
{
    KTimer tm(gate_t ? "decode_step_gated" : "decode_step", s);
    dim3 grid(dm.Hkv, dm.B);
    cudaError_t e;
    if (gate_t && !staged_ok(dm, st)) return cudaErrorNotSupported;   // the gate is in the staged kernel only
    if (staged_ok(dm, st)) {
        const DecodeSmem L = decode_smem(dm);
        CUtensorMap mk, mv;
        memset(&mk, 0, sizeof(mk));
        memset(&mv, 0, sizeof(mv));
        if (L.nslot > 0 && !decode_maps(dm, st, mk, mv)) return cudaErrorInvalidValue;
#define STILL_DECODE(DD, FF, GG)                                                                               \
    {                                                                                                          \
        static size_t set_bytes[64] = {};                                                                      \
        int dev = 0;                                                                                           \
        cudaGetDevice(&dev);                                                                                   \
        std::lock_guard<std::mutex> lk(g_map_mu);                                                              \
        if (dev < 0 || dev >= 64 || set_bytes[dev] < L.total) {                                                \
            e = cudaFuncSetAttribute(decode_kernel<DD, FF, GG>, cudaFuncAttributeMaxDynamicSharedMemorySize,     \
                                     (int)L.total);                                                            \
            if (e != cudaSuccess) return e;                                                                    \
            if (dev >= 0 && dev < 64) set_bytes[dev] = L.total;                                                \
        }                                                                                                      \
    }                                                                                                          \
    e = launch_kernel(decode_kernel<DD, FF, GG>, grid, dim3(DS_THREADS), L.total, s, mk, mv, st, q_t, k_t, v_t, Wf, dm, \
                      L, out_t, gate_t);
#define STILL_DECODE_G(DD, FF)                                                                                 \
    switch (dm.G) {                                                                                              \
    case 1: STILL_DECODE(DD, FF, 1) break;                                                                       \
    case 2: STILL_DECODE(DD, FF, 2) break;                                                                       \
    case 4: STILL_DECODE(DD, FF, 4) break;                                                                       \
    default: STILL_DECODE(DD, FF, 8) break;                                                                      \
    }
        if (dm.d == 64 && dm.df == 64) { STILL_DECODE_G(64, 64) }
        else if (dm.d == 64) { STILL_DECODE_G(64, 128) }
        else if (dm.df == 64) { STILL_DECODE_G(128, 64) }
        else { STILL_DECODE_G(128, 128) }
#undef STILL_DECODE_G
#undef STILL_DECODE
        return cudaGetLastError();
    }
    const DecodeGeneralSmem L = decode_general_smem(dm);
#define STILL_DECODE(DD, FF)                                                                                     \
    e = cudaFuncSetAttribute(decode_general_kernel<DD, FF>, cudaFuncAttributeMaxDynamicSharedMemorySize,         \
                             (int)L.total);                                                                      \
    if (e != cudaSuccess) return e;                                                                              \
    e = launch_kernel(decode_general_kernel<DD, FF>, grid, dim3(256), L.total, s, st, q_t, k_t, v_t, Wf, dm, L, out_t);
    if (dm.d == 64 && dm.df == 64) { STILL_DECODE(64, 64) }
    else if (dm.d == 64) { STILL_DECODE(64, 128) }
    else if (dm.df == 64) { STILL_DECODE(128, 64) }
    else { STILL_DECODE(128, 128) }
#undef STILL_DECODE
    return cudaGetLastError();
}

bool decode_staged(const Dims &dm, const still_decode_state &st) { return staged_ok(dm, st); }

// Shared memory of the variant that runs for these sizes (the general one when
// the staged plan does not fit); the caller rejects sizes above its limit.
size_t decode_smem_bytes(const Dims &dm)
{
    const DecodeSmem L = decode_smem(dm);
    if (L.total <= DS_SMEM_LIMIT && (dm.G == 1 || dm.G == 2 || dm.G == 4 || dm.G == 8)) return L.total;
    return decode_general_smem(dm).total;
}


// ---------------------------------------------------------------------------
// Export: the decode state after the N prefill tokens.
// ---------------------------------------------------------------------------
template <int D, int DF>
__global__ void __launch_bounds__(256) export_kernel(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                                                     const float *__restrict__ scores,
                                                     const int32_t *__restrict__ fsel,
                                                     const float *__restrict__ Ptot, const float *__restrict__ ztot,
                                                     size_t pstride, size_t zstride, Dims dm,
                                                     still_decode_state st)
{
    grid_dep_sync();
    const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const size_t ug = (size_t)b * dm.Hkv + g;
    const int W = dm.W, C = dm.C, lam = dm.lam, m = dm.m, N = dm.N;
    uint16_t *K = st.K + ug * m * D;
    uint16_t *V = st.V + ug * m * D;
    int32_t *pos = st.slot_pos + ug * m;
    int32_t *cnt = st.slot_cnt + ug * m;
    float *ssc = st.slot_score + ug * m;
    const uint16_t *kg = k + ug * (size_t)N * D;
    const uint16_t *vg = v + ug * (size_t)N * D;
    const float *sg = scores ? scores + ug * N : nullptr;
    const int32_t *fs = fsel + ug * dm.T_max * lam;

    // slot -> token
    for (int sl = tid; sl < m; sl += 256) {
        int j = -1, c_ = 0;
        float sc = 0.f;
        if (sl < W) {
            if (N - 1 >= sl) {
                j = sl + W * ((N - 1 - sl) / W);
            }
        } else if (sl < W + lam * dm.T_max) {
            const int c = (sl - W) / lam, r = (sl - W) % lam;
            if (c < dm.n_full) {
                j = fs[c * lam + r];
            } else if (c == dm.tail) {
                // candidates: tail-chunk winners that already left the window,
                // packed in ascending position
                int seen = 0;
                for (int x = 0; x < lam; ++x) {
                    const int jj = fs[c * lam + x];
                    if (jj >= 0 && jj <= N - 1 - W) {
                        if (seen == r) j = jj;
                        ++seen;
                    }
                }
                if (j >= 0) {
                    for (int i = c * C; i < N; ++i)
                        if (i != j && outranks(i, sg[i], j, sg[j])) ++c_;
                }
            }
            if (j >= 0 && sg) sc = sg[j];
        }
        pos[sl] = j;
        cnt[sl] = c_;
        ssc[sl] = sc;
    }
    __syncthreads();
    for (int sl = 0; sl < m; ++sl) {
        const int j = pos[sl];
        for (int x = tid; x < D; x += 256) {
            K[(size_t)sl * D + x] = j >= 0 ? kg[(size_t)j * D + x] : (uint16_t)0;
            V[(size_t)sl * D + x] = j >= 0 ? vg[(size_t)j * D + x] : (uint16_t)0;
        }
    }
    const float *P = Ptot + ug * pstride;
    const float *Z = ztot + ug * zstride;
    for (int i = tid; i < DF * D; i += 256) st.S[ug * DF * D + i] = P[i];
    for (int i = tid; i < DF; i += 256) st.z[ug * DF + i] = Z[i];
    for (int i = tid; i < C; i += 256) {
        float r = 0.f;
        if (dm.tail >= 0 && sg) {
            const int j = dm.tail * C + i;
            if (j < N) r = sg[j];
        }
        st.score_ring[ug * C + i] = r;
    }
    if (tid == 0) st.t[ug] = N;
}

cudaError_t launch_export(const Dims &dm, const SegPlan &sp, const uint16_t *k, const uint16_t *v,
                          const float *scores, const int32_t *fsel, const float *dS, const float *dz,
                          const still_decode_state &st, cudaStream_t s)
{
    KTimer tm("export_state", s);
    dim3 grid(dm.Hkv, dm.B);
    const size_t pstride = (size_t)(sp.nseg + 1) * dm.df * dm.d, zstride = (size_t)(sp.nseg + 1) * dm.df;
    const float *Pt = dS + (size_t)sp.nseg * dm.df * dm.d;
    const float *Zt = dz + (size_t)sp.nseg * dm.df;
    auto kern = dm.d == 64 ? (dm.df == 64 ? export_kernel<64, 64> : export_kernel<64, 128>)
                           : (dm.df == 64 ? export_kernel<128, 64> : export_kernel<128, 128>);
    const cudaError_t e = launch_kernel(kern, grid, dim3(256), 0, s, k, v, scores, fsel, Pt, Zt, pstride, zstride, dm, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace still
