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
#include "common.cuh"

namespace still {

namespace {
constexpr int FB = 8;   // folded keys staged per pass over S
constexpr int CB = 8;   // candidates handled per batch
constexpr int GMAX = 8; // query heads per kv head
}

struct DecodeSmem {
    int G, D, DF, nslot, lam, C;
    size_t off_qs, off_pq, off_kt, off_vt, off_hsc, off_w, off_sa, off_cand, off_fph, off_fv, off_fold, off_cph,
        off_ac, off_red, off_rs, off_win, total;
};

static DecodeSmem decode_smem(const Dims &dm)
{
    DecodeSmem L;
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
__global__ void __launch_bounds__(256) decode_kernel(still_decode_state st, const uint16_t *__restrict__ q_t,
                                                     const uint16_t *__restrict__ k_t,
                                                     const uint16_t *__restrict__ v_t, const float *__restrict__ Wf,
                                                     Dims dm, DecodeSmem L, uint16_t *__restrict__ out_t)
{
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

cudaError_t launch_decode(const Dims &dm, const still_decode_state &st, const uint16_t *q_t, const uint16_t *k_t,
                          const uint16_t *v_t, const float *Wf, uint16_t *out_t, cudaStream_t s)
{
    KTimer tm("decode_step", s);
    DecodeSmem L = decode_smem(dm);
    dim3 grid(dm.Hkv, dm.B);
    cudaError_t e;
#define STILL_DECODE(DD, FF)                                                                                   \
    e = cudaFuncSetAttribute(decode_kernel<DD, FF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total); \
    if (e != cudaSuccess) return e;                                                                            \
    decode_kernel<DD, FF><<<grid, 256, L.total, s>>>(st, q_t, k_t, v_t, Wf, dm, L, out_t);
    if (dm.d == 64 && dm.df == 64) { STILL_DECODE(64, 64) }
    else if (dm.d == 64) { STILL_DECODE(64, 128) }
    else if (dm.df == 64) { STILL_DECODE(128, 64) }
    else { STILL_DECODE(128, 128) }
#undef STILL_DECODE
    return cudaGetLastError();
}

size_t decode_smem_bytes(const Dims &dm) { return decode_smem(dm).total; }

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
    if (dm.d == 64 && dm.df == 64) export_kernel<64, 64><<<grid, 256, 0, s>>>(k, v, scores, fsel, Pt, Zt, pstride, zstride, dm, st);
    else if (dm.d == 64) export_kernel<64, 128><<<grid, 256, 0, s>>>(k, v, scores, fsel, Pt, Zt, pstride, zstride, dm, st);
    else if (dm.df == 64) export_kernel<128, 64><<<grid, 256, 0, s>>>(k, v, scores, fsel, Pt, Zt, pstride, zstride, dm, st);
    else export_kernel<128, 128><<<grid, 256, 0, s>>>(k, v, scores, fsel, Pt, Zt, pstride, zstride, dm, st);
    return cudaGetLastError();
}

}  // namespace still
