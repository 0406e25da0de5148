// Chunk-parallel backward pass of the layer, the routing (the kept set) held
// fixed: gradients of sum(dy * y) with respect to q, k, v and Wf.
//
// "STILL: Content-Aware Intra-Layer Hybrid Attention for Efficient LLM
// Linearization", sections "Content-Aware Routing with Fixed Budget" and
// "NP-Map: Norm-Preserving Feature Map" define the forward
//   y_t = (N_SA + phi(q_t)^T S_t) / (D_SA + phi(q_t).z_t),
//   N_SA = sum_SA p_tj v_j, D_SA = sum_SA p_tj, p_tj = e^{s_tj - c_t},
//   s_tj = q_t.k_j / sqrt(d), c_t = max_SA s_tj,
//   S_t = sum_LA phi(k_j) v_j^T, z_t = sum_LA phi(k_j),
// and its "Experiments" section trains through it.  With g_t = dy_t / D_t and
// delta_t = g_t . y_t (D_t the whole denominator):
//   softmax keys:  dp_tj = g_t.v_j - delta_t,  ds_tj = p_tj dp_tj,
//                  plus -sum_j ds_tj at the row-max key (c_t is part of the
//                  output: the linear terms are not scaled by it);
//                  dq_t += sum ds_tj k_j / sqrt(d), dk_j += ds_tj q_t / sqrt(d),
//                  dv_j += p_tj g_t
//   linear keys:   dphi(q_t) = S_t g_t - delta_t z_t,
//                  dphi(k_j) = R_j v_j - r_j,  dv_j += R_j^T phi(k_j),
//                  R_j = sum_{t : j in LA(t)} phi(q_t) g_t^T, r_j = sum delta_t phi(q_t)
//   NP-Map:        phi = ||x|| u/||u||, u = softmax(x Wf):
//                  dl = phi * (dphi - a phi/||x||), a = dphi.phi/||x||,
//                  dx = a x/||x|| + Wf dl, dWf += x dl^T
// (the softmax term <du, u> of the NP-Map's chain vanishes because u/||u|| has
// unit norm).  A kept key is a softmax key of the queries of later chunks
// outside its window; when W < C it is also a linear key of the later queries
// of its own chunk (t >= j + W) until that chunk completes.
//
// Passes (one sequence and kv head per unit, states at 32-token blocks):
//   mark_kept, phik     each key's kept-table entry, phi(k) (kept rows zero in
//                       the key table, kept in a table of their own)
//   blocksum, scan      S, z before every 32-key block (forward state)
//   query               per 16-row warp tile: c, P V, the linear branch, y,
//                       g, delta, dP, dS, dq (complete, NP-Map included)
//   blocksum, scan      R, r after every 32-token block (reverse state)
//   key                 per 16-key warp tile: dk, dv from the window queries
//                       and, for unkept keys, the linear branch (NP-Map included)
//   kept                dk, dv of the kept keys from the queries of later
//                       chunks outside their window (atomic adds)
//   kept_lin (W < C)    the kept keys as linear keys of their own chunk,
//                       with their NP-Map backward (atomic adds)
//   dwf                 dWf = sum over q and k rows of x dl^T
// The contractions run as warp MMAs (bf16 operands, fp32 accumulation).
#include <climits>

#include "common.cuh"
#include "warp_mma.cuh"

namespace still {

__global__ void scan_kernel(float *__restrict__ dS, float *__restrict__ dz, int nseg, int nel_s, int nel_z);

namespace {

using namespace wmma16;

constexpr int BT = 32;             // tokens per state block

struct BwdArgs {
    Dims dm;
    int nblk;            // state blocks: ceil(N / BT)
    float scale;         // 1 / sqrt(d)
    const uint16_t *q, *k, *v, *dy;
    const float *Wf;
    const int32_t *sel;  // [B, Hkv, T_max * lam]
    const int32_t *kslot; // [B, Hkv, N]: the kept-table entry of a kept key, else -1
    const uint16_t *phk; // [B, Hkv, N, DF], kept rows zero
    const uint16_t *phkk; // [B, Hkv, T_max * lam, DF]: phi(k) of the kept entries (bf16)
    const float *phkk32;  // the same in fp32
    const float *Sp, *zp;   // [units][nblk + 1][DF * D], [units][nblk + 1][DF]: state before block i
    const float *Rs, *rs;   // the same layout, reversed blocks: index nblk - i holds the sums over t >= BT i
    uint16_t *g, *phq;               // g = dy / den (bf16, for the reverse state), phi(q) [B, Hq, N, *]
    float *phq32, *phk32;            // phi(q), phi(k) in fp32 (for the NP-Map backward)
    float *dlq, *dlk;                // dl of the q rows [B, Hq, N, DF] and of the k rows [B, Hkv, N, DF]
    float *rc, *rdelta, *rds, *rinv; // per query row: c, delta, sum of its softmax ds, 1 / den
    int32_t *rjs;                    // per query row: the key position of c
    float *dq, *dk, *dv, *dWf;
    int32_t *cidx;                   // nullable copy of rjs for the caller
};

__device__ __forceinline__ uint32_t ld_pair(const uint16_t *row, int col) { return *reinterpret_cast<const uint32_t *>(row + col); }

// 16-byte rows of a bf16 tile: rows [0, nrows) of `src` (rows of `width` elements,
// `valid(r)` false -> zero row) into a shared tile of stride `ld`, by all threads.
template <int WIDTH, typename RowPtr>
__device__ __forceinline__ void stage_rows(uint16_t *dst, int ld, int nrows, RowPtr rowptr)
{
    constexpr int V = WIDTH / 8;
    for (int i = threadIdx.x; i < nrows * V; i += blockDim.x) {
        const int r = i / V, c = i % V;
        const uint16_t *src = rowptr(r);
        uint4 x = make_uint4(0, 0, 0, 0);
        if (src) x = __ldg(reinterpret_cast<const uint4 *>(src) + c);
        *reinterpret_cast<uint4 *>(dst + r * ld + c * 8) = x;
    }
}

// fp32 [rows][cols] global -> bf16 shared tile of stride ld
__device__ __forceinline__ void stage_f32(uint16_t *dst, int ld, const float *src, int rows, int cols)
{
    const int n4 = rows * cols / 4;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const int r = i / (cols / 4), c = (i % (cols / 4)) * 4;
        const float4 x = __ldg(reinterpret_cast<const float4 *>(src + (size_t)r * cols + c));
        uint2 p;
        p.x = pack(x.x, x.y);
        p.y = pack(x.z, x.w);
        *reinterpret_cast<uint2 *>(dst + r * ld + c) = p;
    }
}

// ---------------------------------------------------------------------------
// kept flags and phi(k)
// ---------------------------------------------------------------------------
__global__ void mark_kept_kernel(const int32_t *__restrict__ sel, int KP, int N, int32_t *__restrict__ kslot)
{
    grid_dep_sync();
    const int unit = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= KP) return;
    const int p = sel[(size_t)unit * KP + e];
    if (p >= 0 && p < N) kslot[(size_t)unit * N + p] = e;
}

// ---------------------------------------------------------------------------
// block sums of outer products: out[f][d] = sum_rows a[row][f] b[row][d],
// zo[f] = sum_rows w[row] a[row][f], for the rows of one 32-token block
// (forward: the block's keys, a = phi(k), b = v, w = 1; reverse: the block's
// tokens x the group's heads, a = phi(q), b = g, w = delta; stored reversed)
// ---------------------------------------------------------------------------
template <int D, int DF>
struct BSLayout {
    static constexpr int LDA = DF + 8, LDB = D + 8, ROWS = 4 * BT;
    static constexpr int A = 0, B = A + ROWS * LDA * 2, W = B + ROWS * LDB * 2, TOTAL = W + ROWS * 4;
};

template <int D, int DF, bool REV>
__global__ void __launch_bounds__(256) blocksum_kernel(BwdArgs P, float *__restrict__ out, float *__restrict__ zo)
{
    grid_dep_sync();
    using L = BSLayout<D, DF>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *sa = (uint16_t *)(smem + L::A), *sb = (uint16_t *)(smem + L::B);
    float *sw = (float *)(smem + L::W);
    const Dims &dm = P.dm;
    const int blk = blockIdx.x, unit = blockIdx.y, b = unit / dm.Hkv, gq = unit % dm.Hkv;
    const int G = REV ? dm.G : 1;
    const int rows = BT * G;   // row r: head r / BT, token blk * BT + r % BT
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto tok = [&](int r) { return blk * BT + r % BT; };
    auto base_row = [&](int r) -> size_t {
        return REV ? ((size_t)(b * dm.Hq + gq * dm.G + r / BT) * dm.N + tok(r)) : ((size_t)unit * dm.N + tok(r));
    };
    const uint16_t *ga = REV ? P.phq : P.phk;
    const uint16_t *gb = REV ? P.g : P.v;
    stage_rows<DF>(sa, L::LDA, rows, [&](int r) -> const uint16_t * {
        return tok(r) < dm.N ? ga + base_row(r) * DF : nullptr;
    });
    stage_rows<D>(sb, L::LDB, rows, [&](int r) -> const uint16_t * {
        return tok(r) < dm.N ? gb + base_row(r) * D : nullptr;
    });
    for (int r = threadIdx.x; r < rows; r += blockDim.x)
        sw[r] = tok(r) < dm.N ? (REV ? P.rdelta[base_row(r)] : 1.f) : 0.f;
    __syncthreads();
    const int slot = REV ? P.nblk - 1 - blk : blk;
    float *o = out + ((size_t)unit * (P.nblk + 1) + slot) * DF * D;
    if (warp < DF / 16) {
        constexpr int NT = D / 8;
        float acc[NT][4];
        zero(acc);
        for (int k0 = 0; k0 < rows; k0 += 16) {
            uint32_t a[1][4];
            load_a_t(sa, L::LDA, warp * 16, k0, a[0]);   // A(m = f, k = row) from [row][f]
            mma_tile<1, NT, true>(acc, a, sb, L::LDB, 0, k0);
        }
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + 2 * tig;
            *reinterpret_cast<float2 *>(o + (size_t)(warp * 16 + gid) * D + col) = make_float2(acc[nt][0], acc[nt][1]);
            *reinterpret_cast<float2 *>(o + (size_t)(warp * 16 + gid + 8) * D + col) = make_float2(acc[nt][2], acc[nt][3]);
        }
    }
    for (int f = threadIdx.x; f < DF; f += blockDim.x) {
        float s = 0.f;
        for (int r = 0; r < rows; ++r) s = fmaf(sw[r], bf2f(sa[r * L::LDA + f]), s);
        zo[((size_t)unit * (P.nblk + 1) + slot) * DF + f] = s;
    }
}

// ---------------------------------------------------------------------------
// query pass
// ---------------------------------------------------------------------------
constexpr int BQ8_THREADS = 256;   // the query pass: eight warps of 16 rows
constexpr int KEPT_MAX = 1024;     // kept positions of a CTA held in shared memory (more: read from global)
constexpr int PKEEP = 10;          // key blocks whose P the query pass keeps for its second pass

__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// NP-Map of a warp's 16 rows x (A fragments xa, bf16): U = x Wf with Wf as a bf16
// pair (hi, lo: shared tiles [d][df]), u = softmax(U), phi = ||x|| u / ||u|| into
// phi (accumulator layout), ||x|| of the thread's two rows into nx.
template <int D>
__device__ __forceinline__ void warp_npmap_rows(const uint32_t (&xa)[D / 16][4], const uint16_t *wf_hi,
                                                const uint16_t *wf_lo, float (&phi)[D / 8][4], float (&nx)[2])
{
    constexpr int LD = D + 8, KC = D / 16, NT = D / 8;
    zero(phi);
    mma_tile<KC, NT, true>(phi, xa, wf_hi, LD, 0, 0);
    mma_tile<KC, NT, true>(phi, xa, wf_lo, LD, 0, 0);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mx = fmaxf(mx, fmaxf(phi[nt][2 * r], phi[nt][2 * r + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        float s2 = 0.f, x2 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            phi[nt][2 * r] = expf(phi[nt][2 * r] - mx);
            phi[nt][2 * r + 1] = expf(phi[nt][2 * r + 1] - mx);
            s2 = fmaf(phi[nt][2 * r], phi[nt][2 * r], fmaf(phi[nt][2 * r + 1], phi[nt][2 * r + 1], s2));
        }
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
            const uint32_t a0 = xa[kc][r], a1 = xa[kc][r + 2];
            x2 = fmaf(lo_f(a0), lo_f(a0), fmaf(hi_f(a0), hi_f(a0), x2));
            x2 = fmaf(lo_f(a1), lo_f(a1), fmaf(hi_f(a1), hi_f(a1), x2));
        }
        s2 = quad_sum(s2);
        x2 = quad_sum(x2);
        nx[r] = sqrtf(x2);
        const float sc = s2 > 0.f ? nx[r] * rsqrtf(s2) : 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            phi[nt][2 * r] *= sc;
            phi[nt][2 * r + 1] *= sc;
        }
    }
}

// Wf [d][df] fp32 -> two shared bf16 tiles hi = bf16(Wf), lo = bf16(Wf - hi)
template <int D>
__device__ __forceinline__ void stage_wf_pair(const float *__restrict__ Wf, uint16_t *hi, uint16_t *lo)
{
    constexpr int LD = D + 8;
    for (int i = threadIdx.x; i < D * D / 4; i += blockDim.x) {
        const int r = i / (D / 4), c = (i % (D / 4)) * 4;
        const float4 x = __ldg(reinterpret_cast<const float4 *>(Wf) + i);
        const uint32_t h0 = pack(x.x, x.y), h1 = pack(x.z, x.w);
        *reinterpret_cast<uint2 *>(hi + r * LD + c) = make_uint2(h0, h1);
        *reinterpret_cast<uint2 *>(lo + r * LD + c) =
            make_uint2(pack(x.x - lo_f(h0), x.y - hi_f(h0)), pack(x.z - lo_f(h1), x.w - hi_f(h1)));
    }
}

// phi(k) of 128 key rows per CTA (eight warps of 16 rows) on warp MMAs, fp32 and
// bf16 copies, kept keys' rows zero
template <int D>
__global__ void __launch_bounds__(256) phik_mma_kernel(BwdArgs A, uint16_t *__restrict__ phk, float *__restrict__ phk32,
                                                       uint16_t *__restrict__ phkk, float *__restrict__ phkk32)
{
    grid_dep_sync();
    constexpr int LD = D + 8, KC = D / 16, NT = D / 8;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *hi = (uint16_t *)smem, *lo = hi + D * LD;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const long long rows = (long long)A.dm.B * A.dm.Hkv * A.dm.N;
    const long long r0 = (long long)blockIdx.x * 128 + warp * 16;
    stage_wf_pair<D>(A.Wf, hi, lo);
    __syncthreads();
    const long long rr[2] = {r0 + gid, r0 + gid + 8};
    uint32_t xa[KC][4];
#pragma unroll
    for (int kc = 0; kc < KC; ++kc)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const long long row = rr[i & 1];
            xa[kc][i] = row < rows ? ld_pair(A.k + row * D, 16 * kc + 8 * (i >> 1) + 2 * tig) : 0u;
        }
    float ph[NT][4], nx[2];
    warp_npmap_rows<D>(xa, hi, lo, ph, nx);
    const int KP = A.dm.T_max * A.dm.lam;
#pragma unroll
    for (int r = 0; r < 2; ++r)
        if (rr[r] < rows) {
            const int e = A.kslot[rr[r]];
            const bool kp = e >= 0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float a = kp ? 0.f : ph[nt][2 * r], b = kp ? 0.f : ph[nt][2 * r + 1];
                *reinterpret_cast<uint32_t *>(phk + rr[r] * D + nt * 8 + 2 * tig) = pack(a, b);
                *reinterpret_cast<float2 *>(phk32 + rr[r] * D + nt * 8 + 2 * tig) = make_float2(a, b);
            }
            if (kp) {   // the kept entry's own features, unmasked
                const size_t kr = ((size_t)(rr[r] / A.dm.N) * KP + e) * D;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    *reinterpret_cast<uint32_t *>(phkk + kr + nt * 8 + 2 * tig) = pack(ph[nt][2 * r], ph[nt][2 * r + 1]);
                    *reinterpret_cast<float2 *>(phkk32 + kr + nt * 8 + 2 * tig) = make_float2(ph[nt][2 * r], ph[nt][2 * r + 1]);
                }
            }
        }
}

template <int D>
struct QLayout {
    static constexpr int LD = D + 8, T32 = BT * LD * 2;
    static constexpr int K = 0, V = K + 2 * T32, PK = V + 2 * T32, VL = PK + T32;   // K, V: two buffers each
    static constexpr int WF = VL + T32;            // Wf [d][df] bf16
    static constexpr int SP = WF + D * LD * 2;     // S before the lag keys, [df][d] bf16
    static constexpr int ZP = SP + D * LD * 2;     // z, fp32 [df]
    static constexpr int POS = ZP + D * 4;         // positions of the two staged key blocks and of the lag block
    static constexpr int KEPT = POS + 3 * BT * 4;  // the CTA's kept positions
    // pass 1's P of the first PKEEP key blocks, per warp in A-fragment order
    // ([block][register][lane] uint32: bf16 pairs), and the running maximum each
    // block's P was taken against ([block][row] fp32)
    static constexpr int PST = KEPT + KEPT_MAX * 4;
    static constexpr int MST = PST + 8 * PKEEP * 8 * 32 * 4;
    static constexpr int TOTAL = MST + 8 * PKEEP * 16 * 4;
};

// The thread's two accumulator rows are gid and gid + 8; element (nt, 2r + e)
// of an accumulator is (row gid + 8r, column 8nt + 2tig + e).  Eight warps: G
// heads x 8/G token tiles of 16.
template <int D, int G>
__global__ void __launch_bounds__(BQ8_THREADS, 1) query_kernel(BwdArgs P)
{
    grid_dep_sync();
    constexpr int LD = D + 8, KC = D / 16, NT = D / 8;
    constexpr int TOK = 16 * (8 / G);   // tokens per CTA
    constexpr int T32E = BT * LD;       // elements of one 32-row tile
    constexpr float LOG2E = 1.4426950408889634f;
    using L = QLayout<D>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *sKb = (uint16_t *)(smem + L::K), *sVb = (uint16_t *)(smem + L::V);
    uint16_t *sPK = (uint16_t *)(smem + L::PK), *sVL = (uint16_t *)(smem + L::VL);
    uint16_t *sWF = (uint16_t *)(smem + L::WF), *sSP = (uint16_t *)(smem + L::SP);
    float *sZ = (float *)(smem + L::ZP);
    int *sPosb = (int *)(smem + L::POS), *sLag = sPosb + 2 * BT;
    int *sKept = (int *)(smem + L::KEPT);

    const Dims &dm = P.dm;
    const int N = dm.N, W = dm.W, C = dm.C;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
    uint32_t *sPst = (uint32_t *)(smem + L::PST) + (size_t)warp * PKEEP * 8 * 32;
    float *sMst = (float *)(smem + L::MST) + (size_t)warp * PKEEP * 16;
    const int unit = blockIdx.y, b = unit / dm.Hkv, gq = unit % dm.Hkv;
    const int t0 = blockIdx.x * TOK;
    const int h = gq * G + warp % G;
    const int tw = t0 + 16 * (warp / G);
    const int tr[2] = {tw + gid, tw + gid + 8};
    const size_t qrow0 = (size_t)(b * dm.Hq + h) * N;
    const size_t krow0 = (size_t)unit * N;
    const float scale = P.scale;

    // ---- Wf as a bf16 pair hi (sWF, resident) + lo (in the S region until S is staged):
    // U = q Wf to about 16 significant bits of Wf
    stage_wf_pair<D>(P.Wf, sWF, sSP);
    // the linear state before the lag keys: keys < BT * i0
    const int i0 = t0 - W > 0 ? (t0 - W) / BT : 0;
    const int lag0 = BT * i0, lag1 = min(t0 + TOK - W, N);   // lag keys [lag0, lag1)
    const int nlag = lag1 > lag0 ? (lag1 - lag0 + BT - 1) / BT : 0;
    for (int f = tid; f < D; f += BQ8_THREADS) sZ[f] = P.zp[((size_t)unit * (P.nblk + 1) + i0) * D + f];
    // the softmax keys: kept keys of chunks before the last row's, then the band
    const int tlast = min(t0 + TOK, N) - 1;
    const int KP = dm.T_max * dm.lam;
    const int nk = dm.lam * min(tlast / C, dm.T_max);
    const int nkb = (nk + BT - 1) / BT;
    const int bs = max(t0 - W + 1, 0), be = tlast + 1;
    const int nblk = nkb + (be - bs + BT - 1) / BT;
    const int32_t *selu = P.sel + (size_t)unit * KP;
    for (int e = tid; e < min(nk, KEPT_MAX); e += BQ8_THREADS) {
        const int p = selu[e];
        sKept[e] = p < N ? p : -1;
    }

    uint32_t qa[KC][4];
    {
        const uint16_t *r0 = P.q + (qrow0 + tr[0]) * D, *r1 = P.q + (qrow0 + tr[1]) * D;
        const bool v0 = tr[0] < N, v1 = tr[1] < N;
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
            qa[kc][0] = v0 ? ld_pair(r0, 16 * kc + 2 * tig) : 0u;
            qa[kc][1] = v1 ? ld_pair(r1, 16 * kc + 2 * tig) : 0u;
            qa[kc][2] = v0 ? ld_pair(r0, 16 * kc + 8 + 2 * tig) : 0u;
            qa[kc][3] = v1 ? ld_pair(r1, 16 * kc + 8 + 2 * tig) : 0u;
        }
    }
    __syncthreads();

    auto key_pos = [&](int blk, int i) -> int {
        if (blk < nkb) {
            const int e = blk * BT + i;
            if (e >= nk) return -1;
            if (e < KEPT_MAX) return sKept[e];
            const int p = selu[e];
            return p < N ? p : -1;
        }
        const int p = bs + (blk - nkb) * BT + i;
        return p < be ? p : -1;
    };
    // key block blk into buffer buf (K, and V when with_v) by cp.async, one commit group
    auto issue = [&](int blk, int buf, bool with_v) {
        int *pos = sPosb + buf * BT;
        for (int i = tid; i < BT; i += BQ8_THREADS) pos[i] = key_pos(blk, i);
        constexpr int V8 = D / 8, NE = BT * V8;
        for (int i = tid; i < NE * (with_v ? 2 : 1); i += BQ8_THREADS) {
            const int which = i / NE, j = i % NE, r = j / V8, c = j % V8;
            const int p = key_pos(blk, r);
            const uint16_t *src = (which ? P.v : P.k) + (krow0 + (p >= 0 ? p : 0)) * D + c * 8;
            cp_async16((which ? sVb : sKb) + buf * T32E + r * LD + c * 8, src, p >= 0 ? 16 : 0);
        }
        cp_commit();
    };
    // for each key block: wait for its copies, run body(buf), prefetch the next one
    auto key_loop = [&](bool with_v, auto body) {
        issue(0, 0, with_v);
        for (int blk = 0; blk < nblk; ++blk) {
            const int buf = blk & 1;
            if (blk + 1 < nblk) {
                issue(blk + 1, buf ^ 1, with_v);
                cp_wait<1>();
            } else {
                cp_wait<0>();
            }
            __syncthreads();
            body(blk, buf);
            __syncthreads();
        }
    };
    // the first token of each row's chunk: a kept key of an earlier chunk lies below it
    // (with W >= C every key at or before t - W does)
    const int tcs[2] = {tr[0] - tr[0] % C, tr[1] - tr[1] % C};
    auto in_sa = [&](int r, int p, bool kept_blk) -> bool {
        const int t = tr[r];
        if (p < 0 || t >= N) return false;
        if (kept_blk) return p <= t - W && p < tcs[r];
        return p <= t && p > t - W;
    };
    auto logits = [&](float (&s)[4][4], int buf) {
        zero(s);
        mma_tile<KC, 4, false>(s, qa, sKb + buf * T32E, LD, 0, 0);
    };

    // ---- NP-Map of the query rows: u = softmax(q Wf), phi = ||q|| u / ||u||
    float nq[2];
    uint32_t pa[KC][4];
    {
        float u[NT][4];
        warp_npmap_rows<D>(qa, sWF, sSP, u, nq);
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (tr[r] < N) {
                uint16_t *dst = P.phq + (qrow0 + tr[r]) * D;
                float *d32 = P.phq32 + (qrow0 + tr[r]) * D;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    *reinterpret_cast<uint32_t *>(dst + nt * 8 + 2 * tig) = pack(u[nt][2 * r], u[nt][2 * r + 1]);
                    *reinterpret_cast<float2 *>(d32 + nt * 8 + 2 * tig) = make_float2(u[nt][2 * r], u[nt][2 * r + 1]);
                }
            }
        acc_to_a<NT>(u, pa);
    }
    // the linear state before the lag keys replaces Wf's low part
    __syncthreads();
    stage_f32(sSP, LD, P.Sp + ((size_t)unit * (P.nblk + 1) + i0) * D * D, D, D);
    __syncthreads();

    // pass 1: O = P V and D_SA = sum P with a running row maximum (O and the sums
    // rescaled when it grows); at the end it is c, the exact row maximum, and the
    // lowest position among equal maxima holds it
    float o[NT][4];
    zero(o);
    float dsa[2] = {0.f, 0.f};
    float mrun[2] = {-INFINITY, -INFINITY};
    float cm[2] = {-INFINITY, -INFINITY};
    int cj[2] = {INT_MAX, INT_MAX};
    key_loop(true, [&](int blk, int buf) {
        const int *pos = sPosb + buf * BT;
        float s[4][4];
        logits(s, buf);
        const bool kb = blk < nkb;
        float bm[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int p = pos[nt * 8 + 2 * tig + e];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const bool in = in_sa(r, p, kb);
                    const float x = in ? s[nt][2 * r + e] * scale : -INFINITY;
                    s[nt][2 * r + e] = x;
                    bm[r] = fmaxf(bm[r], x);
                    if (in && (x > cm[r] || (x == cm[r] && p < cj[r]))) {
                        cm[r] = x;
                        cj[r] = p;
                    }
                }
            }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            bm[r] = fmaxf(bm[r], __shfl_xor_sync(0xffffffffu, bm[r], 1));
            bm[r] = fmaxf(bm[r], __shfl_xor_sync(0xffffffffu, bm[r], 2));
            if (bm[r] > mrun[r]) {
                const float f = mrun[r] == -INFINITY ? 0.f : expf(mrun[r] - bm[r]);
                dsa[r] *= f;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    o[nt][2 * r] *= f;
                    o[nt][2 * r + 1] *= f;
                }
                mrun[r] = bm[r];
            }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float x = s[nt][2 * r + e];
                    const float pe = x == -INFINITY ? 0.f : exp2_mufu((x - mrun[r]) * LOG2E);
                    s[nt][2 * r + e] = pe;
                    dsa[r] += pe;
                }
        uint32_t pf[2][4];
        acc_to_a<4>(s, pf);
        if (blk < PKEEP) {
#pragma unroll
            for (int i = 0; i < 8; ++i) sPst[(blk * 8 + i) * 32 + lane] = pf[i >> 2][i & 3];
            if (tig == 0) {
                sMst[blk * 16 + gid] = mrun[0];
                sMst[blk * 16 + gid + 8] = mrun[1];
            }
        }
        mma_tile<2, NT, true>(o, pf, sVb + buf * T32E, LD, 0, 0);
    });
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int sh = 1; sh <= 2; sh <<= 1) {
            const float x = __shfl_xor_sync(0xffffffffu, cm[r], sh);
            const int p = __shfl_xor_sync(0xffffffffu, cj[r], sh);
            if (x > cm[r] || (x == cm[r] && p < cj[r])) {
                cm[r] = x;
                cj[r] = p;
            }
        }

    // ---- the linear branch: phi(q) S + the lag keys [lag0, t - W]
    mma_tile<KC, NT, true>(o, pa, sSP, LD, 0, 0);
    float dlin[2] = {0.f, 0.f};
    {
        float ph[NT][4];   // phi back from its bf16 copy (the MMA operand)
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
            ph[2 * kc][0] = lo_f(pa[kc][0]); ph[2 * kc][1] = hi_f(pa[kc][0]);
            ph[2 * kc][2] = lo_f(pa[kc][1]); ph[2 * kc][3] = hi_f(pa[kc][1]);
            ph[2 * kc + 1][0] = lo_f(pa[kc][2]); ph[2 * kc + 1][1] = hi_f(pa[kc][2]);
            ph[2 * kc + 1][2] = lo_f(pa[kc][3]); ph[2 * kc + 1][3] = hi_f(pa[kc][3]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float z = sZ[nt * 8 + 2 * tig + e];
                dlin[0] = fmaf(ph[nt][e], z, dlin[0]);
                dlin[1] = fmaf(ph[nt][2 + e], z, dlin[1]);
            }
    }
    // linear keys past the state: the lag keys [lag0, lag1) (kept keys are zero rows of the
    // feature table), then -- when W < C -- the kept entries of the rows' own chunks, which
    // stay linear keys until their chunk completes (blocks nlag .. nlag + nxb - 1)
    const int xc0 = t0 / C, xc1 = min(tlast / C, dm.T_max - 1);
    const int xe0 = xc0 * dm.lam, nx = W < C && dm.lam > 0 && xc1 >= xc0 ? (xc1 - xc0 + 1) * dm.lam : 0;
    const int nxb = (nx + BT - 1) / BT;
    auto stage_lag = [&](int lb) {
        const bool ex = lb >= nlag;
        __syncthreads();
        for (int i = threadIdx.x; i < BT; i += blockDim.x) {
            int p;
            if (!ex) {
                p = lag0 + lb * BT + i;
                p = p < lag1 ? p : -1;
            } else {
                const int e = (lb - nlag) * BT + i;
                p = e < nx ? selu[xe0 + e] : -1;
                p = p < N ? p : -1;
            }
            sLag[i] = p;
        }
        __syncthreads();
        stage_rows<D>(sPK, LD, BT, [&](int r) -> const uint16_t * {
            const int p = sLag[r];
            if (p < 0) return nullptr;
            return ex ? P.phkk + ((size_t)unit * KP + xe0 + (lb - nlag) * BT + r) * D : P.phk + (krow0 + p) * D;
        });
        stage_rows<D>(sVL, LD, BT, [&](int r) -> const uint16_t * {
            const int p = sLag[r];
            return p >= 0 ? P.v + (krow0 + p) * D : nullptr;
        });
        __syncthreads();
    };
    auto lin_key = [&](int r, int p, bool ex) -> bool {
        const int t = tr[r];
        return p >= 0 && t < N && p <= t - W && (!ex || p >= tcs[r]);
    };
    for (int lb = 0; lb < nlag + nxb; ++lb) {
        stage_lag(lb);
        const bool ex = lb >= nlag;
        float a[4][4];
        zero(a);
        mma_tile<KC, 4, false>(a, pa, sPK, LD, 0, 0);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int p = sLag[nt * 8 + 2 * tig + e];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const bool in = lin_key(r, p, ex);
                    const float x = in ? a[nt][2 * r + e] : 0.f;
                    a[nt][2 * r + e] = x;
                    dlin[r] += x;
                }
            }
        uint32_t af[2][4];
        acc_to_a<4>(a, af);
        mma_tile<2, NT, true>(o, af, sVL, LD, 0, 0);
    }

    // ---- y, g = dy / den, delta = g . y
    float den[2], inv[2], delta[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        den[r] = quad_sum(dsa[r]) + quad_sum(dlin[r]);
        inv[r] = den[r] != 0.f ? 1.f / den[r] : 0.f;
    }
    {
        float dd[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint16_t *dyr = P.dy + (qrow0 + tr[r]) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t pr = tr[r] < N ? ld_pair(dyr, nt * 8 + 2 * tig) : 0u;
                const float g0 = lo_f(pr) * inv[r], g1 = hi_f(pr) * inv[r];
                dd[r] = fmaf(g0, o[nt][2 * r] * inv[r], fmaf(g1, o[nt][2 * r + 1] * inv[r], dd[r]));
                o[nt][2 * r] = g0;
                o[nt][2 * r + 1] = g1;
            }
            delta[r] = quad_sum(dd[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
        if (tr[r] < N) {
            uint16_t *dst = P.g + (qrow0 + tr[r]) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<uint32_t *>(dst + nt * 8 + 2 * tig) = pack(o[nt][2 * r], o[nt][2 * r + 1]);
        }
    // dy itself (exact in bf16) is the MMA operand; 1/den scales the products
    uint32_t ya[KC][4];
    {
        const uint16_t *r0 = P.dy + (qrow0 + tr[0]) * D, *r1 = P.dy + (qrow0 + tr[1]) * D;
        const bool v0 = tr[0] < N, v1 = tr[1] < N;
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
            ya[kc][0] = v0 ? ld_pair(r0, 16 * kc + 2 * tig) : 0u;
            ya[kc][1] = v1 ? ld_pair(r1, 16 * kc + 2 * tig) : 0u;
            ya[kc][2] = v0 ? ld_pair(r0, 16 * kc + 8 + 2 * tig) : 0u;
            ya[kc][3] = v1 ? ld_pair(r1, 16 * kc + 8 + 2 * tig) : 0u;
        }
    }

    // pass 2: dP = g V^T = (dy V^T) / den, dS = P (dP - delta), dq = dS K
    const float scale_l2 = scale * LOG2E;
    const float cl2[2] = {cm[0] * LOG2E, cm[1] * LOG2E};
    float dq[NT][4];
    zero(dq);
    float dss[2] = {0.f, 0.f};
    key_loop(true, [&](int blk, int buf) {
        const int *pos = sPosb + buf * BT;
        float s[4][4], dp[4][4];
        zero(dp);
        mma_tile<KC, 4, false>(dp, ya, sVb + buf * T32E, LD, 0, 0);
        if (blk < PKEEP) {
            // P of pass 1 (bf16, masked keys zero), taken against the running maximum of
            // its block: rescaled to c
            float f[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float mb = sMst[blk * 16 + gid + 8 * r];
                f[r] = mb == -INFINITY ? 0.f : exp2_mufu((mb - cm[r]) * LOG2E);
            }
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
                const uint32_t w0 = sPst[(blk * 8 + kc * 4 + 0) * 32 + lane], w1 = sPst[(blk * 8 + kc * 4 + 1) * 32 + lane];
                const uint32_t w2 = sPst[(blk * 8 + kc * 4 + 2) * 32 + lane], w3 = sPst[(blk * 8 + kc * 4 + 3) * 32 + lane];
                s[2 * kc][0] = lo_f(w0) * f[0];
                s[2 * kc][1] = hi_f(w0) * f[0];
                s[2 * kc][2] = lo_f(w1) * f[1];
                s[2 * kc][3] = hi_f(w1) * f[1];
                s[2 * kc + 1][0] = lo_f(w2) * f[0];
                s[2 * kc + 1][1] = hi_f(w2) * f[0];
                s[2 * kc + 1][2] = lo_f(w3) * f[1];
                s[2 * kc + 1][3] = hi_f(w3) * f[1];
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float ds = s[nt][2 * r + e] * (dp[nt][2 * r + e] * inv[r] - delta[r]);
                        s[nt][2 * r + e] = ds;
                        dss[r] += ds;
                    }
        } else {
            logits(s, buf);
            const bool kb = blk < nkb;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int p = pos[nt * 8 + 2 * tig + e];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float pe = in_sa(r, p, kb) ? exp2_mufu(fmaf(s[nt][2 * r + e], scale_l2, -cl2[r])) : 0.f;
                        const float ds = pe * (dp[nt][2 * r + e] * inv[r] - delta[r]);
                        s[nt][2 * r + e] = ds;
                        dss[r] += ds;
                    }
                }
        }
        uint32_t sf[2][4];
        acc_to_a<4>(s, sf);
        mma_tile<2, NT, true>(dq, sf, sKb + buf * T32E, LD, 0, 0);
    });
    // the stabiliser's gradient at the row-max key, then the 1/sqrt(d) of the logits
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        dss[r] = quad_sum(dss[r]);
        const bool ok = tr[r] < N && cj[r] >= 0 && cj[r] < N;
        const uint16_t *kr = P.k + (krow0 + (ok ? cj[r] : 0)) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t pr = ok ? ld_pair(kr, nt * 8 + 2 * tig) : 0u;
            dq[nt][2 * r] = (dq[nt][2 * r] - dss[r] * lo_f(pr)) * scale;
            dq[nt][2 * r + 1] = (dq[nt][2 * r + 1] - dss[r] * hi_f(pr)) * scale;
        }
    }

    // ---- dphi(q) = S g - delta z + sum_lag phi(k) (g . v - delta)
    {
        float dph[NT][4];
        zero(dph);
        mma_tile<KC, NT, false>(dph, ya, sSP, LD, 0, 0);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float z = sZ[nt * 8 + 2 * tig + e];
                dph[nt][e] = dph[nt][e] * inv[0] - delta[0] * z;
                dph[nt][2 + e] = dph[nt][2 + e] * inv[1] - delta[1] * z;
            }
        for (int lb = 0; lb < nlag + nxb; ++lb) {
            stage_lag(lb);
            const bool ex = lb >= nlag;
            float da[4][4];
            zero(da);
            mma_tile<KC, 4, false>(da, ya, sVL, LD, 0, 0);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int p = sLag[nt * 8 + 2 * tig + e];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const bool in = lin_key(r, p, ex);
                        da[nt][2 * r + e] = in ? da[nt][2 * r + e] * inv[r] - delta[r] : 0.f;
                    }
                }
            uint32_t df[2][4];
            acc_to_a<4>(da, df);
            mma_tile<2, NT, true>(dph, df, sPK, LD, 0, 0);
        }
        // NP-Map backward: dl = phi (dphi - a phi / ||q||), a = dphi . phi / ||q||, with the
        // fp32 phi this thread wrote
        float ph[NT][4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float *src = P.phq32 + (qrow0 + (tr[r] < N ? tr[r] : 0)) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float2 x = tr[r] < N ? *reinterpret_cast<const float2 *>(src + nt * 8 + 2 * tig) : make_float2(0.f, 0.f);
                ph[nt][2 * r] = x.x;
                ph[nt][2 * r + 1] = x.y;
            }
        }
        float an[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float a = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) a = fmaf(dph[nt][2 * r], ph[nt][2 * r], fmaf(dph[nt][2 * r + 1], ph[nt][2 * r + 1], a));
            const float iq = nq[r] > 0.f ? 1.f / nq[r] : 0.f;
            a = quad_sum(a) * iq;
            an[r] = a * iq;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    dph[nt][2 * r + e] = ph[nt][2 * r + e] * (dph[nt][2 * r + e] - an[r] * ph[nt][2 * r + e]);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (tr[r] < N) {
                float *dst = P.dlq + (qrow0 + tr[r]) * D;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * tig) = make_float2(dph[nt][2 * r], dph[nt][2 * r + 1]);
            }
        // dq += a x / ||x|| + dl Wf^T
#pragma unroll
        for (int kc = 0; kc < KC; ++kc)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                dq[2 * kc][2 * r] += an[r] * lo_f(qa[kc][r]);
                dq[2 * kc][2 * r + 1] += an[r] * hi_f(qa[kc][r]);
                dq[2 * kc + 1][2 * r] += an[r] * lo_f(qa[kc][r + 2]);
                dq[2 * kc + 1][2 * r + 1] += an[r] * hi_f(qa[kc][r + 2]);
            }
        uint32_t lf[KC][4];
        acc_to_a<NT>(dph, lf);
        mma_tile<KC, NT, false>(dq, lf, sWF, LD, 0, 0);
    }

    // ---- outputs
#pragma unroll
    for (int r = 0; r < 2; ++r)
        if (tr[r] < N) {
            float *dst = P.dq + (qrow0 + tr[r]) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * tig) = make_float2(dq[nt][2 * r], dq[nt][2 * r + 1]);
            if (tig == 0) {
                const size_t ri = qrow0 + tr[r];
                P.rc[ri] = cm[r];
                P.rdelta[ri] = delta[r];
                P.rds[ri] = dss[r];
                P.rinv[ri] = inv[r];
                P.rjs[ri] = cj[r];
                if (P.cidx) P.cidx[ri] = cj[r];
            }
        }
}

// ---------------------------------------------------------------------------
// key passes: a warp owns 16 keys (rows of the transposed products)
// ---------------------------------------------------------------------------
constexpr int BK_KEYS = 128;   // keys (or kept-table entries) per CTA: eight warps of 16

template <int D>
struct KLayout {
    static constexpr int LD = D + 8, T32 = BT * LD * 2;
    static constexpr int NR = 6;                            // per query row: token, c, delta, ds sum, 1/den, c position
    static constexpr int K = 0, V = K + 4 * T32, PK = V + 4 * T32;   // the CTA's 128 keys
    static constexpr int QB = PK + 4 * T32;                 // two buffers of one query block: q, dy, phi(q)
    static constexpr int R = QB + 6 * T32;                  // R [df][d] bf16 of the linear pass, then Wf [d][df]
    static constexpr int RV = R + D * LD * 2;               // r, fp32 [df]
    static constexpr int ROW = RV + D * 4;                  // two buffers of the rows' scalars
    static constexpr int KPOS = ROW + 2 * NR * BT * 4;      // positions of the keys
    static constexpr int TOTAL = KPOS + BK_KEYS * 4;
};

// The query rows of one block (32 tokens of one head) and their scalars in
// shared memory.
struct QRows {
    int *tok;
    float *c, *delta, *dss, *inv;
    int *js;
};

__device__ __forceinline__ QRows qrows_at(int *base)
{
    return QRows{base, (float *)(base + BT), (float *)(base + 2 * BT), (float *)(base + 3 * BT),
                 (float *)(base + 4 * BT), base + 5 * BT};
}

// Query blocks (head, tokens [tq0, tq1)) streamed through two shared buffers by
// cp.async: q and dy rows (and phi(q) rows), the rows' scalars; tokens past
// tq1 are zero rows with token -1.  body(i, sQ, sG, sPQ, R) runs on block i once
// its copies have landed, while block i + 1 is being copied.
template <int D, typename BlockOf, typename Body>
__device__ __forceinline__ void query_blocks(const BwdArgs &P, int b, int nqb, bool with_phq, uint8_t *smem,
                                             BlockOf block_of, Body body)
{
    using L = KLayout<D>;
    constexpr int LD = D + 8, T32E = BT * LD, V8 = D / 8, NE = BT * V8;
    const Dims &dm = P.dm;
    const int tid = threadIdx.x, nth = blockDim.x;
    uint16_t *qb = (uint16_t *)(smem + L::QB);
    int *rows = (int *)(smem + L::ROW);
    auto issue = [&](int i, int buf) {
        int h, tq0, tq1;
        block_of(i, h, tq0, tq1);
        const size_t row0 = (size_t)(b * dm.Hq + h) * dm.N;
        uint16_t *dst = qb + buf * 3 * T32E;
        QRows R = qrows_at(rows + buf * L::NR * BT);
        for (int r = tid; r < BT; r += nth) R.tok[r] = tq0 + r < tq1 ? tq0 + r : -1;
        const int nm = with_phq ? 3 : 2;
        for (int e = tid; e < NE * nm; e += nth) {
            const int which = e / NE, j = e % NE, r = j / V8, c = j % V8;
            const bool ok = tq0 + r < tq1;
            const uint16_t *src = (which == 0 ? P.q : which == 1 ? P.dy : P.phq) + (row0 + (ok ? tq0 + r : 0)) * D + c * 8;
            cp_async16(dst + which * T32E + r * LD + c * 8, src, ok ? 16 : 0);
        }
        // scalars: 5 arrays of 32 values, one 4-byte copy each (a token's row need not
        // start on a 16-byte boundary), the rows past tq1 zero-filled
        for (int e = tid; e < 5 * BT; e += nth) {
            const int a = e / BT, r = e % BT;
            const bool ok = tq0 + r < tq1;
            const float *arr = a == 0 ? P.rc : a == 1 ? P.rdelta : a == 2 ? P.rds : a == 3 ? P.rinv : (const float *)P.rjs;
            float *d = a == 0 ? R.c : a == 1 ? R.delta : a == 2 ? R.dss : a == 3 ? R.inv : (float *)R.js;
            cp_async4(d + r, arr + (ok ? row0 + tq0 + r : 0), ok ? 4 : 0);
        }
        cp_commit();
    };
    if (nqb <= 0) return;
    issue(0, 0);
    for (int i = 0; i < nqb; ++i) {
        const int buf = i & 1;
        if (i + 1 < nqb) {
            issue(i + 1, buf ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        uint16_t *q = qb + buf * 3 * T32E;
        body(i, q, q + T32E, q + 2 * T32E, qrows_at(rows + buf * L::NR * BT));
        __syncthreads();
    }
}

// dK += dS^T Q, dV += P^T G over one staged query block for the warp's 16 keys
// (rows key0 .. key0+15 of sK / sV at positions kpos[]); sG holds dy, and
// G = dy / den takes the row's 1/den after the products.  `pair(t, p)` says
// whether key p is a softmax key of query t in this pass.
template <int D, typename Pair>
__device__ __forceinline__ void kv_block(const uint16_t *sK, const uint16_t *sV, int key0, const int *kpos,
                                         const uint16_t *sQ, const uint16_t *sG, QRows R, float scale,
                                         float (&dK)[D / 8][4], float (&dV)[D / 8][4], Pair pair)
{
    constexpr int LD = D + 8, KC = D / 16, NT = D / 8;
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    float s[4][4], dp[4][4];
    zero(s);
    zero(dp);
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
        uint32_t ka[4], va[4];
        load_a(sK, LD, key0, kc * 16, ka);
        load_a(sV, LD, key0, kc * 16, va);
#pragma unroll
        for (int nt = 0; nt < 4; nt += 2) {
            uint32_t f[4];
            load_b(sQ, LD, nt * 8, kc * 16, f);
            mma(s[nt], ka, f[0], f[1]);
            mma(s[nt + 1], ka, f[2], f[3]);
            load_b(sG, LD, nt * 8, kc * 16, f);
            mma(dp[nt], va, f[0], f[1]);
            mma(dp[nt + 1], va, f[2], f[3]);
        }
    }
    const int kp[2] = {kpos[key0 + gid], kpos[key0 + gid + 8]};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int qi = nt * 8 + 2 * tig + e;
            const int t = R.tok[qi];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const bool in = t >= 0 && kp[r] >= 0 && pair(t, kp[r]);
                const float pe = in ? exp2_mufu((s[nt][2 * r + e] * scale - R.c[qi]) * 1.4426950408889634f) : 0.f;
                float ds = pe * (dp[nt][2 * r + e] * R.inv[qi] - R.delta[qi]);
                if (in && R.js[qi] == kp[r]) ds -= R.dss[qi];
                s[nt][2 * r + e] = pe * R.inv[qi];
                dp[nt][2 * r + e] = ds;
            }
        }
    uint32_t pf[2][4], sf[2][4];
    acc_to_a<4>(s, pf);
    acc_to_a<4>(dp, sf);
    mma_tile<2, NT, true>(dK, sf, sQ, LD, 0, 0);
    mma_tile<2, NT, true>(dV, pf, sG, LD, 0, 0);
}

template <int D, int G>
__global__ void __launch_bounds__(BQ8_THREADS, 1) key_kernel(BwdArgs P)
{
    grid_dep_sync();
    constexpr int LD = D + 8, KC = D / 16, NT = D / 8;
    using L = KLayout<D>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *sK = (uint16_t *)(smem + L::K), *sV = (uint16_t *)(smem + L::V), *sPK = (uint16_t *)(smem + L::PK);
    uint16_t *sR = (uint16_t *)(smem + L::R);
    float *sRV = (float *)(smem + L::RV);
    int *kpos = (int *)(smem + L::KPOS);

    const Dims &dm = P.dm;
    const int N = dm.N, W = dm.W;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const int unit = blockIdx.y, b = unit / dm.Hkv, gq = unit % dm.Hkv;
    const int j0 = blockIdx.x * BK_KEYS;
    const size_t krow0 = (size_t)unit * N;
    const int key0 = warp * 16;
    const int kr[2] = {j0 + key0 + gid, j0 + key0 + gid + 8};

    for (int i = threadIdx.x; i < BK_KEYS; i += blockDim.x) kpos[i] = j0 + i < N ? j0 + i : -1;
    __syncthreads();
    stage_rows<D>(sK, LD, BK_KEYS, [&](int r) -> const uint16_t * { return kpos[r] >= 0 ? P.k + (krow0 + kpos[r]) * D : nullptr; });
    stage_rows<D>(sV, LD, BK_KEYS, [&](int r) -> const uint16_t * { return kpos[r] >= 0 ? P.v + (krow0 + kpos[r]) * D : nullptr; });
    stage_rows<D>(sPK, LD, BK_KEYS, [&](int r) -> const uint16_t * { return kpos[r] >= 0 ? P.phk + (krow0 + kpos[r]) * D : nullptr; });
    __syncthreads();

    // ---- window queries: t in [j, j + W - 1]
    float dK[NT][4], dV[NT][4];
    zero(dK);
    zero(dV);
    {
        const int tq_end = min(j0 + BK_KEYS + W - 1, N);
        const int per = (tq_end - j0 + BT - 1) / BT;
        // a warp's keys [jw, jw + 16) see the queries [jw, jw + 15 + W): it skips the other blocks
        const int jw = j0 + key0;
        query_blocks<D>(P, b, G * per, false, smem,
                        [&](int i, int &h, int &tq0, int &tq1) {
                            h = gq * G + i / per;
                            tq0 = j0 + (i % per) * BT;
                            tq1 = tq_end;
                        },
                        [&](int i, const uint16_t *sQ, const uint16_t *sG, const uint16_t *, QRows R) {
                            const int tq0 = j0 + (i % per) * BT;
                            if (tq0 + BT - 1 < jw || tq0 > jw + 15 + W - 1) return;
                            kv_block<D>(sK, sV, key0, kpos, sQ, sG, R, P.scale, dK, dV,
                                        [&](int t, int p) { return p <= t && p > t - W; });
                        });
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
        if (kr[r] < N) {
            float *dst = P.dk + (krow0 + kr[r]) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * tig) = make_float2(dK[nt][0 + 2 * r] * P.scale, dK[nt][1 + 2 * r] * P.scale);
        }

    // ---- linear branch: R, r over the queries t >= U1, then the lag queries [j + W, U1)
    const int U1 = ((j0 + BK_KEYS - 1 + W + BT - 1) / BT) * BT;
    const int ub = min(U1 / BT, P.nblk);
    const size_t rslot = (size_t)unit * (P.nblk + 1) + (P.nblk - ub);
    stage_f32(sR, LD, P.Rs + rslot * D * D, D, D);
    for (int f = threadIdx.x; f < D; f += blockDim.x) sRV[f] = P.rs[rslot * D + f];
    __syncthreads();
    const bool kk[2] = {kr[0] < N && P.kslot[krow0 + kr[0]] >= 0, kr[1] < N && P.kslot[krow0 + kr[1]] >= 0};
    float dph[NT][4];
    zero(dph);
    {
        uint32_t va[KC][4], pk[KC][4];
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
            load_a(sV, LD, key0, kc * 16, va[kc]);
            load_a(sPK, LD, key0, kc * 16, pk[kc]);
        }
        mma_tile<KC, NT, false>(dph, va, sR, LD, 0, 0);   // V R^T: B(k = d, n = f) = R[f][d]
        mma_tile<KC, NT, true>(dV, pk, sR, LD, 0, 0);     // phi(K) R: B(k = f, n = d) = R[f][d]
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float rv = sRV[nt * 8 + 2 * tig + e];
            dph[nt][e] -= rv;
            dph[nt][2 + e] -= rv;
        }
    {
        const int lq0 = j0 + W, lq1 = min(U1, N);
        const int per = lq1 > lq0 ? (lq1 - lq0 + BT - 1) / BT : 0;
        query_blocks<D>(P, b, G * per, true, smem,
                        [&](int i, int &h, int &tq0, int &tq1) {
                            h = gq * G + i / per;
                            tq0 = lq0 + (i % per) * BT;
                            tq1 = lq1;
                        },
                        [&](int, const uint16_t *, const uint16_t *sG, const uint16_t *sPQ, QRows R) {
                            float dat[4][4], at[4][4];
                            zero(dat);
                            zero(at);
#pragma unroll
                            for (int kc = 0; kc < KC; ++kc) {
                                uint32_t va[4], pk[4];
                                load_a(sV, LD, key0, kc * 16, va);
                                load_a(sPK, LD, key0, kc * 16, pk);
#pragma unroll
                                for (int nt = 0; nt < 4; nt += 2) {
                                    uint32_t f[4];
                                    load_b(sG, LD, nt * 8, kc * 16, f);
                                    mma(dat[nt], va, f[0], f[1]);
                                    mma(dat[nt + 1], va, f[2], f[3]);
                                    load_b(sPQ, LD, nt * 8, kc * 16, f);
                                    mma(at[nt], pk, f[0], f[1]);
                                    mma(at[nt + 1], pk, f[2], f[3]);
                                }
                            }
#pragma unroll
                            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int qi = nt * 8 + 2 * tig + e;
                                    const int t = R.tok[qi];
#pragma unroll
                                    for (int r = 0; r < 2; ++r) {
                                        const bool in = t >= 0 && kr[r] < N && t >= kr[r] + W;
                                        dat[nt][2 * r + e] = in ? dat[nt][2 * r + e] * R.inv[qi] - R.delta[qi] : 0.f;
                                        at[nt][2 * r + e] = in ? at[nt][2 * r + e] * R.inv[qi] : 0.f;
                                    }
                                }
                            uint32_t df[2][4], af[2][4];
                            acc_to_a<4>(dat, df);
                            acc_to_a<4>(at, af);
                            mma_tile<2, NT, true>(dph, df, sPQ, LD, 0, 0);
                            mma_tile<2, NT, true>(dV, af, sG, LD, 0, 0);
                        });
    }
    // kept keys have no linear role
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (kk[r] || kr[r] >= N) dph[nt][2 * r] = dph[nt][2 * r + 1] = 0.f;

    // ---- NP-Map backward of the key rows (Wf replaces R in shared memory)
    __syncthreads();
    for (int i = threadIdx.x; i < D * D / 4; i += blockDim.x) {
        const int r = i / (D / 4), c = (i % (D / 4)) * 4;
        const float4 x = __ldg(reinterpret_cast<const float4 *>(P.Wf) + i);
        *reinterpret_cast<uint2 *>(sR + r * LD + c) = make_uint2(pack(x.x, x.y), pack(x.z, x.w));
    }
    __syncthreads();
    float ph[NT][4], xk[NT][4];
    float an[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = key0 + gid + 8 * r;
        float a = 0.f, x2 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int col = nt * 8 + 2 * tig + e;
                ph[nt][2 * r + e] = kr[r] < N ? P.phk32[(krow0 + kr[r]) * D + col] : 0.f;
                xk[nt][2 * r + e] = bf2f(sK[row * LD + col]);
                a = fmaf(dph[nt][2 * r + e], ph[nt][2 * r + e], a);
                x2 = fmaf(xk[nt][2 * r + e], xk[nt][2 * r + e], x2);
            }
        const float nk = sqrtf(quad_sum(x2));
        const float ik = nk > 0.f ? 1.f / nk : 0.f;
        an[r] = quad_sum(a) * ik * ik;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                dph[nt][2 * r + e] = ph[nt][2 * r + e] * (dph[nt][2 * r + e] - an[r] * ph[nt][2 * r + e]);
    }
    float dkn[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) dkn[nt][i] = an[i >> 1] * xk[nt][i];
    uint32_t lf[KC][4];
    acc_to_a<NT>(dph, lf);
    mma_tile<KC, NT, false>(dkn, lf, sR, LD, 0, 0);   // dl Wf^T: B(k = f, n = i) = Wf[i][f]
#pragma unroll
    for (int r = 0; r < 2; ++r)
        if (kr[r] < N) {
            float *dst = P.dk + (krow0 + kr[r]) * D;
            float *dvd = P.dv + (krow0 + kr[r]) * D;
            float *dl = P.dlk + (krow0 + kr[r]) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float2 *p2 = reinterpret_cast<float2 *>(dst + nt * 8 + 2 * tig);
                const float2 old = *p2;
                *p2 = make_float2(old.x + dkn[nt][2 * r], old.y + dkn[nt][2 * r + 1]);
                *reinterpret_cast<float2 *>(dvd + nt * 8 + 2 * tig) = make_float2(dV[nt][2 * r], dV[nt][2 * r + 1]);
                *reinterpret_cast<float2 *>(dl + nt * 8 + 2 * tig) = make_float2(dph[nt][2 * r], dph[nt][2 * r + 1]);
            }
        }
}

// dk, dv of the kept keys from the queries of later chunks outside the window:
// CTA = 128 entries of the kept table x one range of query tokens.
constexpr int KEPT_TOKENS = 256;

template <int D, int G>
__global__ void __launch_bounds__(BQ8_THREADS, 1) kept_kernel(BwdArgs P)
{
    grid_dep_sync();
    constexpr int LD = D + 8, NT = D / 8;
    using L = KLayout<D>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *sK = (uint16_t *)(smem + L::K), *sV = (uint16_t *)(smem + L::V);
    int *kpos = (int *)(smem + L::KPOS);

    const Dims &dm = P.dm;
    const int N = dm.N, W = dm.W, C = dm.C;
    const int KP = dm.T_max * dm.lam;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const int unit = blockIdx.y, b = unit / dm.Hkv, gq = unit % dm.Hkv;
    const int e0 = blockIdx.x * BK_KEYS;
    const size_t krow0 = (size_t)unit * N;
    const int key0 = warp * 16;
    auto entry = [&](int e) -> int {
        const int p = e < KP ? P.sel[(size_t)unit * KP + e] : -1;
        return p < N ? p : -1;
    };
    // queries of this CTA: tokens [tq_lo, tq_hi), from the end of the first entry's chunk on
    int first = -1;
    for (int i = 0; i < BK_KEYS && first < 0; ++i) first = entry(e0 + i);
    if (first < 0) return;
    const int start = (first / C + 1) * C;
    const int tq_lo = start + blockIdx.z * KEPT_TOKENS, tq_hi = min(tq_lo + KEPT_TOKENS, N);
    if (tq_lo >= tq_hi) return;

    for (int i = threadIdx.x; i < BK_KEYS; i += blockDim.x) kpos[i] = entry(e0 + i);
    __syncthreads();
    stage_rows<D>(sK, LD, BK_KEYS, [&](int r) -> const uint16_t * { return kpos[r] >= 0 ? P.k + (krow0 + kpos[r]) * D : nullptr; });
    stage_rows<D>(sV, LD, BK_KEYS, [&](int r) -> const uint16_t * { return kpos[r] >= 0 ? P.v + (krow0 + kpos[r]) * D : nullptr; });
    __syncthreads();

    float dK[NT][4], dV[NT][4];
    zero(dK);
    zero(dV);
    // the warp's first live query: the smallest p + W over its entries (entries ascend,
    // so the first valid one), or none
    int wfirst = INT_MAX;
    for (int i = 0; i < 16; ++i)
        if (kpos[key0 + i] >= 0) {
            wfirst = kpos[key0 + i] + W;
            break;
        }
    const int per = (tq_hi - tq_lo + BT - 1) / BT;
    query_blocks<D>(P, b, G * per, false, smem,
                    [&](int i, int &h, int &tq0, int &tq1) {
                        h = gq * G + i / per;
                        tq0 = tq_lo + (i % per) * BT;
                        tq1 = tq_hi;
                    },
                    [&](int i, const uint16_t *sQ, const uint16_t *sG, const uint16_t *, QRows R) {
                        if (tq_lo + (i % per) * BT + BT - 1 < wfirst) return;
                        kv_block<D>(sK, sV, key0, kpos, sQ, sG, R, P.scale, dK, dV,
                                    [&](int t, int p) { return p <= t - W && (W >= C || p / C < t / C); });
                    });
    const int kp[2] = {kpos[key0 + gid], kpos[key0 + gid + 8]};
#pragma unroll
    for (int r = 0; r < 2; ++r)
        if (kp[r] >= 0) {
            float *dk = P.dk + (krow0 + kp[r]) * D, *dv = P.dv + (krow0 + kp[r]) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = nt * 8 + 2 * tig;
                atomicAdd(dk + col, dK[nt][2 * r] * P.scale);
                atomicAdd(dk + col + 1, dK[nt][2 * r + 1] * P.scale);
                atomicAdd(dv + col, dV[nt][2 * r]);
                atomicAdd(dv + col + 1, dV[nt][2 * r + 1]);
            }
        }
}

// When W < C a kept key is a linear key of the later queries of its own chunk
// (t >= j + W, t in chunk(j)) until the chunk completes.  CTA = one chunk c of one
// (sequence, kv head): its kept entries (warp w: entries [16w, 16w + 16)) against
// the queries [cC + W, (c + 1)C): dphi(k) = sum phi(q) (g.v - delta) and
// dv += sum (phi(q).phi(k)) g, then the NP-Map backward of those keys; dk, dv
// by atomic additions, dl of their rows written for the dWf pass.
template <int D, int G>
__global__ void __launch_bounds__(BQ8_THREADS, 1) kept_lin_kernel(BwdArgs P)
{
    grid_dep_sync();
    constexpr int LD = D + 8, KC = D / 16, NT = D / 8;
    using L = KLayout<D>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *sK = (uint16_t *)(smem + L::K), *sV = (uint16_t *)(smem + L::V), *sPK = (uint16_t *)(smem + L::PK);
    uint16_t *sR = (uint16_t *)(smem + L::R);
    int *kpos = (int *)(smem + L::KPOS);

    const Dims &dm = P.dm;
    const int N = dm.N, W = dm.W, C = dm.C, lam = dm.lam;
    const int KP = dm.T_max * lam;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const int c = blockIdx.x, unit = blockIdx.y, b = unit / dm.Hkv, gq = unit % dm.Hkv;
    const size_t krow0 = (size_t)unit * N;
    const int key0 = warp * 16;
    const int e0 = c * lam;
    const int tq_lo = c * C + W, tq_hi = min((c + 1) * C, N);
    if (tq_lo >= tq_hi) return;
    for (int i = threadIdx.x; i < BK_KEYS; i += blockDim.x) {
        int p = i < lam ? P.sel[(size_t)unit * KP + e0 + i] : -1;
        kpos[i] = p >= 0 && p < N ? p : -1;
    }
    __syncthreads();
    stage_rows<D>(sK, LD, BK_KEYS, [&](int r) -> const uint16_t * { return kpos[r] >= 0 ? P.k + (krow0 + kpos[r]) * D : nullptr; });
    stage_rows<D>(sV, LD, BK_KEYS, [&](int r) -> const uint16_t * { return kpos[r] >= 0 ? P.v + (krow0 + kpos[r]) * D : nullptr; });
    stage_rows<D>(sPK, LD, BK_KEYS, [&](int r) -> const uint16_t * {
        return kpos[r] >= 0 ? P.phkk + ((size_t)unit * KP + e0 + r) * D : nullptr;
    });
    __syncthreads();
    const bool active = key0 < lam;
    const int kr[2] = {kpos[key0 + gid], kpos[key0 + gid + 8]};

    float dph[NT][4], dV[NT][4];
    zero(dph);
    zero(dV);
    const int per = (tq_hi - tq_lo + BT - 1) / BT;
    query_blocks<D>(P, b, G * per, true, smem,
                    [&](int i, int &h, int &tq0, int &tq1) {
                        h = gq * G + i / per;
                        tq0 = tq_lo + (i % per) * BT;
                        tq1 = tq_hi;
                    },
                    [&](int, const uint16_t *, const uint16_t *sG, const uint16_t *sPQ, QRows R) {
                        if (!active) return;
                        float dat[4][4], at[4][4];
                        zero(dat);
                        zero(at);
#pragma unroll
                        for (int kc = 0; kc < KC; ++kc) {
                            uint32_t va[4], pk[4];
                            load_a(sV, LD, key0, kc * 16, va);
                            load_a(sPK, LD, key0, kc * 16, pk);
#pragma unroll
                            for (int nt = 0; nt < 4; nt += 2) {
                                uint32_t f[4];
                                load_b(sG, LD, nt * 8, kc * 16, f);
                                mma(dat[nt], va, f[0], f[1]);
                                mma(dat[nt + 1], va, f[2], f[3]);
                                load_b(sPQ, LD, nt * 8, kc * 16, f);
                                mma(at[nt], pk, f[0], f[1]);
                                mma(at[nt + 1], pk, f[2], f[3]);
                            }
                        }
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int qi = nt * 8 + 2 * tig + e;
                                const int t = R.tok[qi];
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    const bool in = t >= 0 && kr[r] >= 0 && t >= kr[r] + W;
                                    dat[nt][2 * r + e] = in ? dat[nt][2 * r + e] * R.inv[qi] - R.delta[qi] : 0.f;
                                    at[nt][2 * r + e] = in ? at[nt][2 * r + e] * R.inv[qi] : 0.f;
                                }
                            }
                        uint32_t df[2][4], af[2][4];
                        acc_to_a<4>(dat, df);
                        acc_to_a<4>(at, af);
                        mma_tile<2, NT, true>(dph, df, sPQ, LD, 0, 0);
                        mma_tile<2, NT, true>(dV, af, sG, LD, 0, 0);
                    });

    // ---- NP-Map backward of these keys' rows (Wf in shared memory)
    __syncthreads();
    for (int i = threadIdx.x; i < D * D / 4; i += blockDim.x) {
        const int r = i / (D / 4), cc = (i % (D / 4)) * 4;
        const float4 x = __ldg(reinterpret_cast<const float4 *>(P.Wf) + i);
        *reinterpret_cast<uint2 *>(sR + r * LD + cc) = make_uint2(pack(x.x, x.y), pack(x.z, x.w));
    }
    __syncthreads();
    if (!active) return;
    float ph[NT][4], xk[NT][4];
    float an[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = key0 + gid + 8 * r;
        float a = 0.f, x2 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int col = nt * 8 + 2 * tig + e;
                ph[nt][2 * r + e] = kr[r] >= 0 ? P.phkk32[((size_t)unit * KP + e0 + row) * D + col] : 0.f;
                xk[nt][2 * r + e] = bf2f(sK[row * LD + col]);
                a = fmaf(dph[nt][2 * r + e], ph[nt][2 * r + e], a);
                x2 = fmaf(xk[nt][2 * r + e], xk[nt][2 * r + e], x2);
            }
        const float nk = sqrtf(quad_sum(x2));
        const float ik = nk > 0.f ? 1.f / nk : 0.f;
        an[r] = quad_sum(a) * ik * ik;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                dph[nt][2 * r + e] = ph[nt][2 * r + e] * (dph[nt][2 * r + e] - an[r] * ph[nt][2 * r + e]);
    }
    float dkn[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) dkn[nt][i] = an[i >> 1] * xk[nt][i];
    uint32_t lf[KC][4];
    acc_to_a<NT>(dph, lf);
    mma_tile<KC, NT, false>(dkn, lf, sR, LD, 0, 0);   // dl Wf^T: B(k = f, n = i) = Wf[i][f]
#pragma unroll
    for (int r = 0; r < 2; ++r)
        if (kr[r] >= 0) {
            float *dk = P.dk + (krow0 + kr[r]) * D, *dv = P.dv + (krow0 + kr[r]) * D;
            float *dl = P.dlk + (krow0 + kr[r]) * D;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = nt * 8 + 2 * tig;
                atomicAdd(dk + col, dkn[nt][2 * r]);
                atomicAdd(dk + col + 1, dkn[nt][2 * r + 1]);
                atomicAdd(dv + col, dV[nt][2 * r]);
                atomicAdd(dv + col + 1, dV[nt][2 * r + 1]);
                *reinterpret_cast<float2 *>(dl + col) = make_float2(dph[nt][2 * r], dph[nt][2 * r + 1]);
            }
        }
}

// ---------------------------------------------------------------------------
// dWf = sum_rows x^T dl over the q rows and the k rows: CTA = a range of rows,
// warp w the Wf rows [16w, 16w + 16); partial sums added atomically.  dl is
// fp32; it enters the MMAs as a bf16 pair hi + lo (hi = bf16(dl), lo =
// bf16(dl - hi)), about 16 significant bits.
constexpr int DWF_ROWS_Q = 1024, DWF_ROWS_K = 256;   // rows per CTA of the q rows and of the k rows

template <int D, int DF>
__global__ void __launch_bounds__(256) dwf_kernel(const uint16_t *__restrict__ xq, const float *__restrict__ dlq,
                                                  long long rows_q, const uint16_t *__restrict__ xk,
                                                  const float *__restrict__ dlk, long long rows_k, int ctas_q,
                                                  float *__restrict__ dWf)
{
    grid_dep_sync();
    // CTAs [0, ctas_q) take the q rows, the others the k rows
    const bool kq = (int)blockIdx.x < ctas_q;
    const uint16_t *x = kq ? xq : xk;
    const float *dl = kq ? dlq : dlk;
    const long long rows = kq ? rows_q : rows_k;
    const long long per = kq ? DWF_ROWS_Q : DWF_ROWS_K;
    const long long cta = kq ? blockIdx.x : blockIdx.x - ctas_q;
    constexpr int LDX = D + 8, LDL = DF + 8, NT = DF / 8;
    __shared__ __align__(16) uint16_t sx[BT * LDX];
    __shared__ __align__(16) uint16_t sl[BT * LDL];
    __shared__ __align__(16) uint16_t sl2[BT * LDL];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const long long r0 = cta * per;
    const long long r1 = min(r0 + per, rows);
    float acc[NT][4];
    zero(acc);
    for (long long rb = r0; rb < r1; rb += BT) {
        __syncthreads();
        stage_rows<D>(sx, LDX, BT, [&](int r) -> const uint16_t * { return rb + r < r1 ? x + (rb + r) * D : nullptr; });
        for (int i = threadIdx.x; i < BT * DF / 4; i += blockDim.x) {
            const int r = i / (DF / 4), c = (i % (DF / 4)) * 4;
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
            if (rb + r < r1) f = __ldg(reinterpret_cast<const float4 *>(dl + (rb + r) * DF + c));
            const uint32_t h0 = pack(f.x, f.y), h1 = pack(f.z, f.w);
            *reinterpret_cast<uint2 *>(sl + r * LDL + c) = make_uint2(h0, h1);
            *reinterpret_cast<uint2 *>(sl2 + r * LDL + c) =
                make_uint2(pack(f.x - lo_f(h0), f.y - hi_f(h0)), pack(f.z - lo_f(h1), f.w - hi_f(h1)));
        }
        __syncthreads();
        if (warp < D / 16) {
#pragma unroll
            for (int k0 = 0; k0 < BT; k0 += 16) {
                uint32_t a[1][4];
                load_a_t(sx, LDX, warp * 16, k0, a[0]);
                mma_tile<1, NT, true>(acc, a, sl, LDL, 0, k0);
                mma_tile<1, NT, true>(acc, a, sl2, LDL, 0, k0);
            }
        }
    }
    if (warp < D / 16) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = nt * 8 + 2 * tig;
            float *o0 = dWf + (size_t)(warp * 16 + gid) * DF + col, *o1 = o0 + 8 * DF;
            atomicAdd(o0, acc[nt][0]);
            atomicAdd(o0 + 1, acc[nt][1]);
            atomicAdd(o1, acc[nt][2]);
            atomicAdd(o1 + 1, acc[nt][3]);
        }
    }
}

struct BwdBuffers {
    int32_t *kslot;
    uint16_t *phkk;
    float *phkk32;
    uint16_t *phk;
    float *phk32;
    float *Sp, *zp, *Rs, *rs;
};

template <typename K>
cudaError_t set_smem(K kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int D, int G>
cudaError_t run(const BwdArgs &A, const BwdBuffers &bb, cudaStream_t s)
{
    const Dims &dm = A.dm;
    const int units = dm.B * dm.Hkv;
    const int KP = dm.T_max * dm.lam;
    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess && x != cudaSuccess) e = x;
        if (e == cudaSuccess) e = cudaGetLastError();
    };
    {
        KTimer tm("bwd_prep", s);
        chk(cudaMemsetAsync(bb.kslot, 0xff, (size_t)units * dm.N * 4, s));
        if (KP > 0) chk(launch_kernel(mark_kept_kernel, dim3((KP + 255) / 256, units), dim3(256), 0, s, A.sel, KP, dm.N, bb.kslot));
        const long long rows = (long long)units * dm.N;
        const size_t sm = 2 * (size_t)D * (D + 8) * 2;
        chk(set_smem(phik_mma_kernel<D>, sm));
        chk(launch_kernel(phik_mma_kernel<D>, dim3((unsigned)((rows + 127) / 128)), dim3(256), sm, s, A, bb.phk, bb.phk32,
                          bb.phkk, bb.phkk32));
    }
    const size_t bs_smem = BSLayout<D, D>::TOTAL;
    const int nel_s = D * D, nel_z = D;
    {
        KTimer tm("bwd_state", s);
        chk(set_smem(blocksum_kernel<D, D, false>, bs_smem));
        chk(launch_kernel(blocksum_kernel<D, D, false>, dim3(A.nblk, units), dim3(256), bs_smem, s, A, bb.Sp, bb.zp));
        chk(launch_kernel(scan_kernel, dim3((nel_s + nel_z + 255) / 256, units), dim3(256), 0, s, bb.Sp, bb.zp, A.nblk,
                          nel_s, nel_z));
    }
    {
        KTimer tm("bwd_query", s);
        constexpr int TOK = 16 * (8 / G);
        chk(set_smem(query_kernel<D, G>, QLayout<D>::TOTAL));
        chk(launch_kernel(query_kernel<D, G>, dim3((dm.N + TOK - 1) / TOK, units), dim3(BQ8_THREADS), QLayout<D>::TOTAL, s, A));
    }
    {
        KTimer tm("bwd_rstate", s);
        chk(set_smem(blocksum_kernel<D, D, true>, bs_smem));
        chk(launch_kernel(blocksum_kernel<D, D, true>, dim3(A.nblk, units), dim3(256), bs_smem, s, A, bb.Rs, bb.rs));
        chk(launch_kernel(scan_kernel, dim3((nel_s + nel_z + 255) / 256, units), dim3(256), 0, s, bb.Rs, bb.rs, A.nblk,
                          nel_s, nel_z));
    }
    {
        KTimer tm("bwd_key", s);
        chk(set_smem(key_kernel<D, G>, KLayout<D>::TOTAL));
        chk(launch_kernel(key_kernel<D, G>, dim3((dm.N + BK_KEYS - 1) / BK_KEYS, units), dim3(BQ8_THREADS), KLayout<D>::TOTAL,
                          s, A));
    }
    if (KP > 0) {
        KTimer tm("bwd_kept", s);
        chk(set_smem(kept_kernel<D, G>, KLayout<D>::TOTAL));
        const int nsplit = (dm.N + KEPT_TOKENS - 1) / KEPT_TOKENS;
        chk(launch_kernel(kept_kernel<D, G>, dim3((KP + BK_KEYS - 1) / BK_KEYS, units, nsplit), dim3(BQ8_THREADS),
                          KLayout<D>::TOTAL, s, A));
    }
    if (KP > 0 && dm.W < dm.C) {
        KTimer tm("bwd_kept_lin", s);
        chk(set_smem(kept_lin_kernel<D, G>, KLayout<D>::TOTAL));
        chk(launch_kernel(kept_lin_kernel<D, G>, dim3(dm.T_max, units), dim3(BQ8_THREADS), KLayout<D>::TOTAL, s, A));
    }
    {
        KTimer tm("bwd_dwf", s);
        chk(cudaMemsetAsync(A.dWf, 0, (size_t)D * D * 4, s));
        const long long rq = (long long)dm.B * dm.Hq * dm.N, rk = (long long)units * dm.N;
        const int cq = (int)((rq + DWF_ROWS_Q - 1) / DWF_ROWS_Q), ck = (int)((rk + DWF_ROWS_K - 1) / DWF_ROWS_K);
        chk(launch_kernel(dwf_kernel<D, D>, dim3((unsigned)(cq + ck)), dim3(256), 0, s, A.q, (const float *)A.dlq, rq,
                          A.k, (const float *)A.dlk, rk, cq, A.dWf));
    }
    return e;
}

}  // namespace

BwdLayout bwd_layout(const Dims &dm)
{
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    BwdLayout L;
    const size_t units = (size_t)dm.B * dm.Hkv, rows_q = (size_t)dm.B * dm.Hq * dm.N, rows_k = units * dm.N;
    const int nblk = (dm.N + BT - 1) / BT;
    size_t o = 0;
    const size_t KPs = (size_t)dm.T_max * dm.lam > 0 ? (size_t)dm.T_max * dm.lam : 1;
    L.kslot = o; o += al(rows_k * 4);
    L.phkk = o; o += al(units * KPs * dm.df * 2);
    L.phkk32 = o; o += al(units * KPs * dm.df * 4);
    L.phk = o; o += al(rows_k * dm.df * 2);
    L.Sp = o; o += al(units * (nblk + 1) * (size_t)dm.df * dm.d * 4);
    L.zp = o; o += al(units * (nblk + 1) * (size_t)dm.df * 4);
    L.Rs = o; o += al(units * (nblk + 1) * (size_t)dm.df * dm.d * 4);
    L.rs = o; o += al(units * (nblk + 1) * (size_t)dm.df * 4);
    L.g = o; o += al(rows_q * dm.d * 2);
    L.phq = o; o += al(rows_q * dm.df * 2);
    L.phq32 = o; o += al(rows_q * dm.df * 4);
    L.phk32 = o; o += al(rows_k * dm.df * 4);
    L.dlq = o; o += al(rows_q * dm.df * 4);
    L.dlk = o; o += al(rows_k * dm.df * 4);
    L.rc = o; o += al(rows_q * 4);
    L.rinv = o; o += al(rows_q * 4);
    L.rdelta = o; o += al(rows_q * 4);
    L.rds = o; o += al(rows_q * 4);
    L.rjs = o; o += al(rows_q * 4);
    L.total = o;
    return L;
}

bool backward_supported(const Dims &dm)
{
    // lambda <= 128: the kept entries of a chunk fit the eight warps of the own-chunk pass
    return dm.d == dm.df && (dm.d == 64 || dm.d == 128) && (dm.G == 1 || dm.G == 2 || dm.G == 4) &&
           (dm.W >= dm.C || dm.lam <= BK_KEYS);
}

cudaError_t launch_backward(const Dims &dm, const BwdInputs &in, void *ws)
{
    const BwdLayout L = bwd_layout(dm);
    char *base = (char *)ws;
    BwdArgs A{};
    A.dm = dm;
    A.nblk = (dm.N + BT - 1) / BT;
    A.scale = 1.f / sqrtf((float)dm.d);
    A.q = in.q; A.k = in.k; A.v = in.v; A.dy = in.dy; A.Wf = in.Wf; A.sel = in.sel;
    BwdBuffers bb;
    bb.kslot = (int32_t *)(base + L.kslot);
    bb.phkk = (uint16_t *)(base + L.phkk);
    bb.phkk32 = (float *)(base + L.phkk32);
    bb.Sp = (float *)(base + L.Sp); bb.zp = (float *)(base + L.zp);
    bb.Rs = (float *)(base + L.Rs); bb.rs = (float *)(base + L.rs);
    A.kslot = bb.kslot;
    A.phkk = bb.phkk;
    A.phkk32 = bb.phkk32;
    bb.phk = (uint16_t *)(base + L.phk);
    A.phk = bb.phk;
    A.Sp = bb.Sp; A.zp = bb.zp; A.Rs = bb.Rs; A.rs = bb.rs;
    A.g = (uint16_t *)(base + L.g);
    A.phq = (uint16_t *)(base + L.phq);
    A.phq32 = (float *)(base + L.phq32);
    bb.phk32 = (float *)(base + L.phk32);
    A.phk32 = bb.phk32;
    A.dlq = (float *)(base + L.dlq);
    A.dlk = (float *)(base + L.dlk);
    A.rinv = (float *)(base + L.rinv);
    A.rc = (float *)(base + L.rc);
    A.rdelta = (float *)(base + L.rdelta);
    A.rds = (float *)(base + L.rds);
    A.rjs = (int32_t *)(base + L.rjs);
    A.dq = in.dq; A.dk = in.dk; A.dv = in.dv; A.dWf = in.dWf; A.cidx = in.cidx;
    cudaStream_t s = in.stream;
    if (dm.d == 128) {
        if (dm.G == 4) return run<128, 4>(A, bb, s);
        if (dm.G == 2) return run<128, 2>(A, bb, s);
        return run<128, 1>(A, bb, s);
    }
    if (dm.G == 4) return run<64, 4>(A, bb, s);
    if (dm.G == 2) return run<64, 2>(A, bb, s);
    return run<64, 1>(A, bb, s);
}

}  // namespace still
