// Warp-level bf16 MMA (m16n8k16, fp32 accumulation) on row-padded shared
// tiles, for the passes whose tiles are too small or too irregular for the
// asynchronous tensor-core path (the backward pass).
//
// Fragment layouts are the PTX ISA's for mma.m16n8k16 with .row.col: with
// gid = lane / 4 and tig = lane % 4,
//   A (16 x 16):  a0 = (gid, 2tig..2tig+1), a1 = (gid+8, 2tig..), a2 = (gid, 8+2tig..), a3 = (gid+8, 8+2tig..)
//   B (16 x 8):   b0 = (k = 2tig..2tig+1, n = gid), b1 = (k = 8+2tig.., n = gid)
//   C (16 x 8):   c0, c1 = (gid, 2tig..2tig+1), c2, c3 = (gid+8, 2tig..)
// so the accumulators of two adjacent 8-column tiles are, packed to bf16
// pairs, the A fragment of the 16-wide K step over the same columns.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace still {
namespace wmma16 {

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float lo_f(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float hi_f(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Shared tiles are bf16, row-major, `ld` elements per row (a multiple of 8 whose
// byte stride is an odd multiple of 16, so that the 8 rows of an 8x8 matrix fall
// in distinct banks).

// A fragment of the 16 x 16 block at (row0, k0) of a tile stored [m][k].
__device__ __forceinline__ void load_a(const uint16_t *t, int ld, int row0, int k0, uint32_t (&a)[4])
{
    const int l = threadIdx.x & 31;
    ldsm4(smem_addr(t + (row0 + (l & 15)) * ld + k0 + (l >> 4) * 8), a);
}

// A fragment of the 16 x 16 block (m0.., k0..) of a tile stored [k][m].
__device__ __forceinline__ void load_a_t(const uint16_t *t, int ld, int m0, int k0, uint32_t (&a)[4])
{
    const int l = threadIdx.x & 31, i = l >> 3, r = l & 7;
    ldsm4t(smem_addr(t + (k0 + r + (i >> 1) * 8) * ld + m0 + (i & 1) * 8), a);
}

// B fragments of two adjacent 8-column tiles (n0.., n0+8..) over k0 .. k0+15, tile stored [n][k]:
// b[0], b[1] for the first tile, b[2], b[3] for the second.
__device__ __forceinline__ void load_b(const uint16_t *t, int ld, int n0, int k0, uint32_t (&b)[4])
{
    const int l = threadIdx.x & 31, i = l >> 3, r = l & 7;
    ldsm4(smem_addr(t + (n0 + r + (i >> 1) * 8) * ld + k0 + (i & 1) * 8), b);
}

// The same from a tile stored [k][n].
__device__ __forceinline__ void load_b_t(const uint16_t *t, int ld, int n0, int k0, uint32_t (&b)[4])
{
    const int l = threadIdx.x & 31, i = l >> 3, r = l & 7;
    ldsm4t(smem_addr(t + (k0 + r + (i & 1) * 8) * ld + n0 + (i >> 1) * 8), b);
}

// acc[NT][4] (NT tiles of 8 columns) += A (16 x 16K) * B, A given as KC fragments,
// B (K x 8NT) a shared tile stored [n][k] (kt = false) or [k][n] (kt = true), its
// column n0 and row k0 at (n_base, k_base).
template <int KC, int NT, bool KT>
__device__ __forceinline__ void mma_tile(float (&acc)[NT][4], const uint32_t (&a)[KC][4], const uint16_t *b, int ld,
                                         int n_base, int k_base)
{
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
            uint32_t f[4];
            if (KT)
                load_b_t(b, ld, n_base + nt * 8, k_base + kc * 16, f);
            else
                load_b(b, ld, n_base + nt * 8, k_base + kc * 16, f);
            mma(acc[nt], a[kc], f[0], f[1]);
            mma(acc[nt + 1], a[kc], f[2], f[3]);
        }
    }
}

// A fragments (KC = NT / 2 steps of 16) of the bf16-rounded accumulators.
template <int NT>
__device__ __forceinline__ void acc_to_a(const float (&c)[NT][4], uint32_t (&a)[NT / 2][4])
{
#pragma unroll
    for (int kc = 0; kc < NT / 2; ++kc) {
        a[kc][0] = pack(c[2 * kc][0], c[2 * kc][1]);
        a[kc][1] = pack(c[2 * kc][2], c[2 * kc][3]);
        a[kc][2] = pack(c[2 * kc + 1][0], c[2 * kc + 1][1]);
        a[kc][3] = pack(c[2 * kc + 1][2], c[2 * kc + 1][3]);
    }
}

template <int NT>
__device__ __forceinline__ void zero(float (&c)[NT][4])
{
#pragma unroll
    for (int i = 0; i < NT; ++i) c[i][0] = c[i][1] = c[i][2] = c[i][3] = 0.f;
}

// Sum over the four threads that share an accumulator row.
__device__ __forceinline__ float quad_sum(float x)
{
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
}

}  // namespace wmma16
}  // namespace still
