// Device helpers of the chunkwise prefills (the scalar-gated tensor-core
// kernels and the channel-gated ones): bf16 packing and swizzled tile rows,
// warp-level MMA fragments, and the unit lower triangular inverse of one
// 64-token chunk with split-bf16 operands.  Header-only, internal linkage in
// every translation unit that includes it.
#pragma once

#include "gdn_sm100.cuh"

#include <cuda_bf16.h>
#include <cstdint>

namespace gdn {
namespace {

using namespace sm100;

constexpr int kBarKey = 1;                      // named barrier id of the key-side threads
constexpr long long kSpinLimit = 2000000000LL;  // ~1 s of SM clocks per wait
constexpr int kLD = 68;                         // row stride of the fp32 64 x 64 matrix

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&p);
}
// 32 floats as 16 bf16 pairs, the even index in the low half (a TMEM row of
// a bf16 A operand)
__device__ __forceinline__ void pack_row(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
}

// Store 8*NCH floats (times `scale`) of one tile row as NCH swizzled 16-byte
// chunks starting at chunk c0.
template <int NCH, int N>
__device__ __forceinline__ void store_row(uint8_t *tile, uint32_t row, uint32_t c0,
                                          const float (&v)[N], float scale = 1.f) {
    static_assert(N == 8 * NCH, "row piece");
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
        uint4 w;
        w.x = pack_bf16(v[8 * k + 0] * scale, v[8 * k + 1] * scale);
        w.y = pack_bf16(v[8 * k + 2] * scale, v[8 * k + 3] * scale);
        w.z = pack_bf16(v[8 * k + 4] * scale, v[8 * k + 5] * scale);
        w.w = pack_bf16(v[8 * k + 6] * scale, v[8 * k + 7] * scale);
        *reinterpret_cast<uint4 *>(tile + swz128(row, c0 + k)) = w;
    }
}

// Inclusive prefix sum of log2(alpha) over a 64-token chunk held two per lane
// (tokens lane and lane + 32).  Past `nvalid` alpha counts as 1.
__device__ __forceinline__ void chunk_log2_prefix(float a0, float a1, int lane, int nvalid,
                                                  float &g0, float &g1) {
    g0 = lane < nvalid ? log2f(a0) : 0.f;
    g1 = lane + 32 < nvalid ? log2f(a1) : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float u0 = __shfl_up_sync(0xffffffffu, g0, off);
        const float u1 = __shfl_up_sync(0xffffffffu, g1, off);
        if (lane >= off) { g0 += u0; g1 += u1; }
    }
    g1 += __shfl_sync(0xffffffffu, g0, 31);
}

// Blocks of the fp32 64 x 64 matrix in AF (16 x 16 blocks, row stride kLD):
// A_ij at block position (i, j); the inverse writes D_i = (I + A_ii)^{-1} over
// the diagonal blocks.
__device__ __forceinline__ float *blk(float *AF, int i, int j) {
    return AF + 16 * i * kLD + 16 * j;
}

// ---- the unit lower triangular inverse T = (I + A)^{-1} of one chunk ----
//
// Blocked by 16 x 16: the diagonal blocks D_i = (I + A_ii)^{-1} by forward
// substitution in float32 on the CUDA cores (one column per thread), then the
// off-diagonal blocks from the block form of (I + A) T = I,
//
//     T_ij = -D_i sum_{m=j}^{i-1} A_im T_mj      (i > j),
//
// computed transposed, U = T^T: warp j owns block row j of U (block column j
// of T), U_ji = -(sum_m U_jm A_im^T) D_i^T, so each product's result is the
// left operand of the next one and never leaves the warp's registers.  These
// 16 x 16 x 16 products run on the register-level tensor-core MMA (mma.sync
// m16n8k16; tcgen05 starts at 64 rows and works from shared memory / TMEM,
// which would put a round trip on each of the chain's six dependent steps).
// Operands are float32 values split into bf16 pairs x = hi + lo and each
// product takes hi*hi + hi*lo + lo*hi with float32 accumulation: about 16
// significant bits, where T' and T'' are rounded to bf16 (8 bits) afterwards.

struct FragA {  // 16 x 16 left operand, hi and lo halves (m16n8k16 A layout)
    uint32_t h[4], l[4];
};
struct FragB {  // 16 x 16 right operand as two 16 x 8 column tiles
    uint32_t h[2][2], l[2][2];
};

__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8 x 8 bf16 matrices from shared memory; lane l gives the address of
// row l % 8 of matrix l / 8 and receives row l / 4, columns 2 (l % 4), +1 of
// each, in register order.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// One 16 x 16 block of P = (Q K^T) for rows t in [16 i, +16) and columns s in
// [16 j, +16) of a chunk, from its q and k boxes (64 tokens x 64 channels,
// 128-byte swizzled; q1 / k1 hold channels 64..127 when K = 128), as two
// 16 x 8 accumulator tiles of m16n8k16: d[nt] holds rows g, g + 8 and columns
// 8 nt + 2 t4, +1 (g = lane / 4, t4 = lane % 4).
template <int K>
__device__ __forceinline__ void qk_block(uint32_t q0, uint32_t q1, uint32_t k0, uint32_t k1,
                                         int i, int j, int lane, float (&d)[2][4]) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[nt][e] = 0.f;
    const uint32_t r = lane & 7, mtx = lane >> 3;
    // A: matrices (rows +0, k +0), (rows +8, k +0), (rows +0, k +8), (rows +8, k +8)
    const uint32_t arow = 16 * i + r + 8 * (mtx & 1), achunk = mtx >> 1;
    // B: (s +0, k +0), (s +0, k +8), (s +8, k +0), (s +8, k +8)
    const uint32_t brow = 16 * j + r + 8 * (mtx >> 1), bchunk = mtx & 1;
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks) {
        const uint32_t qb = ks < 4 ? q0 : q1, kb = ks < 4 ? k0 : k1;
        const uint32_t c = 2 * (ks & 3);
        uint32_t a[4], bb[4];
        ldsm_x4(a, qb + swz128(arow, c + achunk));
        ldsm_x4(bb, kb + swz128(brow, c + bchunk));
        mma_16816(d[0], a, bb[0], bb[1]);
        mma_16816(d[1], a, bb[2], bb[3]);
    }
}

// The three terms of A B with split operands (lo*hi, hi*lo, hi*hi) go to
// three accumulators (16 x 16 as two 16 x 8 tiles each), so consecutive
// products into the same result do not wait on one another.
__device__ __forceinline__ void mma_split(float (&d)[3][2][4], const FragA &a, const FragB &b) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        mma_16816(d[0][nt], a.l, b.h[nt][0], b.h[nt][1]);
        mma_16816(d[1][nt], a.h, b.l[nt][0], b.l[nt][1]);
        mma_16816(d[2][nt], a.h, b.h[nt][0], b.h[nt][1]);
    }
}
__device__ __forceinline__ void sum_split(const float (&d)[3][2][4], float (&r)[2][4]) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) r[nt][e] = (d[0][nt][e] + d[1][nt][e]) + d[2][nt][e];
}

// The accumulator layout of a 16 x 16 result (two 16 x 8 tiles) is the A
// layout of m16n8k16: row g = lane / 4 (+ 8), columns 2 (lane % 4) (+ 1, + 8).
__device__ __forceinline__ FragA frag_a(const float (&d)[2][4], float scale) {
    FragA a;
    split_bf16(scale * d[0][0], scale * d[0][1], a.h[0], a.l[0]);
    split_bf16(scale * d[0][2], scale * d[0][3], a.h[1], a.l[1]);
    split_bf16(scale * d[1][0], scale * d[1][1], a.h[2], a.l[2]);
    split_bf16(scale * d[1][2], scale * d[1][3], a.h[3], a.l[3]);
    return a;
}

// Right operand M^T for a 16 x 16 float32 block M (row stride kLD): element
// (k, n) of the operand is M[n][k], so each register pair is two adjacent
// elements of one row of M.
__device__ __forceinline__ FragB frag_bt(const float *M, int g, int t4) {
    FragB b;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const float *row = M + (8 * nt + g) * kLD + 2 * t4;
        const float2 p0 = *reinterpret_cast<const float2 *>(row);
        const float2 p1 = *reinterpret_cast<const float2 *>(row + 8);
        split_bf16(p0.x, p0.y, b.h[nt][0], b.l[nt][0]);
        split_bf16(p1.x, p1.y, b.h[nt][1], b.l[nt][1]);
    }
    return b;
}

// Block row J of U = T^T (warp J of the inverse): U_JJ = D_J^T, then
// U_Ji = -(sum_{m=J}^{i-1} U_Jm A_im^T) D_i^T for i > J; U_Ji = 0 for i < J.
// Each block goes to emit(i, u) in the accumulator layout as soon as it is
// formed, so only the left operands of the later products stay in registers.
// One code path for all four warps (J is warp-uniform, the block indices
// compile-time), so the four block rows share their instructions.
template <class Emit>
__device__ __forceinline__ void inverse_block_row(float *AF, int J, int g, int t4, Emit &&emit) {
    FragA ua[3];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float u[2][4];
        if (i < J) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) u[nt][e] = 0.f;
        } else if (i == J) {
            // U_JJ[r][c] = D_J[c][r]: rows g, g + 8, columns 8 nt + 2 t4 (+ 1)
            const float *D = blk(AF, i, i);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int c = 8 * nt + 2 * t4;
                u[nt][0] = D[c * kLD + g];
                u[nt][1] = D[(c + 1) * kLD + g];
                u[nt][2] = D[c * kLD + g + 8];
                u[nt][3] = D[(c + 1) * kLD + g + 8];
            }
            if (i < 3) ua[i] = frag_a(u, 1.f);
        } else {
            float acc[3][2][4] = {};
#pragma unroll
            for (int m = 0; m < i; ++m)
                if (m >= J) mma_split(acc, ua[m], frag_bt(blk(AF, i, m), g, t4));
            float x[2][4];
            sum_split(acc, x);
            const FragA xa = frag_a(x, -1.f);
            float acc2[3][2][4] = {};
            mma_split(acc2, xa, frag_bt(blk(AF, i, i), g, t4));
            sum_split(acc2, u);
            if (i < 3) ua[i] = frag_a(u, 1.f);
        }
        emit(i, u);
    }
}

// T = (I + A)^{-1} for the strictly lower 64 x 64 A in AF (fp32, zeros on
// and above the diagonal), and from it the bf16 operand tiles
//   T'^T  = diag(beta gamma) T^T,   T''^T = diag(beta) T^T
// each 64 rows (token s) of 64 tokens t, 128 bytes per row with the 128-byte
// swizzle: the MN-major image of the right operand of W^T = K^T T'^T and
// U~^T = V^T T''^T.  The tiles may be shared or global memory.  Run by NT
// threads (named barrier kBarKey): the first 64 solve the diagonal blocks,
// warps 0-3 the off-diagonal ones.  AF's diagonal blocks are overwritten.
template <int NT>
__device__ __forceinline__ void chunk_inverse_tprime(float *AF, const float *bet, const float *gam,
                                                     uint8_t *TPtile, uint8_t *TPPtile, int tid) {
    static_assert(NT >= 128 && NT % 32 == 0, "inverse thread mapping");
    {
        // D_i = (I + A_ii)^{-1}, column c of block i per thread
        float x[16];
        const int bb = tid >> 4, c = tid & 15;
        if (tid < 64) {
            const float *Ab = blk(AF, bb, bb);
#pragma unroll
            for (int t = 0; t < 16; ++t) x[t] = (t == c) ? 1.f : 0.f;
#pragma unroll
            for (int t = 1; t < 16; ++t) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int r = 0; r < t; r += 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(Ab + t * kLD + r);
                    a0 = fmaf(a.x, x[r], a0);
                    if (r + 1 < t) a1 = fmaf(a.y, x[r + 1], a1);
                    if (r + 2 < t) a0 = fmaf(a.z, x[r + 2], a0);
                    if (r + 3 < t) a1 = fmaf(a.w, x[r + 3], a1);
                }
                x[t] -= a0 + a1;
            }
        }
        named_sync(kBarKey, NT);  // every read of the diagonal A blocks done
        if (tid < 64) {
            float *Db = blk(AF, bb, bb);
#pragma unroll
            for (int t = 0; t < 16; ++t) Db[t * kLD + c] = x[t];
        }
        named_sync(kBarKey, NT);
    }
    const int warp = tid >> 5;
    if (warp < 4) {
        const int lane = tid & 31, g = lane >> 2, t4 = lane & 3;
        // rows s0 = 16 warp + g and s0 + 8 of T'^T and T''^T
        const int s0 = 16 * warp + g;
        const float b0 = bet[s0], b1 = bet[s0 + 8];
        const float bg0 = b0 * gam[s0], bg1 = b1 * gam[s0 + 8];
        inverse_block_row(AF, warp, g, t4, [&](int i, const float (&u)[2][4]) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int srow = s0 + 8 * hr;
                const float b = hr ? b1 : b0, bg = hr ? bg1 : bg0;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float v0 = u[nt][2 * hr], v1 = u[nt][2 * hr + 1];
                    const uint32_t off = swz128(srow, 2 * i + nt) + 4 * t4;
                    *reinterpret_cast<uint32_t *>(TPtile + off) = pack_bf16(v0 * bg, v1 * bg);
                    *reinterpret_cast<uint32_t *>(TPPtile + off) = pack_bf16(v0 * b, v1 * b);
                }
            }
        });
    }
}

// 2^x for x <= 0 (a decay between two tokens of a chunk) with the hardware
// approximation (relative error about 2^-22; results below 2^-126 flush to
// zero, far under the bf16 operands these factors scale).
__device__ __forceinline__ float decay_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace
}  // namespace gdn
