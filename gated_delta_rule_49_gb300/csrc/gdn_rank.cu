// Stable rank of recurrent states: er(S) = ||S||_F^2 / sigma_1(S)^2
// ("On State Reduction in Linear Attention" notes, Sec. 2.2, Eq. (5)).
//
// One CTA of 256 threads per state.  sigma_1^2 is the top eigenvalue of
// G = S^T S by power iteration: y = G x, lambda = x . y (Rayleigh quotient,
// |x| = 1), x <- y / |y| -- the same sequence as alternating S and S^T.  The
// start vector is x_j = 1 + j/K; if S x vanishes the iteration restarts from
// the coordinate vector of the largest column.  The loop stops once lambda
// moves by at most tol * lambda between checks, or after max_iter products.
//
// S is staged once in shared memory (rows zero-padded to 128 columns) and G is
// formed once, thread (r, c) accumulating the 8 x 8 block G[8r.., 8c..] in
// registers from float4 row reads; each product is then that block times
// x[8c..] (64 FMAs) and a shuffle reduction over the 16 threads of block row r
// (one half-warp).  The Rayleigh quotient and the renormalisation (block-wide
// reductions) come every 4 products, so tol is checked at that granularity;
// max_iter still counts products.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRankThreads = 256;
constexpr int kRankMaxDim = 128;
constexpr int kRankWarps = kRankThreads / 32;

// Sum of a and b over the CTA (one value each per thread); every thread gets
// both.  red: 2 * kRankWarps floats.
__device__ float2 block_sum2(float a, float b, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
    }
    __syncthreads();  // red may still be read from a previous call
    if (lane == 0) {
        red[warp] = a;
        red[kRankWarps + warp] = b;
    }
    __syncthreads();
    float2 t = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kRankWarps; ++w) {
        t.x += red[w];
        t.y += red[kRankWarps + w];
    }
    return t;
}

__global__ void __launch_bounds__(kRankThreads)
    state_rank_kernel(const float *__restrict__ S, int V, int K, float *__restrict__ fro2,
                      float *__restrict__ sigma1, float *__restrict__ er, int max_iter,
                      float tol, int *status) {
    extern __shared__ __align__(16) float smem[];
    constexpr int D = kRankMaxDim;
    float *Ss = smem;          // [V][D], columns >= K zero
    float *x = Ss + V * D;     // [D], entries >= K zero
    float *red = x + D;        // [2 * kRankWarps]
    const int tid = threadIdx.x;
    const int r = tid >> 4, c = tid & 15;  // 8 x 8 block (r, c) of G
    const float *Sm = S + (size_t)blockIdx.x * V * K;

    float f = 0.f;
    for (int e = tid; e < V * D; e += kRankThreads) {
        const int i = e / D, j = e % D;
        const float s = j < K ? Sm[(size_t)i * K + j] : 0.f;
        Ss[e] = s;
        f = fmaf(s, s, f);
    }
    for (int j = tid; j < D; j += kRankThreads) x[j] = j < K ? 1.f + (float)j / (float)K : 0.f;
    const float2 fn = block_sum2(f, tid < K ? x[tid] * x[tid] : 0.f, red);  // orders the writes
    const float F = fn.x;
    if (F == 0.f) {
        if (tid == 0) {
            fro2[blockIdx.x] = 0.f;
            sigma1[blockIdx.x] = 0.f;
            er[blockIdx.x] = 0.f;
            if (status) atomicOr(status, kStatusZeroState);
        }
        return;
    }

    // G block (r, c) = sum_i S[i][8r + a] S[i][8c + b]
    float g[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int bb = 0; bb < 8; ++bb) g[a][bb] = 0.f;
    for (int i = 0; i < V; ++i) {
        const float4 *row = reinterpret_cast<const float4 *>(Ss + i * D);
        const float4 ra = row[2 * r], rb = row[2 * r + 1];
        const float4 ca = row[2 * c], cb = row[2 * c + 1];
        const float sr[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
        const float sc[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) g[a][bb] = fmaf(sr[a], sc[bb], g[a][bb]);
    }

    float inv = rsqrtf(fn.y);  // normalise the start vector
    __syncthreads();           // every thread has read fn.y's inputs from x
    for (int j = tid; j < D; j += kRankThreads) x[j] *= inv;
    __syncthreads();

    // The iterate is renormalised and lambda checked every kBlock products;
    // in between, y is scaled by 1 / (the latest eigenvalue estimate, or
    // ||S||_F^2 at first), which keeps it near unit size without a reduction.
    constexpr int kBlock = 4;
    float lambda = 0.f, prev = -1.f, scale = 1.f / F;
    bool restarted = false;
    for (int it = 0; it < max_iter;) {
        const int steps = min(kBlock, max_iter - it);
        float y[8], xr[8];
        for (int st = 0; st < steps; ++st) {
            // y[8r + a] = sum_c G block (r, c) x[8c..], reduced over the half-warp
            const float4 xa = reinterpret_cast<const float4 *>(x)[2 * c];
            const float4 xb = reinterpret_cast<const float4 *>(x)[2 * c + 1];
            const float xc[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                float acc = 0.f;
#pragma unroll
                for (int bb = 0; bb < 8; ++bb) acc = fmaf(g[a][bb], xc[bb], acc);
                y[a] = acc;
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
#pragma unroll
                for (int a = 0; a < 8; ++a) y[a] += __shfl_xor_sync(0xffffffffu, y[a], off);
            if (c == 0) {
                const float4 xr0 = reinterpret_cast<const float4 *>(x)[2 * r];
                const float4 xr1 = reinterpret_cast<const float4 *>(x)[2 * r + 1];
                xr[0] = xr0.x; xr[1] = xr0.y; xr[2] = xr0.z; xr[3] = xr0.w;
                xr[4] = xr1.x; xr[5] = xr1.y; xr[6] = xr1.z; xr[7] = xr1.w;
            }
            if (st + 1 < steps) {
                __syncthreads();  // every read of x done
                if (c == 0) {
                    reinterpret_cast<float4 *>(x)[2 * r] =
                        make_float4(y[0] * scale, y[1] * scale, y[2] * scale, y[3] * scale);
                    reinterpret_cast<float4 *>(x)[2 * r + 1] =
                        make_float4(y[4] * scale, y[5] * scale, y[6] * scale, y[7] * scale);
                }
                __syncthreads();
            }
        }
        it += steps;
        // Rayleigh quotient of the block's last iterate x (|x| not 1 here)
        float lp = 0.f, yp = 0.f, xp = 0.f;
        if (c == 0) {
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                lp = fmaf(xr[a], y[a], lp);
                yp = fmaf(y[a], y[a], yp);
                xp = fmaf(xr[a], xr[a], xp);
            }
        }
        const float2 ly = block_sum2(lp, yp, red);  // barrier: every read of x done
        const float xx = block_sum2(xp, 0.f, red).x;
        lambda = xx > 0.f ? ly.x / xx : 0.f;
        if (lambda <= 0.f) {  // (a NaN state runs on and reports NaN)
            lambda = 0.f;
            if (restarted) break;
            // S x = 0 although S != 0: restart from the largest column's axis
            restarted = true;
            if (tid == 0) {
                int best = 0;
                float bn = -1.f;
                for (int j = 0; j < K; ++j) {
                    float cn = 0.f;
                    for (int i = 0; i < V; ++i) cn = fmaf(Ss[i * D + j], Ss[i * D + j], cn);
                    if (cn > bn) { bn = cn; best = j; }
                }
                for (int j = 0; j < D; ++j) x[j] = (j == best) ? 1.f : 0.f;
            }
            __syncthreads();
            prev = -1.f;
            continue;
        }
        const bool done = prev >= 0.f && fabsf(lambda - prev) <= tol * lambda;
        prev = lambda;
        scale = 1.f / lambda;
        if (done || it >= max_iter) break;
        // x = y / |y|
        if (c == 0) {
            const float s = rsqrtf(ly.y);
            reinterpret_cast<float4 *>(x)[2 * r] =
                make_float4(y[0] * s, y[1] * s, y[2] * s, y[3] * s);
            reinterpret_cast<float4 *>(x)[2 * r + 1] =
                make_float4(y[4] * s, y[5] * s, y[6] * s, y[7] * s);
        }
        __syncthreads();
    }
    if (tid == 0) {
        fro2[blockIdx.x] = F;
        sigma1[blockIdx.x] = sqrtf(lambda);
        er[blockIdx.x] = lambda > 0.f ? F / lambda : 0.f;
    }
}

}  // namespace

cudaError_t launch_state_rank(const float *S, int BH, int V, int K, float *fro2,
                              float *sigma1, float *er, int max_iter, float tol,
                              cudaStream_t stream) {
    if (V > kRankMaxDim || K > kRankMaxDim) return cudaErrorInvalidValue;
    const size_t smem = sizeof(float) * ((size_t)V * kRankMaxDim + kRankMaxDim + 2 * kRankWarps);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(
            state_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    state_rank_kernel<<<BH, kRankThreads, smem, stream>>>(S, V, K, fro2, sigma1, er, max_iter,
                                                         tol, device_status_ptr());
    return cudaGetLastError();
}

}  // namespace gdn
