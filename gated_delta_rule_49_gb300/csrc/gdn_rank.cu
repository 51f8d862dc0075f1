// Stable rank of recurrent states: er(S) = ||S||_F^2 / sigma_1(S)^2
// ("On State Reduction in Linear Attention" notes, Sec. 2.2, Eq. (5)).
//
// One CTA per state.  The V x K matrix is staged once in shared memory with an
// odd row stride (conflict-free row and column walks); sigma_1^2 is the top
// eigenvalue of S^T S by power iteration: y = S x, lambda = |y|^2 (Rayleigh
// quotient, |x| = 1), x <- S^T y / |S^T y|.  The start vector is
// x_j = 1 + j/K; if S x happens to vanish the iteration restarts from the
// coordinate vector of the largest column.  The loop stops once lambda moves
// by at most tol * lambda, or after max_iter iterations.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRankThreads = 256;
constexpr int kRankMaxDim = 128;

__device__ float block_sum(float x, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    __syncthreads();  // red may still be read from a previous call
    if (lane == 0) red[warp] = x;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kRankThreads / 32; ++w) t += red[w];
    return t;
}

__global__ void __launch_bounds__(kRankThreads)
    state_rank_kernel(const float *__restrict__ S, int V, int K, float *__restrict__ fro2,
                      float *__restrict__ sigma1, float *__restrict__ er, int max_iter,
                      float tol, int *status) {
    extern __shared__ float smem[];
    const int ld = K + 1;
    float *Ss = smem;               // [V][K+1]
    float *x = Ss + V * ld;         // [K]
    float *y = x + kRankMaxDim;     // [V]
    float *red = y + kRankMaxDim;   // [kRankThreads / 32]
    const int tid = threadIdx.x;
    const float *Sm = S + (size_t)blockIdx.x * V * K;

    float f = 0.f;
    for (int e = tid; e < V * K; e += kRankThreads) {
        const float s = Sm[e];
        Ss[(e / K) * ld + (e % K)] = s;
        f = fmaf(s, s, f);
    }
    const float F = block_sum(f, red);  // also orders the staging writes
    if (F == 0.f) {
        if (tid == 0) {
            fro2[blockIdx.x] = 0.f;
            sigma1[blockIdx.x] = 0.f;
            er[blockIdx.x] = 0.f;
            if (status) atomicOr(status, kStatusZeroState);
        }
        return;
    }

    // start vector x_j = 1 + j/K, normalised
    float n2 = 0.f;
    for (int j = tid; j < K; j += kRankThreads) {
        const float xj = 1.f + (float)j / (float)K;
        x[j] = xj;
        n2 += xj * xj;
    }
    float inv = rsqrtf(block_sum(n2, red));
    for (int j = tid; j < K; j += kRankThreads) x[j] *= inv;
    __syncthreads();

    float lambda = 0.f, prev = -1.f;
    bool restarted = false;
    for (int it = 0; it < max_iter; ++it) {
        // y = S x
        float l = 0.f;
        for (int i = tid; i < V; i += kRankThreads) {
            float acc = 0.f;
            const float *row = Ss + i * ld;
            for (int j = 0; j < K; ++j) acc = fmaf(row[j], x[j], acc);
            y[i] = acc;
            l = fmaf(acc, acc, l);
        }
        lambda = block_sum(l, red);  // barrier: y visible to all
        if (lambda == 0.f) {
            if (restarted) break;
            // S x = 0 although S != 0: restart from the largest column's axis
            restarted = true;
            if (tid == 0) {
                int best = 0;
                float bn = -1.f;
                for (int j = 0; j < K; ++j) {
                    float c = 0.f;
                    for (int i = 0; i < V; ++i) c = fmaf(Ss[i * ld + j], Ss[i * ld + j], c);
                    if (c > bn) { bn = c; best = j; }
                }
                for (int j = 0; j < K; ++j) x[j] = (j == best) ? 1.f : 0.f;
            }
            __syncthreads();
            prev = -1.f;
            continue;
        }
        const bool done = prev >= 0.f && fabsf(lambda - prev) <= tol * lambda;
        prev = lambda;
        if (done || it + 1 == max_iter) break;
        // x = S^T y / |S^T y|
        float z2 = 0.f;
        float zj_local[kRankMaxDim / kRankThreads + 1];
        int c = 0;
        for (int j = tid; j < K; j += kRankThreads, ++c) {
            float acc = 0.f;
            for (int i = 0; i < V; ++i) acc = fmaf(Ss[i * ld + j], y[i], acc);
            zj_local[c] = acc;
            z2 = fmaf(acc, acc, z2);
        }
        inv = rsqrtf(block_sum(z2, red));  // barrier: all reads of x done
        c = 0;
        for (int j = tid; j < K; j += kRankThreads, ++c) x[j] = zj_local[c] * inv;
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
    const size_t smem =
        sizeof(float) * ((size_t)V * (K + 1) + 2 * kRankMaxDim + kRankThreads / 32);
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
