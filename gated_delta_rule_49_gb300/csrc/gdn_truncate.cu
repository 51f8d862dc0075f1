// Rank-r truncation of states ("How much of a Gated DeltaNet state is used"
// blog, Sec. 3): S <- U_r U_r^T S, U_r the left singular vectors of the r
// largest singular values, plus the singular values themselves.
//
// One CTA per state, everything in shared memory.  One-sided (Hestenes)
// Jacobi on the K columns of S: each round of the round-robin ordering
// rotates K/2 disjoint column pairs at once (8 lanes per pair, the column's
// V entries spread as float4 pieces at offsets 32 i + 4 l, so the 8 lanes of
// a pair read 128 contiguous bytes per access), with the rotation that makes
// the pair orthogonal:
//
//   a = |c_p|^2, b = |c_q|^2, g = c_p . c_q,  zeta = (b - a) / (2 g),
//   t = sign(zeta) / (|zeta| + sqrt(1 + zeta^2)),  c = 1/sqrt(1 + t^2), s = c t,
//   c_p <- c c_p - s c_q,   c_q <- s c_p + c c_q,
//
// skipped when |g| <= sqrt(V) eps sqrt(a b) (columns orthogonal to float32
// precision) or |g| <= 1e-12 |S|_F^2 (a coupling far below anything that can
// move the singular values or subspaces at float32 precision; without this
// floor the noise-level columns of a low-rank state keep the sweeps going).
// The rotation itself uses fast reciprocal / square-root forms: an angle that
// is off in the last bits leaves a residual the next sweep removes.  Sweeps repeat until one rotates nothing
// (or max_sweeps; then the not-converged status bit is set).  The converged
// columns are sigma_i u_i; with u_i their directions, W = U^T S (against a
// copy of the original S) has row norms sigma_i, the r largest select U_r,
// and S <- U_r W_r.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kLanesPerPair = 8;
// Orthogonality threshold |g| <= sqrt(V) eps sqrt(a b), eps = 2^-24 (float32).
template <int V>
__host__ __device__ constexpr float jacobi_tol() { return V == 128 ? 6.75e-7f : 3.38e-7f; }

template <int V, int K>
struct TruncSmem {
    static constexpr int A = 0;                       // [K][V] rotated columns
    static constexpr int S = A + K * V * 4;           // [V][K] original state
    static constexpr int W = S + V * K * 4;           // [K][K] U^T S
    static constexpr int NRM = W + K * K * 4;         // [K] 1 / column norms
    static constexpr int SEL = NRM + K * 4;           // [K] column of rank i
    static constexpr int BYTES = SEL + K * 4;
};

__device__ __forceinline__ void pair_of(int round, int m, int n, int &p, int &q) {
    if (m == 0) {
        p = n - 1;
        q = round;
    } else {
        p = (round + m) % (n - 1);
        q = (round + n - 1 - m) % (n - 1);
    }
}

template <int V, int K>
__global__ void __launch_bounds__(K / 2 * kLanesPerPair)
    truncate_kernel(float *__restrict__ Sg, int r, float *__restrict__ sigma, int max_sweeps,
                    int *status) {
    using L = TruncSmem<V, K>;
    constexpr int NCH = V / 32;  // float4 pieces per lane per column
    constexpr int NT = K / 2 * kLanesPerPair;
    extern __shared__ __align__(16) unsigned char smem[];
    float *A = reinterpret_cast<float *>(smem + L::A);
    float *Sc = reinterpret_cast<float *>(smem + L::S);
    float *W = reinterpret_cast<float *>(smem + L::W);
    float *nrm = reinterpret_cast<float *>(smem + L::NRM);
    int *sel = reinterpret_cast<int *>(smem + L::SEL);
    __shared__ int rotated;

    __shared__ float fro2;
    const int tid = threadIdx.x;
    if (tid == 0) fro2 = 0.f;
    __syncthreads();
    float *Sh = Sg + (size_t)blockIdx.x * V * K;
    float part = 0.f;
    for (int e = tid * 4; e < V * K; e += NT * 4) {
        const float4 x = *reinterpret_cast<const float4 *>(Sh + e);
        part += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
        *reinterpret_cast<float4 *>(Sc + e) = x;
        const int v = e / K, c = e % K;
        A[(c + 0) * V + v] = x.x;
        A[(c + 1) * V + v] = x.y;
        A[(c + 2) * V + v] = x.z;
        A[(c + 3) * V + v] = x.w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((tid & 31) == 0) atomicAdd(&fro2, part);
    __syncthreads();
    const float floor_g = 1e-12f * fro2;
    const float tol2 = jacobi_tol<V>() * jacobi_tol<V>();

    const int m = tid / kLanesPerPair, l = tid % kLanesPerPair;
    bool converged = false;
    for (int sweep = 0; sweep < max_sweeps && !converged; ++sweep) {
        if (tid == 0) rotated = 0;
        __syncthreads();
        int p, q;
        pair_of(0, m, K, p, q);
        for (int round = 0; round < K - 1; ++round) {
            float4 cp[NCH], cq[NCH];
            float a = 0.f, b = 0.f, g = 0.f;
#pragma unroll
            for (int i = 0; i < NCH; ++i) {
                cp[i] = *reinterpret_cast<const float4 *>(A + p * V + 32 * i + 4 * l);
                cq[i] = *reinterpret_cast<const float4 *>(A + q * V + 32 * i + 4 * l);
                a += cp[i].x * cp[i].x + cp[i].y * cp[i].y + cp[i].z * cp[i].z + cp[i].w * cp[i].w;
                b += cq[i].x * cq[i].x + cq[i].y * cq[i].y + cq[i].z * cq[i].z + cq[i].w * cq[i].w;
                g += cp[i].x * cq[i].x + cp[i].y * cq[i].y + cp[i].z * cq[i].z + cp[i].w * cq[i].w;
            }
#pragma unroll
            for (int off = kLanesPerPair / 2; off > 0; off >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                b += __shfl_xor_sync(0xffffffffu, b, off);
                g += __shfl_xor_sync(0xffffffffu, g, off);
            }
            if (fabsf(g) > floor_g && g * g > tol2 * a * b) {
                const float zeta = __fdividef(b - a, 2.f * g);
                const float az = fabsf(zeta);
                float t;
                if (az > 1e18f) {
                    t = __fdividef(0.5f, zeta);
                } else {
                    const float e1 = fmaf(zeta, zeta, 1.f);
                    t = __fdividef(copysignf(1.f, zeta), az + e1 * rsqrtf(e1));
                }
                const float c = rsqrtf(fmaf(t, t, 1.f));
                const float s = c * t;
#pragma unroll
                for (int i = 0; i < NCH; ++i) {
                    const float4 x = cp[i], y = cq[i];
                    *reinterpret_cast<float4 *>(A + p * V + 32 * i + 4 * l) =
                        make_float4(c * x.x - s * y.x, c * x.y - s * y.y, c * x.z - s * y.z,
                                    c * x.w - s * y.w);
                    *reinterpret_cast<float4 *>(A + q * V + 32 * i + 4 * l) =
                        make_float4(s * x.x + c * y.x, s * x.y + c * y.y, s * x.z + c * y.z,
                                    s * x.w + c * y.w);
                }
                if (l == 0) rotated = 1;
            }
            __syncthreads();
            // next round of the round-robin ordering: every index but K - 1 steps by one mod K - 1
            if (m != 0) p = p == K - 2 ? 0 : p + 1;
            q = q == K - 2 ? 0 : q + 1;
        }
        converged = rotated == 0;
        __syncthreads();  // everyone has read `rotated` before it is reset
    }
    if (!converged && tid == 0 && status) atomicOr(status, kStatusNotConverged);

    // Directions u_c = c_c / |c_c| of the converged columns.  Their lengths
    // are not used as singular values: rotations that are orthogonal only to
    // rounding let the lengths drift over a few thousand rotations while the
    // directions stay accurate.  So W = U^T S is formed against the original
    // S for every column and sigma_c = |W[c]|.
    for (int c = tid; c < K; c += NT) {
        float n2 = 0.f;
        for (int v = 0; v < V; ++v) n2 = fmaf(A[c * V + v], A[c * V + v], n2);
        nrm[c] = n2 > 0.f ? rsqrtf(n2) : 0.f;  // 1 / |c_c| (0 for a zero column)
    }
    __syncthreads();
    constexpr int JS = NT / K;  // thread (j0, kk): rows j0, j0 + JS, ... of column kk
    const int kk = tid % K, j0 = tid / K;
    for (int j = j0; j < K; j += JS) {
        float acc = 0.f;
        for (int v = 0; v < V; ++v) acc = fmaf(A[j * V + v], Sc[v * K + kk], acc);
        W[j * K + kk] = acc * nrm[j];
    }
    __syncthreads();
    float *sig2 = Sc;  // the copy of S is no longer needed: reuse it for sigma^2
    for (int c = tid; c < K; c += NT) {
        float s2 = 0.f;
        for (int k = 0; k < K; ++k) s2 = fmaf(W[c * K + k], W[c * K + k], s2);
        sig2[c] = s2;
    }
    __syncthreads();
    for (int c = tid; c < K; c += NT) {  // rank of each column, ties by index
        const float sc = sig2[c];
        int rank = 0;
        for (int j = 0; j < K; ++j) rank += (sig2[j] > sc) || (sig2[j] == sc && j < c);
        sel[rank] = c;
    }
    __syncthreads();
    if (sigma)
        for (int i = tid; i < K; i += NT) sigma[(size_t)blockIdx.x * K + i] = sqrtf(sig2[sel[i]]);
    if (r >= K) return;  // nothing to cut (K <= V for every supported variant)

    // S <- U_r W_r
    for (int v = j0; v < V; v += JS) {
        float acc = 0.f;
        for (int j = 0; j < r; ++j) {
            const int c = sel[j];
            acc = fmaf(A[c * V + v] * nrm[c], W[c * K + kk], acc);
        }
        Sh[(size_t)v * K + kk] = acc;
    }
}

template <int V, int K>
cudaError_t launch_trunc_t(float *S, int BH, int r, float *sigma, int max_sweeps,
                           cudaStream_t stream) {
    using L = TruncSmem<V, K>;
    auto kern = truncate_kernel<V, K>;
    static uintptr_t attr_set[64] = {};  // context the attributes were set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev] != context_key()) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = context_key();
    }
    kern<<<BH, K / 2 * kLanesPerPair, L::BYTES, stream>>>(S, r, sigma, max_sweeps,
                                                          device_status_ptr());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_truncate(float *S, int BH, int V, int K, int r, float *sigma,
                                  int max_sweeps, cudaStream_t stream) {
    if (V == 128 && K == 128) return launch_trunc_t<128, 128>(S, BH, r, sigma, max_sweeps, stream);
    if (V == 128 && K == 64) return launch_trunc_t<128, 64>(S, BH, r, sigma, max_sweeps, stream);
    if (V == 32 && K == 32) return launch_trunc_t<32, 32>(S, BH, r, sigma, max_sweeps, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
