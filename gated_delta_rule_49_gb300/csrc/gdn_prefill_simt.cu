// Chunkwise prefill on CUDA cores, all arithmetic in float32.
//
// This is the float32-mode prefill (and the bf16 prefill of the small
// (32, 32) variant).  One CTA owns one (b, h) sequence and a slab of VS value
// rows; value rows are independent systems ("On State Reduction in Linear
// Attention" notes, Sec. 2.5), so slabs of one head run in parallel and only
// the key-side chunk work is repeated per slab.
//
// Per 64-token chunk, with G_t the in-chunk cumulative log-decay,
// gamma_t = exp(G_t) and Gamma_ts = exp(G_t - G_s) (always <= 1, formed as a
// difference, never as a ratio of gammas):
//
//   A_ts = beta_t Gamma_ts (k_t . k_s), s < t      P_ts = Gamma_ts (q_t . k_s), s <= t
//   (I + A) [W | U~] = [diag(beta gamma) K | diag(beta) V]   (forward substitution)
//   U    = U~ - W S^T                     pseudo-values u_t = beta_t (v_t - alpha_t S_{t-1} k_t)
//   O    = diag(gamma) Q S^T + P U
//   S   <- gamma_C S + U^T diag(exp(G_C - G_s)) K
//
// which is the token recurrence unrolled over the chunk (the pseudo-value
// rewriting of the delta rule in the notes' Sec. 2.3).  A ragged last chunk
// is padded with k = q = v = 0, beta = 0, log alpha = 0.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kSimtThreads = 256;
constexpr int C = kChunk;

template <int K, int VS>
struct SimtSmem {
    static constexpr int LK = K + 1, LV = VS + 1, LC = C + 1;
    static constexpr int kKs = 0;
    static constexpr int kQs = kKs + C * LK;
    static constexpr int kW = kQs + C * LK;
    static constexpr int kVs = kW + C * LK;
    static constexpr int kU = kVs + C * LV;
    static constexpr int kA = kU + C * LV;
    static constexpr int kP = kA + C * LC;
    static constexpr int kS = kP + C * LC;
    static constexpr int kG = kS + VS * LK;
    static constexpr int kGam = kG + C;
    static constexpr int kBeta = kGam + C;
    static constexpr int kDecay = kBeta + C;
    static constexpr int kTotal = kDecay + C;
    static constexpr size_t bytes = sizeof(float) * kTotal;
};

template <int K, int VS, typename Tin>
__global__ void __launch_bounds__(kSimtThreads, 1)
    prefill_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                        const Tin *__restrict__ v, const float *__restrict__ alpha,
                        const float *__restrict__ beta, const float *__restrict__ S0,
                        Tin *__restrict__ o, float *__restrict__ ST, int T, int Ts, int H,
                        int V) {
    using L = SimtSmem<K, VS>;
    extern __shared__ float sm[];
    float *Ks = sm + L::kKs;
    float *Qs = sm + L::kQs;
    float *Wm = sm + L::kW;
    float *Vsm = sm + L::kVs;
    float *Um = sm + L::kU;
    float *Am = sm + L::kA;
    float *Pm = sm + L::kP;
    float *Ss = sm + L::kS;
    float *Gs = sm + L::kG;
    float *gam = sm + L::kGam;
    float *bet = sm + L::kBeta;
    float *dcy = sm + L::kDecay;

    const int tid = threadIdx.x;
    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int i0 = slab * VS;  // first value row of this slab
    const size_t seq = (size_t)b * H + h;

    // state slab -> shared
    for (int e = tid; e < VS * K; e += kSimtThreads) {
        const int i = e / K, j = e % K;
        Ss[i * L::LK + j] = S0 ? S0[(seq * V + i0 + i) * K + j] : 0.f;
    }

    for (int c0 = 0; c0 < T; c0 += C) {
        const int n = min(C, T - c0);
        __syncthreads();  // previous chunk fully consumed
        // ---- load the chunk (zero-padded past n) ----
        for (int e = tid; e < C * K; e += kSimtThreads) {
            const int t = e / K, j = e % K;
            float kv = 0.f, qv = 0.f;
            if (t < n) {
                const size_t off = (((size_t)b * Ts + c0 + t) * H + h) * K + j;
                kv = to_f32(k[off]);
                qv = to_f32(q[off]);
            }
            Ks[t * L::LK + j] = kv;
            Qs[t * L::LK + j] = qv;
        }
        for (int e = tid; e < C * VS; e += kSimtThreads) {
            const int t = e / VS, i = e % VS;
            float vv = 0.f;
            if (t < n) vv = to_f32(v[(((size_t)b * Ts + c0 + t) * H + h) * V + i0 + i]);
            Vsm[t * L::LV + i] = vv;
        }
        if (tid < 32) {
            // in-chunk inclusive prefix sum of log alpha over 64 tokens
            const int t0 = tid, t1 = tid + 32;
            const size_t g0i = ((size_t)b * Ts + c0 + t0) * H + h;
            const size_t g1i = ((size_t)b * Ts + c0 + t1) * H + h;
            float g0 = t0 < n ? logf(alpha[g0i]) : 0.f;
            float g1 = t1 < n ? logf(alpha[g1i]) : 0.f;
            bet[t0] = t0 < n ? beta[g0i] : 0.f;
            bet[t1] = t1 < n ? beta[g1i] : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float a0 = __shfl_up_sync(0xffffffffu, g0, off);
                const float a1 = __shfl_up_sync(0xffffffffu, g1, off);
                if (tid >= off) { g0 += a0; g1 += a1; }
            }
            g1 += __shfl_sync(0xffffffffu, g0, 31);
            Gs[t0] = g0;
            Gs[t1] = g1;
            gam[t0] = expf(g0);
            gam[t1] = expf(g1);
            const float gC = __shfl_sync(0xffffffffu, g1, 31);
            dcy[t0] = expf(gC - g0);
            dcy[t1] = expf(gC - g1);
        }
        __syncthreads();

        // ---- A (strictly lower) and P (lower incl. diagonal) ----
        {
            const int t = tid % C;
            const int sb = (tid / C) * (C / (kSimtThreads / C));
            constexpr int NS = C / (kSimtThreads / C);  // 16 columns per thread
            float accA[NS], accP[NS];
#pragma unroll
            for (int c = 0; c < NS; ++c) { accA[c] = 0.f; accP[c] = 0.f; }
            for (int j = 0; j < K; ++j) {
                const float kt = Ks[t * L::LK + j];
                const float qt = Qs[t * L::LK + j];
#pragma unroll
                for (int c = 0; c < NS; ++c) {
                    const float ks = Ks[(sb + c) * L::LK + j];
                    accA[c] = fmaf(kt, ks, accA[c]);
                    accP[c] = fmaf(qt, ks, accP[c]);
                }
            }
            const float Gt = Gs[t], bt = bet[t];
#pragma unroll
            for (int c = 0; c < NS; ++c) {
                const int s = sb + c;
                const float d = s <= t ? expf(Gt - Gs[s]) : 0.f;
                Am[t * L::LC + s] = s < t ? bt * d * accA[c] : 0.f;
                Pm[t * L::LC + s] = d * accP[c];
            }
        }
        __syncthreads();

        // ---- forward substitution, one thread per right-hand-side column ----
        for (int col = tid; col < K + VS; col += kSimtThreads) {
            float x[C];
            if (col < K) {
#pragma unroll
                for (int t = 0; t < C; ++t) x[t] = bet[t] * gam[t] * Ks[t * L::LK + col];
            } else {
#pragma unroll
                for (int t = 0; t < C; ++t) x[t] = bet[t] * Vsm[t * L::LV + (col - K)];
            }
#pragma unroll
            for (int t = 1; t < C; ++t) {
                float acc = x[t];
#pragma unroll
                for (int s = 0; s < t; ++s) acc = fmaf(-Am[t * L::LC + s], x[s], acc);
                x[t] = acc;
            }
            if (col < K) {
#pragma unroll
                for (int t = 0; t < C; ++t) Wm[t * L::LK + col] = x[t];
            } else {
#pragma unroll
                for (int t = 0; t < C; ++t) Um[t * L::LV + (col - K)] = x[t];
            }
        }
        __syncthreads();

        // ---- U = U~ - W S^T and O = diag(gamma) Q S^T + P U ----
        {
            const int t = tid % C;
            constexpr int NI = VS / (kSimtThreads / C);  // value rows per thread
            const int ib = (tid / C) * NI;
            float u[NI], oq[NI];
#pragma unroll
            for (int c = 0; c < NI; ++c) { u[c] = Um[t * L::LV + ib + c]; oq[c] = 0.f; }
            for (int j = 0; j < K; ++j) {
                const float w = Wm[t * L::LK + j];
                const float qq = Qs[t * L::LK + j];
#pragma unroll
                for (int c = 0; c < NI; ++c) {
                    const float s = Ss[(ib + c) * L::LK + j];
                    u[c] = fmaf(-w, s, u[c]);
                    oq[c] = fmaf(qq, s, oq[c]);
                }
            }
            __syncthreads();  // all reads of U~ done before U overwrites it
#pragma unroll
            for (int c = 0; c < NI; ++c) Um[t * L::LV + ib + c] = u[c];
            __syncthreads();
            if (o != nullptr) {
                const float gt = gam[t];
#pragma unroll
                for (int c = 0; c < NI; ++c) oq[c] *= gt;
                for (int s = 0; s <= t; ++s) {
                    const float p = Pm[t * L::LC + s];
#pragma unroll
                    for (int c = 0; c < NI; ++c) oq[c] = fmaf(p, Um[s * L::LV + ib + c], oq[c]);
                }
                if (t < n) {
                    Tin *orow = o + (((size_t)b * Ts + c0 + t) * H + h) * V + i0 + ib;
#pragma unroll
                    for (int c = 0; c < NI; ++c) orow[c] = from_f32<Tin>(oq[c]);
                }
            }
        }
        // No barrier here: the state update below reads only U, K and the
        // decay factors, which are final, and each thread rewrites only the
        // state entries that it alone reads; nothing reads S after the
        // barrier that followed the U write.

        // ---- S <- gamma_C S + U^T diag(exp(G_C - G)) K ----
        {
            constexpr int NG = kSimtThreads / K;  // row groups
            constexpr int NR = VS / NG;           // rows per thread
            const float gC = gam[C - 1];
            const int j = tid % K;
            const int rb = (tid / K) * NR;
            float acc[NR];
#pragma unroll
            for (int c = 0; c < NR; ++c) acc[c] = gC * Ss[(rb + c) * L::LK + j];
            for (int s = 0; s < C; ++s) {
                const float kd = dcy[s] * Ks[s * L::LK + j];
#pragma unroll
                for (int c = 0; c < NR; ++c) acc[c] = fmaf(Um[s * L::LV + rb + c], kd, acc[c]);
            }
#pragma unroll
            for (int c = 0; c < NR; ++c) Ss[(rb + c) * L::LK + j] = acc[c];
        }
    }
    __syncthreads();
    if (ST != nullptr) {
        for (int e = tid; e < VS * K; e += kSimtThreads) {
            const int i = e / K, j = e % K;
            ST[(seq * V + i0 + i) * K + j] = Ss[i * L::LK + j];
        }
    }
}

template <int K, int VS, typename Tin>
cudaError_t launch_simt_t(const void *q, const void *k, const void *v, const float *alpha,
                          const float *beta, const float *S0, void *o, float *ST, int B,
                          int T, int Ts, int H, int V, cudaStream_t stream) {
    static_assert(kSimtThreads % C == 0 && VS % (kSimtThreads / C) == 0, "tiling");
    static_assert(K <= kSimtThreads && kSimtThreads % K == 0 && VS % (kSimtThreads / K) == 0,
                  "tiling");
    if (V % VS != 0) return cudaErrorInvalidValue;
    const size_t smem = SimtSmem<K, VS>::bytes;
    auto kern = prefill_simt_kernel<K, VS, Tin>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    if (B > 65535 || H > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(V / VS, H, B);
    kern<<<grid, kSimtThreads, smem, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        alpha, beta, S0, static_cast<Tin *>(o), ST, T, Ts, H, V);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_simt(const void *q, const void *k, const void *v,
                                const float *alpha, const float *beta, const float *S0,
                                void *o, float *ST, int B, int T, int Ts, int H, int K, int V,
                                gdn_dtype dt, cudaStream_t stream) {
    const bool bf = dt == GDN_BF16;
    if (K == 32 && V == 32)
        return bf ? launch_simt_t<32, 32, __nv_bfloat16>(q, k, v, alpha, beta, S0, o, ST, B, T,
                                                        Ts, H, V, stream)
                  : launch_simt_t<32, 32, float>(q, k, v, alpha, beta, S0, o, ST, B, T, Ts, H,
                                                V, stream);
    if (K == 64 && V == 128)
        return bf ? launch_simt_t<64, 32, __nv_bfloat16>(q, k, v, alpha, beta, S0, o, ST, B, T,
                                                        Ts, H, V, stream)
                  : launch_simt_t<64, 32, float>(q, k, v, alpha, beta, S0, o, ST, B, T, Ts, H,
                                                V, stream);
    if (K == 128 && V == 128)
        return bf ? launch_simt_t<128, 32, __nv_bfloat16>(q, k, v, alpha, beta, S0, o, ST, B,
                                                         T, Ts, H, V, stream)
                  : launch_simt_t<128, 32, float>(q, k, v, alpha, beta, S0, o, ST, B, T, Ts, H,
                                                 V, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
