// Fused decode step: one read and one write of every state row.
//
// Each value channel i (row s of S, K floats) is an independent system given
// (k, q, alpha, beta) -- "On State Reduction in Linear Attention" notes,
// Sec. 2.5 -- so a group of K/4 lanes owns one row as float4 pieces and does
//
//     s <- alpha s                     (forget first)
//     p <- s . k,  r <- s . q          (two dot products, one pass, shuffles)
//     u <- beta (v_i - p)              (error of the decayed state)
//     s <- s + u k                     (write, stored back in place)
//     o_i <- r + u (k . q)             (= (alpha s_old + u k) . q)
//
// Layout: S [B, H, V, K] float32 (K contiguous, 16-byte aligned rows);
// q, k [B, H, K]; v, o [B, H, V]; alpha, beta [B, H].
//
// The gathering variant reads full-width q, k [B, H, K_in] and keeps channels
// idx[h, 0..K) of each head, renormalised over the kept coordinates (the
// pruning prologue of "On State Reduction" notes, Sec. 2.6, fused into the
// step: no separate pass over q and k).
// The kernel is HBM-bound: 8 V K bytes of state traffic per head.  Each lane
// issues all of its row loads before any arithmetic so that every warp keeps
// kRowsPerLane 16-byte loads in flight.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kRowsPerLane = 4;

__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
    const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// K: key width (row length); LPR = K / 4 lanes per row; RPW = 32 / LPR rows
// per warp per pass.  A CTA covers rows_per_cta = 4 warps * RPW * kRowsPerLane
// consecutive rows of one head.
template <int LPR, typename Tin>
__device__ __forceinline__ float4 gather4_normalized(const Tin *row, const int *ih, int cl,
                                                     int Kin, float eps, bool &bad) {
    const int4 i4 = __ldg(reinterpret_cast<const int4 *>(ih) + cl);
    const int ci[4] = {i4.x, i4.y, i4.z, i4.w};
    float g[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int c = ci[e];
        if ((unsigned)c < (unsigned)Kin) {
            g[e] = to_f32(row[c]);
        } else {
            g[e] = 0.f;
            bad = true;
        }
    }
    float ss = g[0] * g[0] + g[1] * g[1] + g[2] * g[2] + g[3] * g[3];
    ss = group_sum<LPR>(ss);
    const float inv = 1.f / fmaxf(sqrtf(ss), eps);
    return make_float4(g[0] * inv, g[1] * inv, g[2] * inv, g[3] * inv);
}

template <int K, typename Tin, bool GATHER>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_step_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                       const Tin *__restrict__ v, const float *__restrict__ alpha,
                       const float *__restrict__ beta, float *__restrict__ S,
                       Tin *__restrict__ o, int V, int blocks_per_head, const int *idx, int Kin,
                       int H, float eps, int *status) {
    constexpr int LPR = K / 4;
    constexpr int RPW = 32 / LPR;
    constexpr int kRowsPerWarp = RPW * kRowsPerLane;
    constexpr int kRowsPerCta = (kDecodeThreads / 32) * kRowsPerWarp;

    const int bh = blockIdx.x / blocks_per_head;
    const int blk = blockIdx.x % blocks_per_head;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane / LPR;  // row within the warp's pass
    const int cl = lane % LPR;   // float4 column index

    // plain steps are launched with programmatic dependent launch: wait for
    // the previous step's state writes before the first global read
    if constexpr (!GATHER) pdl_wait();
    float4 kf, qf;
    if constexpr (!GATHER) {
        kf = load4(k + (size_t)bh * K + 4 * cl);
        qf = load4(q + (size_t)bh * K + 4 * cl);
    }
    const float a = alpha[bh];
    const float be = beta[bh];

    const int row0 = blk * kRowsPerCta + warp * kRowsPerWarp + sub;
    float *Sh = S + (size_t)bh * V * K;

    float4 s[kRowsPerLane];
    float vi[kRowsPerLane];
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
        const int row = row0 + r * RPW;
        if (row < V) {
            s[r] = load4(Sh + (size_t)row * K + 4 * cl);
            vi[r] = to_f32(v[(size_t)bh * V + row]);
        } else {
            s[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            vi[r] = 0.f;
        }
    }
    if constexpr (!GATHER) pdl_trigger();  // the next step may be scheduled early
    if constexpr (GATHER) {
        // The state loads above are already in flight: the index -> channel
        // load chain and the norm reductions overlap them.
        bool bad = false;
        const int *ih = idx + (bh % H) * K;
        kf = gather4_normalized<LPR>(k + (size_t)bh * Kin, ih, cl, Kin, eps, bad);
        qf = gather4_normalized<LPR>(q + (size_t)bh * Kin, ih, cl, Kin, eps, bad);
        if (bad && status && blk == 0) atomicOr(status, kStatusBounds);
    }
    const float kq = group_sum<LPR>(kf.x * qf.x + kf.y * qf.y + kf.z * qf.z + kf.w * qf.w);
#pragma unroll
    for (int r = 0; r < kRowsPerLane; ++r) {
        const int row = row0 + r * RPW;
        float4 x = s[r];
        x.x *= a; x.y *= a; x.z *= a; x.w *= a;
        float p = x.x * kf.x + x.y * kf.y + x.z * kf.z + x.w * kf.w;
        float rq = x.x * qf.x + x.y * qf.y + x.z * qf.z + x.w * qf.w;
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) {
            p += __shfl_xor_sync(0xffffffffu, p, off);
            rq += __shfl_xor_sync(0xffffffffu, rq, off);
        }
        const float u = be * (vi[r] - p);
        x.x = fmaf(u, kf.x, x.x);
        x.y = fmaf(u, kf.y, x.y);
        x.z = fmaf(u, kf.z, x.z);
        x.w = fmaf(u, kf.w, x.w);
        if (row < V) {
            *reinterpret_cast<float4 *>(Sh + (size_t)row * K + 4 * cl) = x;
            if (cl == 0) o[(size_t)bh * V + row] = from_f32<Tin>(fmaf(u, kq, rq));
        }
    }
}

template <int K, typename Tin, bool GATHER = false>
cudaError_t launch_decode_t(const void *q, const void *k, const void *v, const float *alpha,
                            const float *beta, float *S, void *o, int BH, int V,
                            cudaStream_t stream, const int *idx = nullptr, int Kin = K, int H = 1,
                            float eps = 0.f) {
    constexpr int kRowsPerCta = (kDecodeThreads / 32) * (32 / (K / 4)) * kRowsPerLane;
    const int blocks_per_head = (V + kRowsPerCta - 1) / kRowsPerCta;
    const long long grid = (long long)BH * blocks_per_head;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if constexpr (!GATHER) {
        // consecutive plain steps overlap their launch with the previous step's
        // tail (measured: 23.3 -> 21.3 us per step at B = 64, d_k = 128, L2-cold).
        // The gathering step (and the gated step) measured slower with it, and
        // slower even with the wait / trigger instructions present but a plain
        // launch, so they have neither.
        return launch_pdl(decode_step_kernel<K, Tin, GATHER>, (unsigned)grid, kDecodeThreads, 0,
                          stream, static_cast<const Tin *>(q), static_cast<const Tin *>(k),
                          static_cast<const Tin *>(v), alpha, beta, S, static_cast<Tin *>(o), V,
                          blocks_per_head, idx, Kin, H, eps, nullptr);
    }
    decode_step_kernel<K, Tin, GATHER><<<(unsigned)grid, kDecodeThreads, 0, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        alpha, beta, S, static_cast<Tin *>(o), V, blocks_per_head, idx, Kin, H, eps,
        device_status_ptr());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *alpha,
                          const float *beta, float *S, void *o, int B, int H, int K, int V,
                          gdn_dtype dt, cudaStream_t stream) {
    const int BH = B * H;
#define GDN_DECODE_CASE(KK)                                                                \
    case KK:                                                                               \
        return dt == GDN_BF16                                                              \
                   ? launch_decode_t<KK, __nv_bfloat16>(q, k, v, alpha, beta, S, o, BH, V, \
                                                        stream)                            \
                   : launch_decode_t<KK, float>(q, k, v, alpha, beta, S, o, BH, V, stream);
    switch (K) {
        GDN_DECODE_CASE(32)
        GDN_DECODE_CASE(64)
        GDN_DECODE_CASE(128)
        default:
            return cudaErrorInvalidValue;
    }
#undef GDN_DECODE_CASE
}

cudaError_t launch_decode_gathered(const void *q, const void *k, const int *idx, int Kin,
                                   const void *v, const float *alpha, const float *beta,
                                   float *S, void *o, int B, int H, int K, int V, gdn_dtype dt,
                                   float eps, cudaStream_t stream) {
    const int BH = B * H;
#define GDN_DECODE_G(KK)                                                                       \
    case KK:                                                                                   \
        return dt == GDN_BF16                                                                  \
                   ? launch_decode_t<KK, __nv_bfloat16, true>(q, k, v, alpha, beta, S, o, BH, V, \
                                                              stream, idx, Kin, H, eps)        \
                   : launch_decode_t<KK, float, true>(q, k, v, alpha, beta, S, o, BH, V,       \
                                                      stream, idx, Kin, H, eps);
    switch (K) {
        GDN_DECODE_G(32)
        GDN_DECODE_G(64)
        GDN_DECODE_G(128)
        default:
            return cudaErrorInvalidValue;
    }
#undef GDN_DECODE_G
}

}  // namespace gdn
