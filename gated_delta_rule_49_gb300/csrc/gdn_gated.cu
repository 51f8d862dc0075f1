// Channel-gated delta rules ("Linear Attention Architectures" notes,
// Secs. 2.4-2.6), token by token on the CUDA cores:
//
//   SCALAR (GDN):  S <- a S;              u = beta (v - S k)
//   KDA:           S <- S diag(alpha);    u = beta (v - S k)
//   GDN2:          S <- S diag(alpha);    u = w (.) v - S (b (.) k)
//   then           S <- S + u k^T,        o = S q
//
// Each value row of S is an independent system (the gates act on the key
// channels or per value row), so the state is split by rows across CTAs and
// lanes and nothing is exchanged between rows.
//
// Prefill: a CTA owns R = 32 rows of one (b, h) sequence; a row is spread
// over K / CPL lanes holding CPL channels each in registers (CPL = 16 at
// d_k = 128, 8 otherwise), and every lane holds four rows, so that the
// per-token operands it reads from shared memory (k, q, the channel decay,
// the erase direction) serve all of them.  The per-token operands and the
// CTA's slice of v / w are staged 8 tokens at a time into a two-stage
// shared-memory ring by cp.async (block n+1 in flight while block n is
// processed); bf16 k / q are converted to float32 once per CTA.  Per token
// and row: decay, the erase read p = s~ . e and r = s~ . q (reduced together
// over the row's lanes), the rank-one write, and o = r + u (k . q); the state
// arithmetic runs on packed float2 FMA.  Outputs are collected per block in
// shared memory and written with 16-byte stores.  Bound: the latency of the
// token-serial chain per warp (few warps per SM at these row counts).
// This kernel is also the prefill for float32 inputs and for the (32, 32)
// variant (scalar gate).
//
// Decode: the layout of the plain decode step (K/4 lanes per row, four rows
// per lane, all state loads issued first); HBM-bound on the state.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

enum GateMode : int { kScalar = GDN_GATE_SCALAR, kKda = GDN_GATE_KDA, kGdn2 = GDN_GATE_GDN2 };

constexpr int kTB = 8;   // tokens per staged block

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all_but_one() {
    asm volatile("cp.async.wait_group 1;\n" ::: "memory");
}

// The CPL channels a lane holds: CPL/4 float4 pieces at channel offsets
// 4 cl + 4 LPR j, so the LPR lanes of a row read 16 LPR contiguous floats per
// piece (conflict-free shared-memory reads).  As float2 pairs: x[CPL / 2].
template <int LPR, int CPL>
__device__ __forceinline__ void ldc(const float *row, int cl, float2 (&x)[CPL / 2]) {
#pragma unroll
    for (int j = 0; j < CPL / 4; ++j) {
        const float4 v = *reinterpret_cast<const float4 *>(row + 4 * cl + 4 * LPR * j);
        x[2 * j] = make_float2(v.x, v.y);
        x[2 * j + 1] = make_float2(v.z, v.w);
    }
}
template <int LPR, int CPL>
__device__ __forceinline__ void stc(float *row, int cl, const float2 (&x)[CPL / 2]) {
#pragma unroll
    for (int j = 0; j < CPL / 4; ++j)
        *reinterpret_cast<float4 *>(row + 4 * cl + 4 * LPR * j) =
            make_float4(x[2 * j].x, x[2 * j].y, x[2 * j + 1].x, x[2 * j + 1].y);
}

template <int L>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Shared-memory layout (byte offsets, all multiples of 16): two stages of raw
// per-token operands, the current block's k/q as float32, and the outputs.
template <int K, int R, typename Tin, int GATE>
struct GatedStage {
    static constexpr bool kBf = sizeof(Tin) == 2;
    static constexpr int KA = GATE == kScalar ? 4 : K;  // floats of alpha per token
    static constexpr int KQ = 0;                                           // [kTB][2][K] Tin
    static constexpr int AL = KQ + kTB * 2 * K * (int)sizeof(Tin);          // [kTB][KA] f32
    static constexpr int BG = AL + kTB * KA * 4;                            // [kTB][K] f32
    static constexpr int BE = BG + (GATE == kGdn2 ? kTB * K * 4 : 0);       // [kTB] f32
    static constexpr int VV = BE + (kTB * 4 + 15) / 16 * 16;                // [kTB][R] Tin
    static constexpr int WW = VV + kTB * R * (int)sizeof(Tin);              // [kTB][R] f32
    static constexpr int BYTES = WW + (GATE == kGdn2 ? kTB * R * 4 : 0);
    static constexpr int KQF = 2 * BYTES;                                   // [kTB][2][K] f32
    static constexpr int OB = KQF + (kBf ? kTB * 2 * K * 4 : 0);            // [kTB][R] Tin
    static constexpr int SMEM = OB + kTB * R * (int)sizeof(Tin);
    static_assert(AL % 16 == 0 && BG % 16 == 0 && VV % 16 == 0 && WW % 16 == 0 &&
                      BYTES % 16 == 0 && KQF % 16 == 0 && OB % 16 == 0,
                  "16-byte aligned regions");
};

// Issue the cp.async copies of tokens [t0, t0 + n) of sequence (b, h) for
// rows [r0, r0 + R) into one stage.
template <int K, int R, typename Tin, int GATE>
__device__ __forceinline__ void stage_block(unsigned char *st, const Tin *q, const Tin *k,
                                            const Tin *v, const float *alpha,
                                            const float *beta, const float *bg,
                                            const float *wg, size_t th0, int H, int V, int r0,
                                            int n) {
    using L = GatedStage<K, R, Tin, GATE>;
    constexpr int EPC = 16 / (int)sizeof(Tin);  // elements per 16-byte chunk
    constexpr int nK = K / EPC;                 // chunks of one k (or q) row
    constexpr int nA = GATE == kScalar ? 0 : K / 4;
    constexpr int nB = GATE == kGdn2 ? K / 4 : 0;
    constexpr int nV = R / EPC;
    constexpr int nW = GATE == kGdn2 ? R / 4 : 0;
    constexpr int nTok = 2 * nK + nA + nB + nV + nW;
    for (int j = threadIdx.x; j < n * nTok; j += blockDim.x) {
        const int tau = j / nTok;
        int c = j - tau * nTok;
        const size_t th = th0 + (size_t)tau * H;  // token-head index of token t0 + tau
        if (c < 2 * nK) {
            const int which = c / nK;  // 0: k, 1: q
            c -= which * nK;
            const Tin *src = (which ? q : k) + th * K + c * EPC;
            cp_async16(st + L::KQ + ((tau * 2 + which) * K + c * EPC) * (int)sizeof(Tin), src);
            continue;
        }
        c -= 2 * nK;
        if (c < nA) {
            cp_async16(st + L::AL + (tau * K + c * 4) * 4, alpha + th * K + c * 4);
            continue;
        }
        c -= nA;
        if (c < nB) {
            cp_async16(st + L::BG + (tau * K + c * 4) * 4, bg + th * K + c * 4);
            continue;
        }
        c -= nB;
        if (c < nV) {
            cp_async16(st + L::VV + (tau * R + c * EPC) * (int)sizeof(Tin),
                       v + th * V + r0 + c * EPC);
            continue;
        }
        c -= nV;
        cp_async16(st + L::WW + (tau * R + c * 4) * 4, wg + th * V + r0 + c * 4);
    }
    for (int tau = threadIdx.x; tau < n; tau += blockDim.x) {
        const size_t th = th0 + (size_t)tau * H;
        if (GATE == kScalar) cp_async4(st + L::AL + tau * L::KA * 4, alpha + th);
        if (GATE != kGdn2) cp_async4(st + L::BE + tau * 4, beta + th);
    }
}

// grid: B*H*(V/R) CTAs; CTA x -> sequence x / (V/R), slab x % (V/R).  A row's
// K channels sit on K / CPL lanes (CPL each); a warp holds RPI * RPL rows:
// lane group g holds rows w RPI RPL + rr RPI + g, rr < RPL, so the per-token
// operands a lane loads (k, q, the channel decay, the erase direction) serve
// RPL rows.  Per token and row the two dot products p = s~ . e and
// r = s~ . q of the decayed state are reduced together, then
// u = (write) - p, s = s~ + u k and o = r + u (k . q), k . q being shared by
// all rows.
template <int K, int R, int CPL, int RPL, typename Tin, int GATE>
__global__ void __launch_bounds__(128)
    prefill_gated_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                         const Tin *__restrict__ v, const float *__restrict__ alpha,
                         const float *__restrict__ beta, const float *__restrict__ bg,
                         const float *__restrict__ wg, const float *__restrict__ S0,
                         Tin *__restrict__ o, float *__restrict__ ST, int T, int Ts, int H,
                         int V) {
    using L = GatedStage<K, R, Tin, GATE>;
    constexpr int LPR = K / CPL;  // lanes per row
    constexpr int RPI = 32 / LPR;
    constexpr int NP = CPL / 2;   // float2 pairs per lane
    constexpr int EPC = 16 / (int)sizeof(Tin);
    extern __shared__ __align__(16) unsigned char smem[];

    const int slabs = V / R;
    const int seq = blockIdx.x / slabs;
    const int r0 = (blockIdx.x % slabs) * R;
    const int b = seq / H, h = seq % H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / LPR, cl = lane % LPR;
    int row[RPL];
#pragma unroll
    for (int rr = 0; rr < RPL; ++rr) row[rr] = (warp * RPL + rr) * RPI + g;  // within the slab

    float2 s[RPL][NP];
#pragma unroll
    for (int rr = 0; rr < RPL; ++rr) {
        if (S0) {
            ldc<LPR, CPL>(S0 + ((size_t)seq * V + r0 + row[rr]) * K, cl, s[rr]);
        } else {
#pragma unroll
            for (int e = 0; e < NP; ++e) s[rr][e] = make_float2(0.f, 0.f);
        }
    }

    const int nblk = (T + kTB - 1) / kTB;
    auto th_of = [&](int t) { return ((size_t)b * Ts + t) * H + h; };
    if (nblk > 0)
        stage_block<K, R, Tin, GATE>(smem, q, k, v, alpha, beta, bg, wg, th_of(0), H, V, r0,
                                     min(kTB, T));
    cp_async_commit();
    Tin *ob = reinterpret_cast<Tin *>(smem + L::OB);
    for (int n = 0; n < nblk; ++n) {
        const int t0 = n * kTB;
        if (n + 1 < nblk)
            stage_block<K, R, Tin, GATE>(smem + ((n + 1) & 1) * L::BYTES, q, k, v, alpha, beta,
                                         bg, wg, th_of(t0 + kTB), H, V, r0,
                                         min(kTB, T - t0 - kTB));
        cp_async_commit();
        cp_async_wait_all_but_one();
        __syncthreads();
        const unsigned char *st = smem + (n & 1) * L::BYTES;
        const int nt = min(kTB, T - t0);
        const float *kqf;
        if constexpr (L::kBf) {  // this block's k and q as float32, once per CTA
            const __nv_bfloat162 *src = reinterpret_cast<const __nv_bfloat162 *>(st + L::KQ);
            float2 *dst = reinterpret_cast<float2 *>(smem + L::KQF);
            for (int e = threadIdx.x; e < nt * K; e += blockDim.x)
                dst[e] = __bfloat1622float2(src[e]);
            __syncthreads();
            kqf = reinterpret_cast<const float *>(smem + L::KQF);
        } else {
            kqf = reinterpret_cast<const float *>(st + L::KQ);
        }
        const float *al = reinterpret_cast<const float *>(st + L::AL);
        const float *bgs = reinterpret_cast<const float *>(st + L::BG);
        const float *bes = reinterpret_cast<const float *>(st + L::BE);
        const Tin *vv = reinterpret_cast<const Tin *>(st + L::VV);
        const float *ww = reinterpret_cast<const float *>(st + L::WW);
        for (int tau = 0; tau < nt; ++tau) {
            float2 kk[NP], qq[NP], ee[NP], aa[NP];
            ldc<LPR, CPL>(kqf + (tau * 2) * K, cl, kk);
            ldc<LPR, CPL>(kqf + (tau * 2 + 1) * K, cl, qq);
            if constexpr (GATE == kScalar) {
                const float a = al[tau * L::KA];
#pragma unroll
                for (int e = 0; e < NP; ++e) aa[e] = make_float2(a, a);
            } else {
                ldc<LPR, CPL>(al + tau * K, cl, aa);
            }
            if constexpr (GATE == kGdn2) {
                ldc<LPR, CPL>(bgs + tau * K, cl, ee);
#pragma unroll
                for (int e = 0; e < NP; ++e) ee[e] = __fmul2_rn(ee[e], kk[e]);
            } else {
#pragma unroll
                for (int e = 0; e < NP; ++e) ee[e] = kk[e];
            }
            float2 kq2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < NP; ++e) kq2 = __ffma2_rn(kk[e], qq[e], kq2);
            float kq = kq2.x + kq2.y;
            float p[RPL], r[RPL];
#pragma unroll
            for (int rr = 0; rr < RPL; ++rr) {
                float2 p2 = make_float2(0.f, 0.f), r2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    s[rr][e] = __fmul2_rn(s[rr][e], aa[e]);
                    p2 = __ffma2_rn(s[rr][e], ee[e], p2);
                    r2 = __ffma2_rn(s[rr][e], qq[e], r2);
                }
                p[rr] = p2.x + p2.y;
                r[rr] = r2.x + r2.y;
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) {
                kq += __shfl_xor_sync(0xffffffffu, kq, off);
#pragma unroll
                for (int rr = 0; rr < RPL; ++rr) {
                    p[rr] += __shfl_xor_sync(0xffffffffu, p[rr], off);
                    r[rr] += __shfl_xor_sync(0xffffffffu, r[rr], off);
                }
            }
#pragma unroll
            for (int rr = 0; rr < RPL; ++rr) {
                const float vi = to_f32(vv[tau * R + row[rr]]);
                float u;
                if constexpr (GATE == kGdn2)
                    u = ww[tau * R + row[rr]] * vi - p[rr];
                else
                    u = bes[tau] * (vi - p[rr]);
                const float2 u2 = make_float2(u, u);
#pragma unroll
                for (int e = 0; e < NP; ++e) s[rr][e] = __ffma2_rn(u2, kk[e], s[rr][e]);
                if (cl == 0) ob[tau * R + row[rr]] = from_f32<Tin>(fmaf(u, kq, r[rr]));
            }
        }
        __syncthreads();  // outputs complete; stage n & 1 (and the float32 k/q) free
        if (o) {
            constexpr int nO = R / EPC;
            for (int j = threadIdx.x; j < nt * nO; j += blockDim.x) {
                const int tau = j / nO, c = j % nO;
                *reinterpret_cast<uint4 *>(o + th_of(t0 + tau) * V + r0 + c * EPC) =
                    *reinterpret_cast<const uint4 *>(ob + tau * R + c * EPC);
            }
        }
    }
    if (ST)
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
            stc<LPR, CPL>(ST + ((size_t)seq * V + r0 + row[rr]) * K, cl, s[rr]);
}

template <int K, int R, int CPL, int RPL, typename Tin, int GATE>
cudaError_t launch_pg(const void *q, const void *k, const void *v, const float *alpha,
                      const float *beta, const float *bg, const float *wg, const float *S0,
                      void *o, float *ST, int B, int T, int Ts, int H, int V,
                      cudaStream_t stream) {
    using L = GatedStage<K, R, Tin, GATE>;
    constexpr int RPI = 32 / (K / CPL);
    constexpr int threads = R / (RPI * RPL) * 32;
    static_assert(threads >= 32 && threads <= 128 && R % (RPI * RPL) == 0, "tiling");
    static_assert(CPL % 4 == 0 && K % CPL == 0 && 32 % (K / CPL) == 0, "channels per lane");
    auto kern = prefill_gated_kernel<K, R, CPL, RPL, Tin, GATE>;
    static uintptr_t attr_set[64] = {};  // context the attributes were set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (L::SMEM > 48 * 1024 && attr_set[dev] != context_key()) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = context_key();
    }
    const long long grid = (long long)B * H * (V / R);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, threads, L::SMEM, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        alpha, beta, bg, wg, S0, static_cast<Tin *>(o), ST, T, Ts, H, V);
    return cudaGetLastError();
}

// (K, V) -> rows per CTA R, channels per lane CPL, rows per lane RPL:
// (128, 128): 16 lanes x 8 channels per row, 4 rows per lane, 4 warps of 8
// rows; (64, 128): 8 lanes x 8 channels, 4 rows per lane, 2 warps of 16 rows;
// (32, 32): 4 lanes x 8 channels, 4 rows per lane, 1 warp of 32 rows.
template <typename Tin, int GATE>
cudaError_t pg_dispatch(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *bg, const float *wg, const float *S0,
                        void *o, float *ST, int B, int T, int Ts, int H, int K, int V,
                        cudaStream_t stream) {
    if (K == 128 && V == 128)
        return launch_pg<128, 32, 16, 4, Tin, GATE>(q, k, v, alpha, beta, bg, wg, S0, o, ST, B, T,
                                                    Ts, H, V, stream);
    if (K == 64 && V == 128)
        return launch_pg<64, 32, 8, 4, Tin, GATE>(q, k, v, alpha, beta, bg, wg, S0, o, ST, B, T,
                                                  Ts, H, V, stream);
    if (K == 32 && V == 32)
        return launch_pg<32, 32, 8, 4, Tin, GATE>(q, k, v, alpha, beta, bg, wg, S0, o, ST, B, T,
                                                  Ts, H, V, stream);
    return cudaErrorInvalidValue;
}

// ---- decode -----------------------------------------------------------------

constexpr int kDecThreads = 128;
constexpr int kDecRowsPerLane = 4;

__device__ __forceinline__ float4 ld4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

template <int K, typename Tin, int GATE>
__global__ void __launch_bounds__(kDecThreads)
    decode_gated_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                        const Tin *__restrict__ v, const float *__restrict__ alpha,
                        const float *__restrict__ beta, const float *__restrict__ bg,
                        const float *__restrict__ wg, float *__restrict__ S,
                        Tin *__restrict__ o, int V, int blocks_per_head) {
    constexpr int LPR = K / 4;
    constexpr int RPW = 32 / LPR;
    constexpr int kRowsPerWarp = RPW * kDecRowsPerLane;
    constexpr int kRowsPerCta = (kDecThreads / 32) * kRowsPerWarp;
    const int bh = blockIdx.x / blocks_per_head;
    const int blk = blockIdx.x % blocks_per_head;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane / LPR, cl = lane % LPR;
    const int row0 = blk * kRowsPerCta + warp * kRowsPerWarp + sub;
    float *Sh = S + (size_t)bh * V * K;

    float4 s[kDecRowsPerLane];
    float vi[kDecRowsPerLane], wi[kDecRowsPerLane];
#pragma unroll
    for (int r = 0; r < kDecRowsPerLane; ++r) {
        const int row = row0 + r * RPW;
        const bool ok = row < V;
        s[r] = ok ? ld4(Sh + (size_t)row * K + 4 * cl) : make_float4(0.f, 0.f, 0.f, 0.f);
        vi[r] = ok ? to_f32(v[(size_t)bh * V + row]) : 0.f;
        wi[r] = (GATE == kGdn2 && ok) ? wg[(size_t)bh * V + row] : 0.f;
    }
    const float4 kf = ld4(k + (size_t)bh * K + 4 * cl);
    const float4 qf = ld4(q + (size_t)bh * K + 4 * cl);
    float4 af;
    if constexpr (GATE == kScalar) {
        const float a = alpha[bh];
        af = make_float4(a, a, a, a);
    } else {
        af = ld4(alpha + (size_t)bh * K + 4 * cl);
    }
    float4 ef = kf;
    if constexpr (GATE == kGdn2) {
        const float4 bb = ld4(bg + (size_t)bh * K + 4 * cl);
        ef = make_float4(bb.x * kf.x, bb.y * kf.y, bb.z * kf.z, bb.w * kf.w);
    }
    const float be = GATE == kGdn2 ? 0.f : beta[bh];
    const float kq = group_sum<LPR>(dot4(kf, qf));
#pragma unroll
    for (int r = 0; r < kDecRowsPerLane; ++r) {
        const int row = row0 + r * RPW;
        float4 x = s[r];
        x.x *= af.x; x.y *= af.y; x.z *= af.z; x.w *= af.w;
        float p = dot4(x, ef);
        float rq = dot4(x, qf);
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) {
            p += __shfl_xor_sync(0xffffffffu, p, off);
            rq += __shfl_xor_sync(0xffffffffu, rq, off);
        }
        const float u = GATE == kGdn2 ? wi[r] * vi[r] - p : be * (vi[r] - p);
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

template <int K, typename Tin, int GATE>
cudaError_t launch_dg(const void *q, const void *k, const void *v, const float *alpha,
                      const float *beta, const float *bg, const float *wg, float *S, void *o,
                      int BH, int V, cudaStream_t stream) {
    constexpr int kRowsPerCta = (kDecThreads / 32) * (32 / (K / 4)) * kDecRowsPerLane;
    const int bph = (V + kRowsPerCta - 1) / kRowsPerCta;
    const long long grid = (long long)BH * bph;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    decode_gated_kernel<K, Tin, GATE><<<(unsigned)grid, kDecThreads, 0, stream>>>(
        static_cast<const Tin *>(q), static_cast<const Tin *>(k), static_cast<const Tin *>(v),
        alpha, beta, bg, wg, S, static_cast<Tin *>(o), V, bph);
    return cudaGetLastError();
}

template <typename Tin, int GATE>
cudaError_t dg_dispatch(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *bg, const float *wg, float *S, void *o,
                        int BH, int K, int V, cudaStream_t stream) {
    if (K == 128) return launch_dg<128, Tin, GATE>(q, k, v, alpha, beta, bg, wg, S, o, BH, V, stream);
    if (K == 64) return launch_dg<64, Tin, GATE>(q, k, v, alpha, beta, bg, wg, S, o, BH, V, stream);
    if (K == 32) return launch_dg<32, Tin, GATE>(q, k, v, alpha, beta, bg, wg, S, o, BH, V, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_gated(const void *q, const void *k, const void *v,
                                 const float *alpha, const float *beta, const float *bg,
                                 const float *wg, const float *S0, void *o, float *ST, int B,
                                 int T, int Ts, int H, int K, int V, gdn_gate gate, gdn_dtype dt,
                                 cudaStream_t stream) {
#define GDN_PG(TIN, G) \
    pg_dispatch<TIN, G>(q, k, v, alpha, beta, bg, wg, S0, o, ST, B, T, Ts, H, K, V, stream)
    const bool bf = dt == GDN_BF16;
    switch (gate) {
        case GDN_GATE_SCALAR: return bf ? GDN_PG(__nv_bfloat16, kScalar) : GDN_PG(float, kScalar);
        case GDN_GATE_KDA: return bf ? GDN_PG(__nv_bfloat16, kKda) : GDN_PG(float, kKda);
        case GDN_GATE_GDN2: return bf ? GDN_PG(__nv_bfloat16, kGdn2) : GDN_PG(float, kGdn2);
    }
#undef GDN_PG
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_gated(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *bg, const float *wg, float *S,
                                void *o, int B, int H, int K, int V, gdn_gate gate, gdn_dtype dt,
                                cudaStream_t stream) {
    const int BH = B * H;
#define GDN_DG(TIN, G) dg_dispatch<TIN, G>(q, k, v, alpha, beta, bg, wg, S, o, BH, K, V, stream)
    const bool bf = dt == GDN_BF16;
    switch (gate) {
        case GDN_GATE_SCALAR: return bf ? GDN_DG(__nv_bfloat16, kScalar) : GDN_DG(float, kScalar);
        case GDN_GATE_KDA: return bf ? GDN_DG(__nv_bfloat16, kKda) : GDN_DG(float, kKda);
        case GDN_GATE_GDN2: return bf ? GDN_DG(__nv_bfloat16, kGdn2) : GDN_DG(float, kGdn2);
    }
#undef GDN_DG
    return cudaErrorInvalidValue;
}

}  // namespace gdn
