// Chunkwise tensor-core prefill of the channel-gated delta rules ("Linear
// Attention Architectures" notes, Secs. 2.4-2.6), d_k = d_v = 128, bf16:
//
//   KDA:   S <- S diag(alpha_t);  u_t = beta_t (v_t - S k_t)
//   GDN2:  S <- S diag(alpha_t);  u_t = w_t (.) v_t - S (b_t (.) k_t)
//   then   S <- S + u_t k_t^T,    o_t = S q_t
//
// With G the in-chunk cumulative log-decay per key channel (C = 64 tokens,
// G_t in R^K) and the erase rows E = diag(beta) K (KDA) or b (.) K (GDN2), the
// chunk unrolls to ("On State Reduction" notes, Sec. 2.3, with per-channel
// decay):
//
//   A_ts = sum_j e_tj k_sj e^(G_tj - G_sj)  (s < t),   P_ts = sum_j q_tj k_sj e^(G_tj - G_sj)  (s <= t)
//   T    = (I + A)^{-1},  T_b = T diag(beta) (KDA) or T (GDN2, beta folded into E)
//   W    = T_b (K~ (.) e^G) with K~ = K (KDA) or b (.) K (GDN2),   U~ = T_b Z,
//          Z = V (KDA) or w (.) V (GDN2)
//   U^T  = U~^T - S W^T,   O^T = S (Q (.) e^G)^T + U^T P^T,
//   S   <- S diag(e^(G_C)) + U^T (K (.) e^(G_C - G))
//
// For the per-channel exponent inside A and P each 16-token row block I is
// referred to its reference token m = 16 I + 7:
// e^(G_t - G_s) = e^(G_t - G_m) e^(G_m - G_s), so row block I of A and P is one
// product of [E_I (.) e^(G_I - G_m); Q_I (.) e^(G_I - G_m)] with
// K_{<=I} (.) e^(G_m - G_{<=I}); every factor stays below e^(8 max |log alpha|).
//
// Two kernels, like the scalar-gated two-pass prefill:
//   prefill_gated_prep_kernel: every chunk of every sequence at once
//     (persistent CTAs of 128 threads, two per SM): the gate prefix, the
//     block products of A and P on warp-level MMAs (one row block per warp),
//     the inverse (the scalar prefill's split-bf16 blocked inverse), W^T on
//     tcgen05, and the state pass's operands -- T_b^T, P, -W^T, Q (.) e^G,
//     K (.) e^(G_C - G) and e^(G_C) -- written to the workspace as
//     their swizzled shared-memory images.
//   gated_z_kernel (GDN2): Z = w (.) V into the same workspace, element by
//     element, on a second stream beside the key-side pass: HBM-bound work
//     that cost the instruction-bound key-side pass ~128 us interleaved with
//     its own, and runs in that pass's shadow here (0.578 ms per call on the
//     gated workload; 0.606 ms with the two kernels one after the other, and
//     0.647 ms with Z inside the key-side pass).
//   prefill_gated_state_kernel: one CTA per sequence; the scalar state pass's
//     chain without its key group: U~ by an issuer thread, U, dS and O by the
//     state thread, the float32 state in registers with a bf16 copy in TMEM.
#include "gdn_internal.cuh"
#include "gdn_sm100.cuh"
#include "gdn_chunk.cuh"

#include <algorithm>
#include <mutex>

namespace gdn {
namespace {

constexpr int kKda = GDN_GATE_KDA, kGdn2 = GDN_GATE_GDN2;

// One chunk's operands in the workspace (bytes), each the swizzled image of
// its shared-memory tile.
constexpr uint32_t kGwTB = 0;        // T_b^T            [64][64] bf16
constexpr uint32_t kGwNW = 8192;     // -W^T             [128][64] bf16
constexpr uint32_t kGwP = 24576;     // P                [64][64] bf16
constexpr uint32_t kGwQ = 32768;     // Q (.) e^G        two [64][64] boxes
constexpr uint32_t kGwK = 49152;     // K (.) e^(G_C-G)  two [64][64] boxes
constexpr uint32_t kGwF = 65536;     // e^(G_C)          [128] float
constexpr uint32_t kGwZ = 66048;     // w (.) V (GDN2)   two [64][64] boxes
__host__ __device__ constexpr uint32_t gw_chunk_bytes(int gate) {
    return gate == kGdn2 ? kGwZ + 16384 : kGwZ;
}

// 2^x with the hardware approximation (relative error about 2^-22; results
// below 2^-126 flush to zero).
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
// Two bf16 channels (j, j + 1) of row r of a [64][128] tile stored as two
// 128-byte-swizzled [64][64] boxes.
__device__ __forceinline__ uint32_t ld_pair(const uint8_t *tile, int r, int j) {
    return *reinterpret_cast<const uint32_t *>(tile + (j >> 6) * 8192 + swz128(r, (j & 63) >> 3) +
                                               (j & 7) * 2);
}
// Byte offset of the 16-byte piece (row r, channels 8 c16 .. + 7) in that layout.
__device__ __forceinline__ uint32_t piece_off(int r, int c16) {
    return (c16 >> 3) * 8192 + swz128(r, c16 & 7);
}

// ---------------------------------------------------------------- key-side pass
constexpr int kGpThreads = 128;
constexpr int kGpCtasPerSm = 2;
constexpr int kGLD = 136;  // row stride of the float G table (conflict-free pair reads)
struct GpLayout {
    static constexpr uint32_t KB = 0;              // k boxes
    static constexpr uint32_t QB = 16384;          // q boxes
    static constexpr uint32_t KT = 32768;          // K~ (.) e^G boxes (W^T's operand)
    static constexpr uint32_t TB = 49152;          // T_b^T
    static constexpr uint32_t AF = 57344;          // float [64][kLD]; GDN2: E boxes before A
    static constexpr uint32_t G = AF + 64 * kLD * 4;  // float [64][kGLD], log2 prefix
    static constexpr uint32_t BET = G + 64 * kGLD * 4;  // beta[64], ones[64]
    static constexpr uint32_t END = BET + 2 * 64 * 4;
    static constexpr size_t SMEM = END;
};
static_assert(GpLayout::AF % 1024 == 0 && 64 * kLD * 4 >= 16384, "E boxes fit the A scratch");
static_assert(kGpCtasPerSm * (GpLayout::SMEM + 2048) <= 233472, "key-side residency");

template <int GATE>
__global__ void __launch_bounds__(kGpThreads, kGpCtasPerSm)
    prefill_gated_prep_kernel(const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_k,
                              const float *__restrict__ alpha, const float *__restrict__ beta,
                              const float *__restrict__ bgate, uint8_t *__restrict__ ws,
                              int T, int H, long long nchunk_all, int *status) {
    using L = GpLayout;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0 && status) atomicOr(status, kStatusBounds);
        return;
    }
    uint8_t *sm = smem_raw;
    __shared__ uint64_t kq_full, bar_w, drain;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    volatile int *abort_v = &abort_flag;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int nch = (T + 63) / 64;

    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 64);
        tmem_relinquish();
    }
    if (tid == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        mbar_init(&kq_full, 1);
        mbar_init(&bar_w, 1);
        mbar_init(&drain, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;
    const uint32_t base = smem_u32(sm);
    float *AF = reinterpret_cast<float *>(sm + L::AF);
    float *Gt = reinterpret_cast<float *>(sm + L::G);
    float *bet = reinterpret_cast<float *>(sm + L::BET);
    float *ones = bet + 64;
    if (tid < 64) ones[tid] = 1.f;

    auto load_kq = [&](long long j) {
        if (!bounds_ok(j >= 0 && j < nchunk_all, status)) return;
        const long long seq = j / nch;
        const int n = (int)(j - seq * nch);
        const int b = (int)(seq / H), h = (int)(seq % H);
        mbar_arrive_expect_tx(&kq_full, 32768);
        tma_load_4d(sm + L::KB, &tm_k, &kq_full, 0, h, n * 64, b);
        tma_load_4d(sm + L::KB + 8192, &tm_k, &kq_full, 64, h, n * 64, b);
        tma_load_4d(sm + L::QB, &tm_q, &kq_full, 0, h, n * 64, b);
        tma_load_4d(sm + L::QB + 8192, &tm_q, &kq_full, 64, h, n * 64, b);
    };
    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        const long long c0 = clock64();
        while (!mbar_try_wait(bar, parity)) {
            if (*abort_v || clock64() - c0 > kSpinLimit) {
                *abort_v = 1;
                return false;
            }
            __nanosleep(64);
        }
        return true;
    };
    constexpr uint32_t I_ABMN = idesc_bf16(128, 64, true, true);

    const long long Gs = gridDim.x;
    long long j = blockIdx.x;
    if (tid == 0 && j < nchunk_all) load_kq(j);
    bool failed = false;
    for (int it = 0; j < nchunk_all; j += Gs, ++it) {
        const long long seq = j / nch;
        const int n = (int)(j - seq * nch);
        const int b = (int)(seq / H), h = (int)(seq % H);
        const int nvalid = min(64, T - n * 64);
        // token-head index of the chunk's first token; alpha / b / w rows are
        // 128 floats per token-head
        const size_t th0 = ((size_t)b * T + (size_t)n * 64) * H + h;
        uint8_t *out = ws + (size_t)j * gw_chunk_bytes(GATE);

        // ---- gates: G[t][c] = sum_{s <= t} log2 alpha[s][c] (thread = channel);
        // ---- the 64 loads go out together, then the prefix ----
        {
            float a[64];
#pragma unroll
            for (int t = 0; t < 64; ++t)
                a[t] = t < nvalid ? __ldg(alpha + (th0 + (size_t)t * H) * 128 + tid) : 1.f;
            // the hardware log2 (absolute error about 2^-22 per term: the
            // decay factors it gives are exact to ~1e-5 relative, far below
            // the bf16 operands they scale)
            float g = 0.f;
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                g += __log2f(a[t]);
                Gt[t * kGLD + tid] = g;
            }
            reinterpret_cast<float *>(out + kGwF)[tid] = exp2f(g);  // e^(G_C) of the state update
            if (tid < 64)
                bet[tid] = tid < nvalid ? (GATE == kKda ? beta[th0 + (size_t)tid * H] : 1.f) : 0.f;
        }
        bool ok = true;
        if (tid == 0) ok = wait(&kq_full, it & 1);
        if (named_sync_or(kBarKey, kGpThreads, !ok)) { failed = true; break; }

        // ---- scaled tiles, 16-byte pieces: K~ (.) e^G (W's operand), the
        // ---- erase rows E (GDN2, A's left operand), Q (.) e^G, K (.) e^(G_C - G) ----
#pragma unroll
        for (int p = tid; p < 1024; p += kGpThreads) {
            const int t = p >> 4, c16 = p & 15, c0 = c16 * 8;
            const uint32_t off = piece_off(t, c16);
            const uint4 kr = *reinterpret_cast<const uint4 *>(sm + L::KB + off);
            const uint4 qr = *reinterpret_cast<const uint4 *>(sm + L::QB + off);
            const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w}, qw[4] = {qr.x, qr.y, qr.z, qr.w};
            float bgv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) bgv[e] = 1.f;
            if (GATE == kGdn2 && t < nvalid) {
                const float4 *bp = reinterpret_cast<const float4 *>(
                    bgate + (th0 + (size_t)t * H) * 128 + c0);
                const float4 b0 = bp[0], b1 = bp[1];
                bgv[0] = b0.x; bgv[1] = b0.y; bgv[2] = b0.z; bgv[3] = b0.w;
                bgv[4] = b1.x; bgv[5] = b1.y; bgv[6] = b1.z; bgv[7] = b1.w;
            }
            uint32_t kt[4], qt[4], kh[4], ev[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 g = *reinterpret_cast<const float2 *>(Gt + t * kGLD + c0 + 2 * e);
                const float2 gc = *reinterpret_cast<const float2 *>(Gt + 63 * kGLD + c0 + 2 * e);
                const float2 kf = bf16x2_to_f2(kw[e]), qf = bf16x2_to_f2(qw[e]);
                const float f0 = ex2f(g.x), f1 = ex2f(g.y);
                const float e0 = bgv[2 * e] * kf.x, e1 = bgv[2 * e + 1] * kf.y;
                kt[e] = pack_bf16(e0 * f0, e1 * f1);
                ev[e] = pack_bf16(e0, e1);
                qt[e] = pack_bf16(qf.x * f0, qf.y * f1);
                kh[e] = pack_bf16(kf.x * ex2f(gc.x - g.x), kf.y * ex2f(gc.y - g.y));
            }
            *reinterpret_cast<uint4 *>(sm + L::KT + off) = make_uint4(kt[0], kt[1], kt[2], kt[3]);
            if (GATE == kGdn2)
                *reinterpret_cast<uint4 *>(sm + L::AF + off) = make_uint4(ev[0], ev[1], ev[2], ev[3]);
            *reinterpret_cast<uint4 *>(out + kGwQ + off) = make_uint4(qt[0], qt[1], qt[2], qt[3]);
            *reinterpret_cast<uint4 *>(out + kGwK + off) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
        }
        named_sync(kBarKey, kGpThreads);

        // ---- row block I = warp of A and P: rows 16 I .. 16 I + 15, columns
        // ---- s < 16 (I + 1), referred to token m = 16 I + 7 ----
        {
            const int I = warp, m = 16 * I + 7;
            const int g = lane >> 2, t4 = lane & 3;
            const uint8_t *LT = sm + (GATE == kGdn2 ? L::AF : L::KB);  // E or K rows
            float acc[2][8][4];
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[a][nt][e] = 0.f;
#pragma unroll 1
            for (int ks = 0; ks < 8; ++ks) {
                const int ja = 16 * ks + 2 * t4;  // channels ja, ja + 1 and ja + 8, ja + 9
                const float2 gm0 = *reinterpret_cast<const float2 *>(Gt + m * kGLD + ja);
                const float2 gm1 = *reinterpret_cast<const float2 *>(Gt + m * kGLD + ja + 8);
                uint32_t aL[4], aQ[4];
#pragma unroll
                for (int rh = 0; rh < 2; ++rh) {
                    const int t = 16 * I + g + 8 * rh;
                    const float2 gt0 = *reinterpret_cast<const float2 *>(Gt + t * kGLD + ja);
                    const float2 gt1 = *reinterpret_cast<const float2 *>(Gt + t * kGLD + ja + 8);
                    const float f00 = ex2f(gt0.x - gm0.x), f01 = ex2f(gt0.y - gm0.y);
                    const float f10 = ex2f(gt1.x - gm1.x), f11 = ex2f(gt1.y - gm1.y);
                    const float2 l0 = bf16x2_to_f2(ld_pair(LT, t, ja));
                    const float2 l1 = bf16x2_to_f2(ld_pair(LT, t, ja + 8));
                    const float2 q0 = bf16x2_to_f2(ld_pair(sm + L::QB, t, ja));
                    const float2 q1 = bf16x2_to_f2(ld_pair(sm + L::QB, t, ja + 8));
                    aL[rh] = pack_bf16(l0.x * f00, l0.y * f01);
                    aL[2 + rh] = pack_bf16(l1.x * f10, l1.y * f11);
                    aQ[rh] = pack_bf16(q0.x * f00, q0.y * f01);
                    aQ[2 + rh] = pack_bf16(q1.x * f10, q1.y * f11);
                }
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    if (nt < 2 * (I + 1)) {
                        const int s = 8 * nt + g;
                        const float2 gs0 = *reinterpret_cast<const float2 *>(Gt + s * kGLD + ja);
                        const float2 gs1 =
                            *reinterpret_cast<const float2 *>(Gt + s * kGLD + ja + 8);
                        const float2 k0 = bf16x2_to_f2(ld_pair(sm + L::KB, s, ja));
                        const float2 k1 = bf16x2_to_f2(ld_pair(sm + L::KB, s, ja + 8));
                        const uint32_t b0 = pack_bf16(k0.x * ex2f(gm0.x - gs0.x),
                                                      k0.y * ex2f(gm0.y - gs0.y));
                        const uint32_t b1 = pack_bf16(k1.x * ex2f(gm1.x - gs1.x),
                                                      k1.y * ex2f(gm1.y - gs1.y));
                        mma_16816(acc[0][nt], aL, b0, b1);
                        mma_16816(acc[1][nt], aQ, b0, b1);
                    }
                }
            }
            // every warp has read the K / Q boxes (and E): the next chunk's
            // boxes may land; A's rows go where E was
            named_sync(kBarKey, kGpThreads);
            if (tid == 0 && j + Gs < nchunk_all) load_kq(j + Gs);
#pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
                const int t = 16 * I + g + 8 * rh;
                const float bt = bet[t];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const int s = 8 * nt + 2 * t4;
                    const float a0 = (s < t) ? bt * acc[0][nt][2 * rh] : 0.f;
                    const float a1 = (s + 1 < t) ? bt * acc[0][nt][2 * rh + 1] : 0.f;
                    *reinterpret_cast<float2 *>(AF + t * kLD + s) = make_float2(a0, a1);
                    const float p0 = (s <= t) ? acc[1][nt][2 * rh] : 0.f;
                    const float p1 = (s + 1 <= t) ? acc[1][nt][2 * rh + 1] : 0.f;
                    *reinterpret_cast<uint32_t *>(out + kGwP + swz128(t, nt) + 4 * t4) =
                        pack_bf16(p0, p1);
                }
            }
        }
        named_sync(kBarKey, kGpThreads);

        // ---- T = (I + A)^{-1}; T_b^T (both images: the inverse's T'^T with
        // ---- gamma = 1 equals T''^T) into shared memory and the workspace ----
        chunk_inverse_tprime<kGpThreads>(AF, bet, ones, sm + L::TB, out + kGwTB, tid);
        fence_proxy_async_smem();
        named_sync(kBarKey, kGpThreads);

        // ---- W^T = (K~ (.) e^G)^T T_b^T (tcgen05, 128 channels x 64 tokens) ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tb, sdesc(base + L::KT + ks * 2048, 8192, 1024),
                         sdesc(base + L::TB + ks * 2048, 8192, 1024), I_ABMN, ks > 0);
            mma_commit(&bar_w);
            ok = wait(&bar_w, it & 1);
        }
        if (named_sync_or(kBarKey, kGpThreads, !ok)) { failed = true; break; }
        {
            tc_fence_after();
            const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
            const int row = warp * 32 + lane;  // key channel
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
                float vv[32];
                tmem_ld32(tb + lane_off + 32 * ch, vv);
                tmem_ld_wait();
                store_row<4>(out + kGwNW, row, 4 * ch, vv, -1.f);
            }
            tc_fence_before();
        }
        named_sync(kBarKey, kGpThreads);  // TMEM, KT, TB, AF and G are rewritten next
    }

    if (failed) *abort_v = 1;
    tc_fence_before();
    __syncthreads();
    if (*abort_v) {
        if (tid == 0) {
            if (status) atomicOr(status, kStatusTimeout);
            mma_commit(&drain);
            mbar_wait(&drain, 0, kSpinLimit / 16);
            mbar_wait(&kq_full, 0, kSpinLimit / 16);
            mbar_wait(&kq_full, 1, kSpinLimit / 16);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 64);
    }
}

// ---------------------------------------------------------------- GDN2 write content
// Z = w (.) V of every chunk into the workspace as its two 128-byte-swizzled
// [64][64] bf16 boxes.  One 16-byte piece (8 channels of a token and head) per
// thread and step, taken in the memory order of v and w (piece p covers
// elements 8 p .. 8 p + 7 of both: contiguous streams), four steps' loads
// issued together; then the rows of each sequence's last chunk past T are
// zeroed.  One 128-thread CTA per SM, beside the key-side pass's two: no
// shared memory and at most 80 registers a thread (what those two CTAs leave
// on an SM), which the minimum of six resident CTAs in the launch bounds asks
// of the compiler.
constexpr int kZThreads = 128, kZUnroll = 4;
__device__ __forceinline__ uint8_t *z_piece(uint8_t *ws, int T, int H, long long tok, int h,
                                            int c16) {
    const int nch = (T + 63) / 64;
    const long long b = tok / T;
    const int t = (int)(tok - b * T);
    const long long j = (b * H + h) * nch + (t >> 6);
    return ws + (size_t)j * gw_chunk_bytes(kGdn2) + kGwZ + piece_off(t & 63, c16);
}
__global__ void __launch_bounds__(kZThreads, 6)
    gated_z_kernel(const __nv_bfloat16 *__restrict__ v, const float *__restrict__ wgate,
                   uint8_t *__restrict__ ws, int B, int T, int H) {
    const long long npieces = (long long)B * T * H * 16;
    const long long stride = (long long)gridDim.x * kZThreads;
    for (long long p0 = (long long)blockIdx.x * kZThreads + threadIdx.x; p0 < npieces;
         p0 += stride * kZUnroll) {
        uint4 vr[kZUnroll];
        float4 w0[kZUnroll], w1[kZUnroll];
#pragma unroll
        for (int u = 0; u < kZUnroll; ++u) {
            const long long p = p0 + u * stride;
            vr[u] = make_uint4(0u, 0u, 0u, 0u);
            w0[u] = w1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p < npieces) {
                vr[u] = __ldcs(reinterpret_cast<const uint4 *>(v) + p);
                w0[u] = __ldcs(reinterpret_cast<const float4 *>(wgate) + 2 * p);
                w1[u] = __ldcs(reinterpret_cast<const float4 *>(wgate) + 2 * p + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < kZUnroll; ++u) {
            const long long p = p0 + u * stride;
            if (p >= npieces) break;
            const long long row = p >> 4;  // token-head
            const float wv[8] = {w0[u].x, w0[u].y, w0[u].z, w0[u].w,
                                 w1[u].x, w1[u].y, w1[u].z, w1[u].w};
            const uint32_t vw[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
            uint32_t zw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 vf = bf16x2_to_f2(vw[e]);
                zw[e] = pack_bf16(wv[2 * e] * vf.x, wv[2 * e + 1] * vf.y);
            }
            *reinterpret_cast<uint4 *>(z_piece(ws, T, H, row / H, (int)(row % H), (int)p & 15)) =
                make_uint4(zw[0], zw[1], zw[2], zw[3]);
        }
    }
    // rows of the last chunk past T: zero
    const int pad = (64 - T % 64) % 64;
    const long long npad = (long long)B * H * pad * 16;
    for (long long p = (long long)blockIdx.x * kZThreads + threadIdx.x; p < npad; p += stride) {
        const int c16 = (int)(p & 15);
        const long long r = p >> 4;  // (b, h, padded row)
        const int pr = (int)(r % pad);
        const long long bh = r / pad;
        const int nch = (T + 63) / 64;
        const long long j = bh * nch + nch - 1;
        *reinterpret_cast<uint4 *>(ws + (size_t)j * gw_chunk_bytes(kGdn2) + kGwZ +
                                   piece_off(T % 64 + pr, c16)) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// The side stream for gated_z_kernel on the current device and context, with
// the fork / join events; created once, nullptr when that fails (the kernel
// then runs on the caller's stream).
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    uintptr_t ctx = 0;
};
std::mutex g_side_mu;  // also held while a call enqueues its fork and join
SideStream g_side[64];
SideStream *side_stream(int dev) {
    SideStream &ss = g_side[dev];
    if (ss.ctx != context_key() || !ss.s) {
        ss = SideStream{};
        if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            ss = SideStream{};
            return nullptr;
        }
        ss.ctx = context_key();
    }
    return &ss;
}

// ---------------------------------------------------------------- state pass
// Rings (slots): Q (.) e^G, K (.) e^(G_C - G) with e^(G_C), P (three each);
// Z / V and [T_b^T | -W^T] (two each).  The issuer loads chunk n + 2 in chunk
// n's window, once U(n) has completed: that covers dS(n - 1), O^T(n - 1) and
// this thread's earlier products, the readers of the slots it refills.
struct GsLayout {
    static constexpr uint32_t KR = 0;                 // 3 x 16 KB
    static constexpr uint32_t QR = KR + 3 * 16384;    // 3 x 16 KB
    static constexpr uint32_t VB = QR + 3 * 16384;    // 2 x 16 KB
    static constexpr uint32_t TW = VB + 2 * 16384;    // 2 x 24 KB: T_b^T, -W^T
    static constexpr uint32_t PP = TW + 2 * 24576;    // 3 x 8 KB
    static constexpr uint32_t OST = PP + 3 * 8192;    // output staging, 2 x 64 x 64
    static constexpr uint32_t FR = OST + 16384;       // 3 x 512 B
    static constexpr uint32_t END = FR + 3 * 512;
    static constexpr size_t SMEM = END;
    static_assert(SMEM + 1024 <= 232448, "shared memory budget");
    static __device__ __forceinline__ uint32_t kbuf(int n) { return KR + (n % 3) * 16384; }
    static __device__ __forceinline__ uint32_t qbuf(int n) { return QR + (n % 3) * 16384; }
    static __device__ __forceinline__ uint32_t vbuf(int n) { return VB + (n & 1) * 16384; }
    static __device__ __forceinline__ uint32_t tbuf(int n) { return TW + (n & 1) * 24576; }
    static __device__ __forceinline__ uint32_t nwbuf(int n) { return tbuf(n) + 8192; }
    static __device__ __forceinline__ uint32_t pbuf(int n) { return PP + (n % 3) * 8192; }
    static __device__ __forceinline__ uint32_t fbuf(int n) { return FR + (n % 3) * 512; }
    // TMEM columns: O^T of even / odd chunks, U~^T / U^T of even / odd
    // chunks (bf16 U^T written back into the first 16 columns of each 32),
    // the bf16 state, dS
    static constexpr uint32_t O0 = 0, O1 = 64, UA = 128, SBT = 256, DS = 384;
    static __device__ __forceinline__ uint32_t ocol(int n) { return (n & 1) ? O1 : O0; }
    static __device__ __forceinline__ uint32_t ua(int n) { return UA + 64 * (n & 1); }
    static __device__ __forceinline__ uint32_t ut_col(int n, int ks) {
        return ua(n) + 32 * (ks >> 1) + 8 * (ks & 1);
    }
};
constexpr int kGsThreads = 288;  // warp 0: issuer (lane 0); warps 1-8: state group
constexpr int kGsBarState = 2, kGsBarOut = 3, kGsBarOut2 = 4;

template <int GATE>
__global__ void __launch_bounds__(kGsThreads, 1)
    prefill_gated_state_kernel(const __grid_constant__ CUtensorMap tm_v,
                               const __grid_constant__ CUtensorMap tm_o,
                               const float *__restrict__ S0, bool want_o, float *__restrict__ ST,
                               int T, int H, int BH, const uint8_t *__restrict__ ws, int *status) {
    using L = GsLayout;
    constexpr int K = 128, KH = 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0 && status) atomicOr(status, kStatusBounds);
        return;
    }
    uint8_t *sm = smem_raw;
    __shared__ uint64_t k_full[3], q_full[3], p_full[3], v_full[2], t_full[2], bar_w, bar_u,
        bar_s, bar_os, bar_o2, u_sig, drain[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    volatile int *abort_v = &abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const size_t seq = blockIdx.x;
    if (!bounds_ok(seq < (size_t)BH && T >= 1, status)) return;
    const int b = (int)(seq / H), h = (int)(seq % H);
    const int nchunks = (T + 63) / 64;
    const bool outs = want_o;
    const uint32_t base = smem_u32(sm);
    const uint32_t cb = gw_chunk_bytes(GATE);
    const uint8_t *ws_seq = ws + seq * (size_t)nchunks * cb;

    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        uint64_t *bars[] = {&k_full[0], &k_full[1], &k_full[2], &q_full[0], &q_full[1],
                            &q_full[2], &p_full[0], &p_full[1], &p_full[2], &v_full[0],
                            &v_full[1], &t_full[0], &t_full[1], &bar_w,     &bar_u,
                            &bar_s,     &bar_os,    &bar_o2,    &u_sig,     &drain[0],
                            &drain[1]};
        for (uint64_t *bb : bars) mbar_init(bb, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int quad_row = (warp & 3) * 32 + lane;

    auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait_or_abort(bar, parity, kSpinLimit, abort_v);
        if (!ok) *abort_v = 1;
        return ok;
    };
    constexpr uint32_t I_MM = idesc_bf16(128, 64, false, false);
    constexpr uint32_t I_ABMN = idesc_bf16(128, 64, true, true);
    constexpr uint32_t I_BMN = idesc_bf16(128, 64, false, true);
    constexpr uint32_t I_DS = idesc_bf16(128, K, false, true);

    bool failed = false;
    if (warp == 0) {
        // ================================================================ issuer
        if (lane == 0) {
            tma_prefetch_desc(&tm_v);
            if (outs) tma_prefetch_desc(&tm_o);
            auto chunk = [&](int n) { return ws_seq + (size_t)n * cb; };
            auto load_k = [&](int n) {  // K (.) e^(G_C - G) and e^(G_C)
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                uint64_t *bar = &k_full[n % 3];
                mbar_arrive_expect_tx(bar, 16384 + 512);
                bulk_load(sm + L::kbuf(n), chunk(n) + kGwK, 16384, bar);
                bulk_load(sm + L::fbuf(n), chunk(n) + kGwF, 512, bar);
            };
            auto load_q = [&](int n) {
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                mbar_arrive_expect_tx(&q_full[n % 3], 16384);
                bulk_load(sm + L::qbuf(n), chunk(n) + kGwQ, 16384, &q_full[n % 3]);
            };
            auto load_p = [&](int n) {
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                mbar_arrive_expect_tx(&p_full[n % 3], 8192);
                bulk_load(sm + L::pbuf(n), chunk(n) + kGwP, 8192, &p_full[n % 3]);
            };
            auto load_t = [&](int n) {  // T_b^T and -W^T (adjacent in the workspace)
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                mbar_arrive_expect_tx(&t_full[n & 1], 24576);
                bulk_load(sm + L::tbuf(n), chunk(n) + kGwTB, 24576, &t_full[n & 1]);
            };
            auto load_v = [&](int n) {  // V (KDA) or w (.) V (GDN2)
                if (!bounds_ok(n >= 0 && n < nchunks, status)) return;
                uint64_t *bar = &v_full[n & 1];
                uint8_t *dst = sm + L::vbuf(n);
                mbar_arrive_expect_tx(bar, 16384);
                if (GATE == kGdn2) {
                    bulk_load(dst, chunk(n) + kGwZ, 16384, bar);
                } else {
                    tma_load_4d(dst, &tm_v, bar, 0, h, n * 64, b);
                    tma_load_4d(dst + 8192, &tm_v, bar, 64, h, n * 64, b);
                }
            };
            auto load_all = [&](int n) {
                load_k(n);
                load_q(n);
                load_t(n);
                load_v(n);
                if (outs) load_p(n);
            };
            // U~^T(n) = Z^T T_b^T (U slot n % 2)
            auto issue_ut = [&](int n) -> bool {
                if (!wait(&t_full[n & 1], (n >> 1) & 1)) return false;
                if (!wait(&v_full[n & 1], (n >> 1) & 1)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tb + L::ua(n), sdesc(base + L::vbuf(n) + ks * 2048, 8192, 1024),
                             sdesc(base + L::tbuf(n) + ks * 2048, 8192, 1024), I_ABMN, ks > 0);
                mma_commit(&bar_w);
                return true;
            };
            for (int m = 0; m < 2 && m < nchunks; ++m) load_all(m);
            bool ok = issue_ut(0);
            for (int n = 0; ok && n < nchunks; ++n) {
                if (outs) {
                    // O^T(n) = S(n-1) (Q (.) e^G)^T once the state thread has
                    // issued U(n), which reads the same S(n-1)
                    ok = wait(&u_sig, n & 1) && wait(&q_full[n % 3], (n / 3) & 1);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < K / 16; ++ks) {
                            const uint32_t ko = (ks / 4) * 8192 + (ks % 4) * 32;
                            mma_bf16_ta(tb + L::ocol(n), tb + L::SBT + 8 * ks,
                                        sdesc(base + L::qbuf(n) + ko, 16, 1024), I_MM, ks > 0);
                        }
                        mma_commit(&bar_os);
                    }
                }
                ok = ok && wait(&bar_u, n & 1);
                if (!ok) break;
                if (n + 2 < nchunks) load_all(n + 2);
                if (n + 1 < nchunks) ok = issue_ut(n + 1);
            }
            if (!ok) failed = true;
        }
    } else {
        // ================================================================ state group
        const int sid = tid - 32;  // 0..255
        const int sw = sid >> 5;   // state warp 0..7
        const int c = quad_row;    // state row = TMEM lane = value channel
        const int hf = sw >> 2;    // column half
        float S[KH];
        {
            const int j0 = hf * KH;
#pragma unroll
            for (int jj = 0; jj < KH; jj += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (S0) x = *reinterpret_cast<const float4 *>(S0 + seq * K * K + (size_t)c * K + j0 + jj);
                S[jj] = x.x; S[jj + 1] = x.y; S[jj + 2] = x.z; S[jj + 3] = x.w;
            }
#pragma unroll
            for (int p = 0; p < KH / 32; ++p) {
                float vv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) vv[i] = S[32 * p + i];
                uint32_t w[16];
                pack_row(vv, w);
                tmem_st16(tb + lane_off + L::SBT + (j0 + 32 * p) / 2, w);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        named_sync(kGsBarState, 256);

        // U^T(m) = U~^T(m) + S (-W^T(m)) (state thread), then u_sig
        auto issue_u = [&](int m) -> bool {
            if (!wait(&bar_w, m & 1)) return false;
            if (!wait(&t_full[m & 1], (m >> 1) & 1)) return false;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks)
                mma_bf16_ta(tb + L::ua(m), tb + L::SBT + 8 * ks,
                            sdesc(base + L::nwbuf(m) + ks * 2048, 8192, 1024), I_BMN, 1u);
            mma_commit(&bar_u);
            tc_fence_before();
            if (outs) mbar_arrive(&u_sig);
            return true;
        };
        auto store_out = [&](int m) -> bool {
            bool okw = true;
            if (sid == 128) okw = wait(&bar_o2, m & 1);
            if (sw == 3 && lane == 0) bulk_wait_read_all();
            if (named_sync_or(kGsBarOut, 160, !okw)) return false;
            if (sw >= 4) {
                tc_fence_after();
                const bool odd = lane & 1;
                uint8_t *tile = sm + L::OST + (c >> 6) * 8192;
                const uint32_t cbk = (uint32_t)(c & 63) >> 3, cw = (uint32_t)(c & 6) * 2;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float vv[32];
                    tmem_ld32(tb + lane_off + L::ocol(m) + 32 * half, vv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float got = __shfl_xor_sync(0xffffffffu, odd ? vv[i] : vv[i + 1], 1);
                        const uint32_t t = 32 * half + i + (odd ? 1 : 0);
                        const float lo = odd ? got : vv[i], hi = odd ? vv[i + 1] : got;
                        *reinterpret_cast<uint32_t *>(tile + swz128(t, cbk) + cw) =
                            pack_bf16(lo, hi);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
            }
            named_sync(kGsBarOut2, 160);
            if (sw == 3 && lane == 0) {
                if (bounds_ok(m >= 0 && m < nchunks, status)) {
                    tma_store_4d(&tm_o, sm + L::OST, 0, h, m * 64, b);
                    tma_store_4d(&tm_o, sm + L::OST + 8192, 64, h, m * 64, b);
                }
                bulk_commit_group();
            }
            return true;
        };
        if (sw == 0) {
            bool ok0 = true;
            if (lane == 0) ok0 = issue_u(0);
            ok0 = __shfl_sync(0xffffffffu, ok0, 0);
            failed = !ok0;
        }
        for (int n = 0; n < nchunks; ++n) {
            bool ok = !failed;
            if (sid == 0 && ok) ok = wait(&bar_u, n & 1);
            if (named_sync_or(kGsBarState, 256, !ok)) { failed = true; break; }
            // ---- U epilogue: bf16 U^T into the U slot (first 16 of each 32 columns) ----
            {
                tc_fence_after();
                float vv[32];
                tmem_ld32(tb + lane_off + L::ua(n) + 32 * hf, vv);
                tmem_ld_wait();
                uint32_t w[16];
                pack_row(vv, w);
                tmem_st16(tb + lane_off + L::ua(n) + 32 * hf, w);
                tmem_st_wait();
            }
            tc_fence_before();
            named_sync(kGsBarState, 256);
            // ---- dS = U^T (K (.) e^(G_C - G)), then O^T += U^T P^T (warp 1) ----
            if (sid == 0) {
                ok = wait(&k_full[n % 3], (n / 3) & 1);
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16_ta(tb + L::DS, tb + L::ut_col(n, ks),
                                    sdesc(base + L::kbuf(n) + ks * 2048, 8192, 1024), I_DS,
                                    ks > 0);
                    mma_commit(&bar_s);
                }
                if (ok && outs) {
                    ok = wait(&bar_os, n & 1) && wait(&p_full[n % 3], (n / 3) & 1);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_bf16_ta(tb + L::ocol(n), tb + L::ut_col(n, ks),
                                        sdesc(base + L::pbuf(n) + ks * 32, 16, 1024), I_MM, 1);
                        mma_commit(&bar_o2);
                    }
                }
                ok = ok && wait(&bar_s, n & 1);
            }
            if (named_sync_or(kGsBarState, 256, !ok)) { failed = true; break; }
            // ---- S <- S diag(e^(G_C)) + dS, and its bf16 copy ----
            {
                // e^(G_C) arrived with the K operand (k_full(n), seen above by
                // thread 0; every thread takes the completed phase itself)
                ok = wait(&k_full[n % 3], (n / 3) & 1);
                tc_fence_after();
                const float *f = reinterpret_cast<const float *>(sm + L::fbuf(n));
                const int j0 = hf * KH;
#pragma unroll
                for (int p = 0; p < KH / 32; ++p) {
                    float vv[32];
                    tmem_ld32(tb + lane_off + L::DS + j0 + 32 * p, vv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        S[32 * p + i] = fmaf(f[j0 + 32 * p + i], S[32 * p + i], vv[i]);
                        vv[i] = S[32 * p + i];
                    }
                    uint32_t w[16];
                    pack_row(vv, w);
                    tmem_st16(tb + lane_off + L::SBT + (j0 + 32 * p) / 2, w);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            if (named_sync_or(kGsBarState, 256, !ok)) { failed = true; break; }
            bool ok1 = true;
            if (sw == 0) {
                if (lane == 0 && n + 1 < nchunks) ok1 = issue_u(n + 1);
                ok1 = __shfl_sync(0xffffffffu, ok1, 0);
            } else if (sw >= 3 && outs) {
                ok1 = store_out(n);
            }
            if (!ok1) failed = true;
        }
        if (sw == 3 && lane == 0 && outs) bulk_wait_all();
        if (!failed && ST != nullptr) {
            const int j0 = hf * KH;
#pragma unroll
            for (int jj = 0; jj < KH; jj += 4)
                *reinterpret_cast<float4 *>(ST + seq * K * K + (size_t)c * K + j0 + jj) =
                    make_float4(S[jj], S[jj + 1], S[jj + 2], S[jj + 3]);
        }
    }

    if (failed) *abort_v = 1;
    tc_fence_before();
    __syncthreads();
    if (*abort_v) {
        if (tid == 0 || tid == 32) {
            uint64_t *d = &drain[tid == 0 ? 0 : 1];
            mma_commit(d);
            mbar_wait(d, 0, kSpinLimit / 16);
        }
        if (tid == 0) {
            if (status) atomicOr(status, kStatusTimeout);
            uint64_t *loads[] = {&k_full[0], &k_full[1], &k_full[2], &q_full[0], &q_full[1],
                                 &q_full[2], &p_full[0], &p_full[1], &p_full[2], &v_full[0],
                                 &v_full[1], &t_full[0], &t_full[1]};
            for (uint64_t *lb : loads) {
                mbar_wait(lb, 0, kSpinLimit / 16);
                mbar_wait(lb, 1, kSpinLimit / 16);
            }
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

template <int GATE>
cudaError_t launch_gated_tc_t(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *bgate, const float *wgate,
                              const float *S0, void *o, float *ST, int B, int T, int H,
                              uint8_t *ws, cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_token_map(&mq, q, B, T, T, H, 128) || !make_token_map(&mk, k, B, T, T, H, 128) ||
        !make_token_map(&mv, v, B, T, T, H, 128))
        return cudaErrorInvalidValue;
    if (o) {
        if (!make_token_map(&mo, o, B, T, T, H, 128)) return cudaErrorInvalidValue;
    } else {
        mo = mv;
    }
    auto prep = prefill_gated_prep_kernel<GATE>;
    auto state = prefill_gated_state_kernel<GATE>;
    static uintptr_t attr_set[64] = {};  // context the attributes were set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev] != context_key()) {
        cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)GpLayout::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prep, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)GsLayout::SMEM);
        // the Z kernel (no shared memory) shares SMs with the key-side pass:
        // the same carveout, so that an SM it reaches first still takes that
        // pass's two CTAs
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gated_z_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev] = context_key();
    }
    const long long BH = (long long)B * H;
    const long long total = BH * ((T + 63) / 64);
    const long long grid = std::min<long long>(total, (long long)kGpCtasPerSm * sm_count());
    int *status = device_status_ptr();
    if (GATE != kGdn2) {
        prep<<<(unsigned)grid, kGpThreads, GpLayout::SMEM, stream>>>(mq, mk, alpha, beta, bgate,
                                                                     ws, T, H, total, status);
    } else {
        // Z on the side stream, forked from the caller's stream (after its
        // writes of v and w) and joined back before the state pass
        std::lock_guard<std::mutex> lock(g_side_mu);
        SideStream *ss = side_stream(dev);
        cudaStream_t zs = ss ? ss->s : stream;
        cudaError_t e = cudaSuccess;
        // (the key-side pass is launched first, so that its CTAs are placed
        // first; the fork event marks the caller's earlier work only)
        if (ss) {
            e = cudaEventRecord(ss->fork, stream);
            if (e != cudaSuccess) return e;
        }
        prep<<<(unsigned)grid, kGpThreads, GpLayout::SMEM, stream>>>(mq, mk, alpha, beta, bgate,
                                                                     ws, T, H, total, status);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (ss) {
            e = cudaStreamWaitEvent(zs, ss->fork, 0);
            if (e != cudaSuccess) return e;
        }
        gated_z_kernel<<<(unsigned)sm_count(), kZThreads, 0, zs>>>(
            static_cast<const __nv_bfloat16 *>(v), wgate, ws, B, T, H);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (ss) {
            e = cudaEventRecord(ss->join, zs);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ss->join, 0);
            if (e != cudaSuccess) return e;
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    state<<<(unsigned)BH, kGsThreads, GsLayout::SMEM, stream>>>(mv, mo, S0, o != nullptr, ST, T,
                                                                H, (int)BH, ws, status);
    return cudaGetLastError();
}

}  // namespace

size_t prefill_gated_tc_workspace(int B, int T, int H, int gate) {
    if (gate != kKda && gate != kGdn2) return 0;
    return (size_t)B * H * (size_t)((T + 63) / 64) * gw_chunk_bytes(gate);
}

cudaError_t launch_prefill_gated_tc(const void *q, const void *k, const void *v,
                                    const float *alpha, const float *beta, const float *bgate,
                                    const float *wgate, const float *S0, void *o, float *ST,
                                    int B, int T, int H, int gate, void *workspace,
                                    cudaStream_t stream) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (gate == kKda)
        return launch_gated_tc_t<kKda>(q, k, v, alpha, beta, nullptr, nullptr, S0, o, ST, B, T,
                                       H, ws, stream);
    if (gate == kGdn2)
        return launch_gated_tc_t<kGdn2>(q, k, v, alpha, nullptr, bgate, wgate, S0, o, ST, B, T,
                                        H, ws, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
