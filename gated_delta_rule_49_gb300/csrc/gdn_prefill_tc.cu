// Chunkwise prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// bf16 q/k/v, float32 state carried on chip from chunk to chunk.
//
// One CTA (8 warps) owns one (b, h) sequence and walks its 64-token chunks.
// With G_t the in-chunk cumulative log-decay, gamma_t = exp(G_t),
// Gamma_ts = exp(G_t - G_s) (a difference, never a ratio of gammas):
//
//   A_ts = beta_t Gamma_ts (k_t . k_s) (s < t)     P_ts = Gamma_ts (q_t . k_s) (s <= t)
//   T    = (I + A)^{-1},  T' = T diag(beta gamma),  T'' = T diag(beta)
//   W^T  = K^T T'^T,      U~^T = V^T T''^T
//   U^T  = U~^T - S W^T          pseudo-values u_t = beta_t (v_t - alpha_t S_{t-1} k_t)
//   O^T  = diag-scaled S Q^T (by gamma_t) + U^T P^T
//   S   <- gamma_C S + U^T diag(exp(G_C - G_s)) K
//
// -- the token recurrence unrolled over a chunk (the pseudo-value rewriting
// of the delta rule, "On State Reduction in Linear Attention" notes, Sec. 2.3).
// Everything is written transposed so that every product has M = 128 rows
// (value channels or stacked tiles), the natural TMEM layout (row = lane).
//
// Data movement: TMA loads 64-token x 64-channel bf16 boxes of q, k, v with
// the 128-byte swizzle into a two-stage ring; the same K tile serves as a
// K-major operand (contraction over channels) and as an MN-major operand
// (contraction over tokens).  Intermediate operands (P, T', T'', -W^T, U^T,
// U^T diag(decay), the bf16 copy of S) are written by threads in the same
// swizzled layout.  The float32 state lives in registers: thread (lane c,
// half h) holds row c, columns [h K/2, (h+1) K/2).
//
// A ragged last chunk: TMA fills tokens past T with zeros; beta = 0 and
// log alpha = 0 there, which leaves every valid row unchanged.
#include "gdn_internal.cuh"
#include "gdn_sm100.cuh"

#include <cudaTypedefs.h>

namespace gdn {
namespace {

using namespace sm100;

constexpr int kTcThreads = 256;
constexpr long long kSpinLimit = 2000000000LL;  // ~1 s of SM clocks per wait

template <int K>
struct TcLayout {
    // one TMA stage: 64 x 64 bf16 boxes, 8 KB each
    static constexpr uint32_t KC0 = 0, QC0 = 8192, KC1 = 16384, QC1 = 24576;
    static constexpr uint32_t VC0 = K == 128 ? 32768 : 16384, VC1 = VC0 + 8192;
    static constexpr uint32_t STAGE = VC1 + 8192;
    static constexpr uint32_t TP = 2 * STAGE, TPP = TP + 8192, PT = TPP + 8192;
    static constexpr uint32_t NW = PT + 8192;                // K rows x 128 B (MN-major)
    static constexpr uint32_t SB = NW + K * 128;             // K/64 blocks of 128 rows
    static constexpr uint32_t UT = SB + (K / 64) * 16384;
    static constexpr uint32_t UD = UT + 16384;
    static constexpr uint32_t AF = UD + 16384;               // float [64][65]
    static constexpr uint32_t GATE = AF + 64 * 65 * 4;       // G, gamma, beta, decay
    static constexpr uint32_t END = GATE + 4 * 64 * 4;
    static constexpr uint32_t TX_BYTES = (K == 128 ? 6u : 4u) * 8192u;
    static constexpr size_t SMEM = END + 1024;               // + alignment slack
    // TMEM columns
    static constexpr uint32_t D1 = 0, WT = 64, UA = 128, OA = 192, OB = 256, DS = 320;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// Store 32 floats of one tile row as 4 swizzled 16-byte chunks starting at chunk c0.
__device__ __forceinline__ void store_row32(uint8_t *tile, uint32_t row, uint32_t c0,
                                            const float (&v)[32], float scale = 1.f) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint4 w;
        w.x = pack_bf16(v[8 * k + 0] * scale, v[8 * k + 1] * scale);
        w.y = pack_bf16(v[8 * k + 2] * scale, v[8 * k + 3] * scale);
        w.z = pack_bf16(v[8 * k + 4] * scale, v[8 * k + 5] * scale);
        w.w = pack_bf16(v[8 * k + 6] * scale, v[8 * k + 7] * scale);
        *reinterpret_cast<uint4 *>(tile + swz128(row, c0 + k)) = w;
    }
}

template <int K>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ alpha,
                      const float *__restrict__ beta, const float *__restrict__ S0,
                      __nv_bfloat16 *__restrict__ o, float *__restrict__ ST, int T, int H,
                      int *status) {
    using L = TcLayout<K>;
    constexpr int V = 128;
    constexpr int KH = K / 2;  // state columns per thread
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t bar_full[2];
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base_sh;

    float *AF = reinterpret_cast<float *>(sm + L::AF);
    float *Gs = reinterpret_cast<float *>(sm + L::GATE);
    float *gam = Gs + 64;
    float *bet = Gs + 128;
    float *dcy = Gs + 192;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;  // TMEM lane owned by this thread
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const size_t seq = (size_t)blockIdx.x;
    const int nchunks = (T + 63) / 64;
    const uint32_t base = smem_u32(sm);

    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }

    // initial state: fp32 in registers, bf16 copy in the SB tile
    float S[KH];
    {
        const int c = row;
        const int j0 = half * KH;
#pragma unroll
        for (int j = 0; j < KH; j += 4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (S0) x = *reinterpret_cast<const float4 *>(S0 + (seq * V + c) * K + j0 + j);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
#pragma unroll
        for (int p = 0; p < KH / 32; ++p) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = S[32 * p + i];
            const int j = j0 + 32 * p;
            store_row32(sm + L::SB + (j / 64) * 16384, c, (j % 64) / 8, v);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;

    auto issue_loads = [&](int n) {
        const int st = n & 1;
        uint8_t *stg = sm + st * L::STAGE;
        const int t0 = n * 64;
        mbar_arrive_expect_tx(&bar_full[st], L::TX_BYTES);
        tma_load_4d(stg + L::KC0, &tm_k, &bar_full[st], 0, h, t0, b);
        tma_load_4d(stg + L::QC0, &tm_q, &bar_full[st], 0, h, t0, b);
        if (K == 128) {
            tma_load_4d(stg + L::KC1, &tm_k, &bar_full[st], 64, h, t0, b);
            tma_load_4d(stg + L::QC1, &tm_q, &bar_full[st], 64, h, t0, b);
        }
        tma_load_4d(stg + L::VC0, &tm_v, &bar_full[st], 0, h, t0, b);
        tma_load_4d(stg + L::VC1, &tm_v, &bar_full[st], 64, h, t0, b);
    };
    if (tid == 0) {
        issue_loads(0);
        if (nchunks > 1) issue_loads(1);
    }

    constexpr uint32_t I_MM = idesc_bf16(128, 64, false, false);   // K-major x K-major
    constexpr uint32_t I_AMN = idesc_bf16(128, 64, true, false);   // MN-major A
    constexpr uint32_t I_BMN = idesc_bf16(128, 64, false, true);   // MN-major B, N = 64
    constexpr uint32_t I_DS = idesc_bf16(128, K, false, true);     // MN-major B, N = K

    uint32_t mma_phase = 0;
    bool failed = false;

    auto wait_mma = [&]() -> bool {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma, mma_phase & 1, kSpinLimit));
        ++mma_phase;
        tc_fence_after();
        return ok;
    };

    for (int n = 0; n < nchunks; ++n) {
        const int st = n & 1;
        const uint32_t stg = base + st * L::STAGE;
        const int c0 = n * 64;
        const int nvalid = min(64, T - c0);

        // ---- (1) chunk operands landed: KK^T, QK^T and S Q^T ----
        bool ok = true;
        if (tid == 0) {
            ok = mbar_wait(&bar_full[st], (n >> 1) & 1, kSpinLimit);
            tc_fence_after();
            if (ok) {
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const uint32_t kb = ks / 4, ko = (ks % 4) * 32;
                    const uint32_t kblk = stg + (kb ? L::KC1 : L::KC0) + ko;
                    const uint32_t qblk = stg + (kb ? L::QC1 : L::QC0) + ko;
                    mma_bf16(tb + L::D1, sdesc(kblk, 16, 1024), sdesc(kblk, 16, 1024), I_MM,
                             ks > 0);
                    mma_bf16(tb + L::OA, sdesc(base + L::SB + kb * 16384 + ko, 16, 1024),
                             sdesc(qblk, 16, 1024), I_MM, ks > 0);
                }
                mma_commit(&bar_mma);
            }
        }
        // gates of this chunk (warp 0): prefix sum of log alpha over 64 tokens
        if (warp == 0) {
            const int t0 = lane, t1 = lane + 32;
            const size_t i0 = ((size_t)b * T + c0 + t0) * H + h;
            const size_t i1 = ((size_t)b * T + c0 + t1) * H + h;
            float g0 = t0 < nvalid ? logf(alpha[i0]) : 0.f;
            float g1 = t1 < nvalid ? logf(alpha[i1]) : 0.f;
            bet[t0] = t0 < nvalid ? beta[i0] : 0.f;
            bet[t1] = t1 < nvalid ? beta[i1] : 0.f;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float a0 = __shfl_up_sync(0xffffffffu, g0, off);
                const float a1 = __shfl_up_sync(0xffffffffu, g1, off);
                if (lane >= off) { g0 += a0; g1 += a1; }
            }
            g1 += __shfl_sync(0xffffffffu, g0, 31);
            const float gC = __shfl_sync(0xffffffffu, g1, 31);
            Gs[t0] = g0; Gs[t1] = g1;
            gam[t0] = expf(g0); gam[t1] = expf(g1);
            dcy[t0] = expf(gC - g0); dcy[t1] = expf(gC - g1);
        }
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // ---- (2) A (fp32, for the solve) and P (bf16 operand) ----
        ok = wait_mma();
        if (ok) {
            float v[32];
            tmem_ld32(tb + lane_off + L::D1 + half * 32, v);
            tmem_ld_wait();
            const int t = row & 63;
            const float Gt = Gs[t];
            if (quad < 2) {
                const float bt = bet[t];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int s = half * 32 + i;
                    AF[t * 65 + s] = s < t ? bt * expf(Gt - Gs[s]) * v[i] : 0.f;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int s = half * 32 + i;
                    v[i] = s <= t ? expf(Gt - Gs[s]) * v[i] : 0.f;
                }
                store_row32(sm + L::PT, t, half * 4, v);
            }
        }
        fence_proxy_async_smem();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // ---- (3) T = (I + A)^{-1}, one column per thread; T' and T'' tiles ----
        if (tid < 64) {
            const int s = tid;
            float x[64];
#pragma unroll
            for (int t = 0; t < 64; ++t) x[t] = (t == s) ? 1.f : 0.f;
#pragma unroll
            for (int t = 1; t < 64; ++t) {
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int r = 0; r < t; ++r) {
                    const float a = AF[t * 65 + r];
                    if ((r & 3) == 0) a0 = fmaf(a, x[r], a0);
                    else if ((r & 3) == 1) a1 = fmaf(a, x[r], a1);
                    else if ((r & 3) == 2) a2 = fmaf(a, x[r], a2);
                    else a3 = fmaf(a, x[r], a3);
                }
                x[t] -= (a0 + a1) + (a2 + a3);
            }
            const float bs = bet[s], bgs = bet[s] * gam[s];
            const uint32_t off = (s & 7) * 2;
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                const uint32_t at = swz128(t, s >> 3) + off;
                *reinterpret_cast<__nv_bfloat16 *>(sm + L::TP + at) = __float2bfloat16_rn(x[t] * bgs);
                *reinterpret_cast<__nv_bfloat16 *>(sm + L::TPP + at) = __float2bfloat16_rn(x[t] * bs);
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- (4) W^T = K^T T'^T and U~^T = V^T T''^T ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma_bf16(tb + L::WT, sdesc(stg + L::KC0 + ks * 2048, 16384, 1024),
                         sdesc(base + L::TP + ks * 32, 16, 1024), I_AMN, ks > 0);
                mma_bf16(tb + L::UA, sdesc(stg + L::VC0 + ks * 2048, 8192, 1024),
                         sdesc(base + L::TPP + ks * 32, 16, 1024), I_AMN, ks > 0);
            }
            mma_commit(&bar_mma);
        }
        ok = wait_mma();
        if (ok && row < K) {
            float v[32];
            tmem_ld32(tb + lane_off + L::WT + half * 32, v);
            tmem_ld_wait();
            store_row32(sm + L::NW, row, half * 4, v, -1.f);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // ---- (5) U^T = U~^T - S W^T ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks) {
                const uint32_t kb = ks / 4, ko = (ks % 4) * 32;
                mma_bf16(tb + L::UA, sdesc(base + L::SB + kb * 16384 + ko, 16, 1024),
                         sdesc(base + L::NW + ks * 2048, 8192, 1024), I_BMN, 1);
            }
            mma_commit(&bar_mma);
        }
        ok = wait_mma();
        if (ok) {
            float v[32];
            tmem_ld32(tb + lane_off + L::UA + half * 32, v);
            tmem_ld_wait();
            store_row32(sm + L::UT, row, half * 4, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= dcy[half * 32 + i];
            store_row32(sm + L::UD, row, half * 4, v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // ---- (6) O_b^T = U^T P^T and dS = U^T diag(decay) K ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma_bf16(tb + L::OB, sdesc(base + L::UT + ks * 32, 16, 1024),
                         sdesc(base + L::PT + ks * 32, 16, 1024), I_MM, ks > 0);
                mma_bf16(tb + L::DS, sdesc(base + L::UD + ks * 32, 16, 1024),
                         sdesc(stg + L::KC0 + ks * 2048, 16384, 1024), I_DS, ks > 0);
            }
            mma_commit(&bar_mma);
        }
        ok = wait_mma();
        if (ok) {
            // state: S <- gamma_C S + dS, then its bf16 copy for the next chunk
            const float gC = gam[63];
            const int j0 = half * KH;
#pragma unroll
            for (int p = 0; p < KH / 32; ++p) {
                float v[32];
                tmem_ld32(tb + lane_off + L::DS + j0 + 32 * p, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    S[32 * p + i] = fmaf(gC, S[32 * p + i], v[i]);
                    v[i] = S[32 * p + i];
                }
                const int j = j0 + 32 * p;
                store_row32(sm + L::SB + (j / 64) * 16384, row, (j % 64) / 8, v);
            }
            // output: o[t][c] = gamma_t (S Q^T)[c][t] + (U^T P^T)[c][t]
            float oa[32], ob[32];
            tmem_ld32(tb + lane_off + L::OA + half * 32, oa);
            tmem_ld32(tb + lane_off + L::OB + half * 32, ob);
            tmem_ld_wait();
            __nv_bfloat16 *orow = o + (((size_t)b * T + c0) * H + h) * V + row;
            const size_t tstride = (size_t)H * V;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int t = half * 32 + i;
                if (o != nullptr && t < nvalid)
                    orow[t * tstride] = __float2bfloat16_rn(fmaf(gam[t], oa[i], ob[i]));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        // this stage's tiles are consumed: prefetch chunk n + 2 into it
        if (tid == 0 && n + 2 < nchunks) issue_loads(n + 2);
    }

    if (failed) {
        if (tid == 0 && status) atomicOr(status, kStatusTimeout);
        // let in-flight loads land before the CTA's shared memory is released
        if (tid == 0) {
            for (int s = 0; s < 2; ++s) {
                // a stage with an outstanding load has had more arrivals issued than waited;
                // bounded waits on both parities cover it
                mbar_wait(&bar_full[s], 0, kSpinLimit / 8);
                mbar_wait(&bar_full[s], 1, kSpinLimit / 8);
            }
        }
    } else if (ST != nullptr) {
        const int j0 = half * KH;
#pragma unroll
        for (int j = 0; j < KH; j += 4)
            *reinterpret_cast<float4 *>(ST + (seq * V + row) * K + j0 + j) =
                make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [B, T, H, C] bf16 tensor viewed as 4-D (C, H, T, B) with 64 x 1 x 64 x 1 boxes.
bool make_token_map(CUtensorMap *m, const void *ptr, int B, int T, int H, int C) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)C * 2 * H,
                             (cuuint64_t)C * 2 * H * T};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int K>
cudaError_t launch_tc_t(const void *q, const void *k, const void *v, const float *alpha,
                        const float *beta, const float *S0, void *o, float *ST, int B, int T,
                        int H, cudaStream_t stream) {
    CUtensorMap mq, mk, mv;
    if (!make_token_map(&mq, q, B, T, H, K) || !make_token_map(&mk, k, B, T, H, K) ||
        !make_token_map(&mv, v, B, T, H, 128))
        return cudaErrorInvalidValue;
    auto kern = prefill_tc_kernel<K>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)TcLayout<K>::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const long long grid = (long long)B * H;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, kTcThreads, TcLayout<K>::SMEM, stream>>>(
        mq, mk, mv, alpha, beta, S0, static_cast<__nv_bfloat16 *>(o), ST, T, H,
        device_status_ptr());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *ST, int B,
                              int T, int H, int K, int V, cudaStream_t stream) {
    if (V != 128) return cudaErrorInvalidValue;
    if (K == 128) return launch_tc_t<128>(q, k, v, alpha, beta, S0, o, ST, B, T, H, stream);
    if (K == 64) return launch_tc_t<64>(q, k, v, alpha, beta, S0, o, ST, B, T, H, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
