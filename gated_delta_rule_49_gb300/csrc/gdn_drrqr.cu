// DRRQR channel selection ("On State Reduction in Linear Attention" notes,
// Sec. 2.8): choose d_k' of the d_k key/query channels of every head so that
// the kept columns of the calibration matrix M = [K_cal; Q_cal] form a
// well-conditioned basis.
//
// 1. Gram (tensor cores).  Only R of a QR of M is needed, and R^T R = M^T M,
//    so the bulk work is G_h = K_h^T K_h + Q_h^T Q_h over all calibration
//    tokens: a contraction over tokens with both operands the same token-major
//    bf16 tiles read as MN-major tcgen05 operands.  A CTA owns one head and a
//    contiguous range of 64-token chunks; one thread issues the TMA loads
//    (3-stage ring of 64-token x 128-channel k and q tiles; a stage is
//    refilled one chunk after its MMAs were issued, so they overlap) and the MMAs
//    (M = N = 128, the accumulator is a 128 x 128 float32 TMEM tile); the
//    four warps then write the partial Gram to a workspace slot and a second
//    kernel sums the slots in a fixed order (deterministic).  HBM-bound:
//    every calibration byte is read once.
//
// 2. Selection (CUDA cores, one CTA per head, float32 in shared memory).
//    Column-pivoted QR's permutation is the pivot order of the pivoted
//    Cholesky factorisation of G (largest remaining diagonal first, ties to
//    the lowest position, as LAPACK's geqp3 picks the largest remaining
//    column norm).  Then, as in the notes: R = chol(P^T G P) gives A_k, B_k,
//    C_k; U = A_k^{-1} B_k, omega_i = 1 / |row i of A_k^{-1}|, gamma_j =
//    |column j of C_k|, rho_ij = sqrt(U_ij^2 + (gamma_j / omega_i)^2); while
//    max rho > f swap kept column i with candidate j and refactor.  The kept
//    channels are the first k entries of the final permutation.
#include "gdn_internal.cuh"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

using namespace sm100;

constexpr int kGramStages = 3;  // 96 KB of tiles: two CTAs per SM
constexpr int kGramThreads = 128;
constexpr uint32_t kTile = 8192;                // 64 tokens x 64 channels bf16
constexpr uint32_t kStageBytes = 4 * kTile;     // k (2 boxes) + q (2 boxes)
constexpr long long kGramSpin = 2000000000LL;   // ~1 s of SM clocks per wait

struct GramSmem {
    static constexpr uint32_t BAR = kGramStages * kStageBytes;  // full[S], empty[S], done
    static constexpr uint32_t TMEM_SLOT = BAR + (2 * kGramStages + 1) * 8;
    static constexpr uint32_t BYTES = TMEM_SLOT + 16 + 1024;    // + alignment slack
};

// grid (splits, H); CTA (split, h) sums chunks [split * per, min(total, ...)).
__global__ void __launch_bounds__(kGramThreads)
    gram_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                float *__restrict__ partial, int T, int chunks_total, int chunks_per_split,
                int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + GramSmem::BAR);
    uint64_t *empty = full + kGramStages;
    uint64_t *done = empty + kGramStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + GramSmem::TMEM_SLOT);
    __shared__ int failed;

    const int split = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int c0 = split * chunks_per_split;
    const int c1 = min(chunks_total, c0 + chunks_per_split);
    const int n = max(0, c1 - c0);
    const int nct = (T + 63) / 64;  // chunks per batch entry

    if (tid == 0) {
        for (int s = 0; s < kGramStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
        failed = 0;
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tmem_slot;

    if (tid == 0) {
        auto load = [&](int i) {
            const int c = c0 + i, s = i % kGramStages;
            const int b = c / nct, t0 = (c % nct) * 64;
            uint8_t *st = sm + s * kStageBytes;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            tma_load_4d(st, &tm_k, &full[s], 0, h, t0, b);
            tma_load_4d(st + kTile, &tm_k, &full[s], 64, h, t0, b);
            tma_load_4d(st + 2 * kTile, &tm_q, &full[s], 0, h, t0, b);
            tma_load_4d(st + 3 * kTile, &tm_q, &full[s], 64, h, t0, b);
        };
        constexpr uint32_t I_G = idesc_bf16(128, 128, true, true);  // both MN-major
        int issued = 0;
        for (; issued < n && issued < kGramStages; ++issued) load(issued);
        bool ok = true;
        int i = 0;
        for (; i < n; ++i) {
            const int s = i % kGramStages;
            if (!mbar_wait(&full[s], (i / kGramStages) & 1, kGramSpin)) { ok = false; break; }
            tc_fence_after();
            const uint32_t st = smem_u32(sm + s * kStageBytes);
#pragma unroll
            for (int op = 0; op < 2; ++op)  // k then q
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t d = sdesc(st + op * 2 * kTile + ks * 2048, kTile, 1024);
                    mma_bf16(tb, d, d, I_G, (i > 0 || op > 0 || ks > 0) ? 1u : 0u);
                }
            mma_commit(&empty[s]);
            // refill the stage of chunk i - 1, whose MMAs were issued an iteration ago
            if (i >= 1 && issued < n) {
                const int ip = i - 1;
                if (!mbar_wait(&empty[ip % kGramStages], (ip / kGramStages) & 1, kGramSpin)) {
                    ok = false;
                    ++i;
                    break;
                }
                load(issued++);
            }
        }
        if (!ok) {
            failed = 1;
            if (status) atomicOr(status, kStatusTimeout);
            // loads still in flight must land before the CTA's shared memory goes away
            for (int j = i; j < issued; ++j)
                mbar_wait(&full[j % kGramStages], (j / kGramStages) & 1, kGramSpin);
        }
        // completes once every MMA issued above has finished (at once if none was)
        mma_commit(done);
    }
    __syncwarp();
    const bool got = mbar_wait(done, 0, kGramSpin);
    tc_fence_after();
    __syncthreads();
    if (!got && tid == 0 && status) atomicOr(status, kStatusTimeout);
    float *out = partial + ((size_t)h * gridDim.x + split) * 128 * 128;
    if (got && !failed && n > 0) {
        const int row = warp * 32 + (tid & 31);
#pragma unroll 1
        for (int cb = 0; cb < 128; cb += 32) {
            float v[32];
            tmem_ld32(tb + ((uint32_t)(warp * 32) << 16) + cb, v);
            tmem_ld_wait();
            float4 *dst = reinterpret_cast<float4 *>(out + (size_t)row * 128 + cb);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
    } else {
        for (int e = tid; e < 128 * 128; e += kGramThreads) out[e] = 0.f;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 128);
}

// G[h] = sum over splits of partial[h][split] (fixed order).
__global__ void gram_reduce_kernel(const float *__restrict__ partial, float *__restrict__ G,
                                   int splits) {
    const int h = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;  // < 128 * 128
    const float *p = partial + (size_t)h * splits * 128 * 128 + e;
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += p[(size_t)s * 128 * 128];
    G[(size_t)h * 128 * 128 + e] = acc;
}

// ---------------------------------------------------------------- selection

constexpr int kSelThreads = 256;

struct SelSmem {
    int n, k, ld;
    __host__ __device__ size_t gram() const { return 0; }
    __host__ __device__ size_t rfac() const { return gram() + (size_t)n * ld * 4; }
    __host__ __device__ size_t xinv() const { return rfac() + (size_t)n * ld * 4; }
    __host__ __device__ size_t vec() const { return xinv() + (size_t)k * ld * 4; }  // 4 n floats
    __host__ __device__ size_t bytes() const { return vec() + (size_t)4 * n * 4 + 64; }
};

// Largest value of v[i] over i in [lo, n) (ties: lowest i); all threads return it.
__device__ void block_argmax(float val, int idx, float *red_v, int *red_i, float &best,
                             int &bi) {
    // warp level
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, val, off);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
        if (ov > val || (ov == val && oi < idx)) { val = ov; idx = oi; }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { red_v[warp] = val; red_i[warp] = idx; }
    __syncthreads();
    if (warp == 0) {
        val = lane < kSelThreads / 32 ? red_v[lane] : -1.f;
        idx = lane < kSelThreads / 32 ? red_i[lane] : 0x7fffffff;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, val, off);
            const int oi = __shfl_xor_sync(0xffffffffu, idx, off);
            if (ov > val || (ov == val && oi < idx)) { val = ov; idx = oi; }
        }
        if (lane == 0) { red_v[0] = val; red_i[0] = idx; }
    }
    __syncthreads();
    best = red_v[0];
    bi = red_i[0];
    __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads)
    drrqr_select_kernel(const float *__restrict__ Gg, int n, int k, float f, int max_swaps,
                        int *__restrict__ idx_out, float *__restrict__ rho_out,
                        int *__restrict__ swaps_out, int *status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const SelSmem L{n, k, n + 1};
    const int ld = L.ld;
    float *G = reinterpret_cast<float *>(smem + L.gram());
    float *R = reinterpret_cast<float *>(smem + L.rfac());
    float *X = reinterpret_cast<float *>(smem + L.xinv());
    float *vec = reinterpret_cast<float *>(smem + L.vec());
    float *dres = vec;            // [n] residual diagonal (greedy phase)
    float *xn2 = vec + n;         // [k] |row i of A_k^{-1}|^2
    float *gam2 = vec + 2 * n;    // [n - k] |column j of C_k|^2
    __shared__ int perm[128];
    __shared__ float red_v[kSelThreads / 32];
    __shared__ int red_i[kSelThreads / 32];
    __shared__ int deficient;
    const int h = blockIdx.x, tid = threadIdx.x;
    const float *Gh = Gg + (size_t)h * n * n;
    for (int e = tid; e < n * n; e += kSelThreads) G[(e / n) * ld + e % n] = Gh[e];
    for (int i = tid; i < n; i += kSelThreads) perm[i] = i;
    if (tid == 0) deficient = 0;
    __syncthreads();
    float gmax = 0.f;
    for (int i = 0; i < n; ++i) gmax = fmaxf(gmax, G[i * ld + i]);
    // Pivots below 1e-6 of the largest diagonal (sigma below ~1e-3 sigma_1) are
    // float32 elimination noise of a Gram matrix: treated as zero.
    const float tiny = gmax * 1e-6f;

    // ---- greedy: pivoted Cholesky, first k pivots (R rows in position order) ----
    for (int i = tid; i < n; i += kSelThreads) dres[i] = G[i * ld + i];
    __syncthreads();
    for (int j = 0; j < k; ++j) {
        float best;
        int bpos;
        const float v = tid >= j && tid < n ? dres[perm[tid]] : -1.f;
        block_argmax(v, tid < n ? tid : 0x7fffffff, red_v, red_i, best, bpos);
        if (best <= tiny) {  // rank(M) < k: keep the greedy order, no swaps
            if (tid == 0) deficient = 1;
            break;
        }
        if (tid == 0 && bpos != j) {
            const int t = perm[j];
            perm[j] = perm[bpos];
            perm[bpos] = t;
        }
        if (tid < j && bpos != j) {  // swap the computed columns of rows < j
            const float t = R[tid * ld + j];
            R[tid * ld + j] = R[tid * ld + bpos];
            R[tid * ld + bpos] = t;
        }
        __syncthreads();
        const int pj = perm[j];
        const float rjj = sqrtf(dres[pj]);
        for (int pos = j + 1 + tid; pos < n; pos += kSelThreads) {
            const int i = perm[pos];
            float s = G[pj * ld + i];
            for (int l = 0; l < j; ++l) s = fmaf(-R[l * ld + j], R[l * ld + pos], s);
            const float r = s / rjj;
            R[j * ld + pos] = r;
            dres[i] -= r * r;
        }
        if (tid == 0) R[j * ld + j] = rjj;
        __syncthreads();
    }

    // ---- strong-RRQR swaps ----
    int swaps = 0;
    float rho_max = 0.f;
    const int m = n - k;
    while (!deficient) {
        // R = chol(P^T G P), all n columns
        for (int j = 0; j < n; ++j) {
            const int pj = perm[j];
            for (int pos = j + tid; pos < n; pos += kSelThreads) {
                float s = G[pj * ld + perm[pos]];
                for (int l = 0; l < j; ++l) s = fmaf(-R[l * ld + j], R[l * ld + pos], s);
                R[j * ld + pos] = s;
            }
            __syncthreads();
            const float d = R[j * ld + j];
            const float rjj = d > tiny ? sqrtf(d) : 0.f;  // trailing rank deficiency: C_k = 0
            __syncthreads();
            for (int pos = j + 1 + tid; pos < n; pos += kSelThreads)
                R[j * ld + pos] = rjj > 0.f ? R[j * ld + pos] / rjj : 0.f;
            if (tid == 0) R[j * ld + j] = rjj;
            __syncthreads();
        }
        // X = A_k^{-1} (upper triangular), one column per thread
        for (int c = tid; c < k; c += kSelThreads) {
            for (int i = c; i >= 0; --i) {
                float s = i == c ? 1.f : 0.f;
                for (int l = i + 1; l <= c; ++l) s = fmaf(-R[i * ld + l], X[l * ld + c], s);
                X[i * ld + c] = s / R[i * ld + i];
            }
            for (int i = c + 1; i < k; ++i) X[i * ld + c] = 0.f;
        }
        __syncthreads();
        for (int i = tid; i < k; i += kSelThreads) {
            float s = 0.f;
            for (int l = i; l < k; ++l) s = fmaf(X[i * ld + l], X[i * ld + l], s);
            xn2[i] = s;  // 1 / omega_i^2
        }
        for (int j = tid; j < m; j += kSelThreads) {
            float s = 0.f;
            for (int l = k; l <= k + j; ++l) s = fmaf(R[l * ld + k + j], R[l * ld + k + j], s);
            gam2[j] = s;
        }
        __syncthreads();
        // rho_ij^2 = (A_k^{-1} B_k)_ij^2 + gamma_j^2 / omega_i^2; arg max
        float best = -1.f;
        int bidx = 0x7fffffff;
        for (int e = tid; e < k * m; e += kSelThreads) {
            const int i = e / m, j = e % m;
            float u = 0.f;
            for (int l = i; l < k; ++l) u = fmaf(X[i * ld + l], R[l * ld + k + j], u);
            const float r2 = fmaf(u, u, gam2[j] * xn2[i]);
            if (r2 > best) { best = r2; bidx = e; }
        }
        float b2;
        int be;
        block_argmax(best, bidx, red_v, red_i, b2, be);
        rho_max = sqrtf(fmaxf(b2, 0.f));
        if (rho_max <= f || swaps >= max_swaps) break;
        if (tid == 0) {
            const int i = be / m, j = be % m;
            const int t = perm[i];
            perm[i] = perm[k + j];
            perm[k + j] = t;
        }
        ++swaps;
        __syncthreads();
    }
    if (tid == 0) {
        if (deficient && status) atomicOr(status, kStatusRankDeficient);
        if (rho_out) rho_out[h] = deficient ? 0.f : rho_max;
        if (swaps_out) swaps_out[h] = swaps;
    }
    for (int i = tid; i < k; i += kSelThreads) idx_out[(size_t)h * k + i] = perm[i];
}

}  // namespace

// Splits of each head's chunks over CTAs: about two CTAs per SM in all, and
// no split left empty (per = ceil(chunks / s), then s = ceil(chunks / per)).
int gram_splits(int B, int T, int H) {
    const long long chunks = (long long)B * ((T + 63) / 64);
    if (chunks < 1 || H < 1) return 1;
    const int sms = sm_count() > 0 ? sm_count() : 152;
    long long s = (2LL * sms + H - 1) / H;
    if (s > chunks) s = chunks;
    if (s < 1) s = 1;
    const long long per = (chunks + s - 1) / s;
    return (int)((chunks + per - 1) / per);
}

cudaError_t launch_channel_gram(const void *k, const void *q, int B, int T, int H, float *G,
                                void *workspace, cudaStream_t stream) {
    CUtensorMap mk, mq;
    if (!make_token_map(&mk, k, B, T, T, H, 128) || !make_token_map(&mq, q, B, T, T, H, 128))
        return cudaErrorInvalidValue;
    const int splits = gram_splits(B, T, H);
    const int chunks = B * ((T + 63) / 64);
    const int per = (chunks + splits - 1) / splits;
    static uintptr_t attr_set[64] = {};  // context the attributes were set in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (attr_set[dev] != context_key()) {
        const cudaError_t e = cudaFuncSetAttribute(
            gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)GramSmem::BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = context_key();
    }
    float *partial = static_cast<float *>(workspace);
    gram_kernel<<<dim3(splits, H), kGramThreads, GramSmem::BYTES, stream>>>(
        mk, mq, partial, T, chunks, per, device_status_ptr());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    gram_reduce_kernel<<<dim3(128 * 128 / 256, H), 256, 0, stream>>>(partial, G, splits);
    return cudaGetLastError();
}

size_t drrqr_select_smem(int n, int k) { return SelSmem{n, k, n + 1}.bytes(); }

cudaError_t launch_drrqr_select(const float *G, int H, int n, int k, float f, int max_swaps,
                                int *idx, float *rho, int *swaps, cudaStream_t stream) {
    const size_t bytes = drrqr_select_smem(n, k);
    const cudaError_t e = cudaFuncSetAttribute(
        drrqr_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    drrqr_select_kernel<<<H, kSelThreads, bytes, stream>>>(G, n, k, f, max_swaps, idx, rho,
                                                           swaps, device_status_ptr());
    return cudaGetLastError();
}

}  // namespace gdn
