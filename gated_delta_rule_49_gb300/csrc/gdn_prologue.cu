// Pruning prologue: keep d_k' of the d_k key/query channels of every head and
// recompute the L2 normalisation on the kept coordinates ("On State Reduction
// in Linear Attention" notes, Sec. 2.6 and Alg. 1):
//
//     y[n, h, :] = x[n, h, idx[h, :]] / max(|x[n, h, idx[h, :]]|, eps)
//
// Memory-bound.  A random half of a row's channels touches every 32-byte
// sector of it, so the row is read whole: the staged kernel moves a warp's
// tile of consecutive rows (one contiguous block of up to 4 KB) with one TMA
// bulk copy into the warp's two-slot ring (the next tile in flight while one
// is gathered; 64 KB per CTA keeps three CTAs per SM) and gathers the kept
// channels from shared memory; each output
// row is written by K_out/8 lanes with one 16-byte (bf16) or 32-byte (fp32)
// store per lane.  Rows whose byte width is not a multiple of 16 take the
// row-wise kernel (a warp per row, channel loads straight from global memory).
// An index outside [0, K_in) is not read in either: it contributes 0 and sets
// the device status's bounds bit.
#include "gdn_internal.cuh"
#include "gdn_sm100.cuh"

namespace gdn {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kTileBytes = 4096;                  // per warp and slot
constexpr int kBulkStages = 2;                    // slots per warp
constexpr int kStagedWarps = 8;
constexpr long long kBulkSpin = 2000000000LL;     // ~1 s of SM clocks per wait
constexpr size_t kStagedSmem =
    (size_t)kStagedWarps * kBulkStages * kTileBytes + kStagedWarps * kBulkStages * 8;

template <typename T, int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ void store8(__nv_bfloat16 *dst, const float *g, float inv) {
    uint4 w;
    unsigned *u = reinterpret_cast<unsigned *>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(g[2 * e] * inv, g[2 * e + 1] * inv);
        u[e] = *reinterpret_cast<const unsigned *>(&b);
    }
    *reinterpret_cast<uint4 *>(dst) = w;
}
__device__ __forceinline__ void store8(float *dst, const float *g, float inv) {
    reinterpret_cast<float4 *>(dst)[0] = make_float4(g[0] * inv, g[1] * inv, g[2] * inv, g[3] * inv);
    reinterpret_cast<float4 *>(dst)[1] = make_float4(g[4] * inv, g[5] * inv, g[6] * inv, g[7] * inv);
}

// rows_per_tile = floor(4096 / row bytes) >= 1 consecutive rows per warp tile;
// row bytes (K_in * sizeof(T)) is a multiple of 16 and at most 4096, so a
// tile is one contiguous, 16-byte aligned block: lane 0 of each warp fetches
// it with one bulk copy into the warp's ring of kBulkStages slots, completing
// on the slot's mbarrier (every wait bounded).
template <typename T, int KOUT>
__global__ void __launch_bounds__(kStagedWarps * 32)
    gather_normalize_staged(const T *__restrict__ x, const int *__restrict__ idx,
                            T *__restrict__ y, long long rows, int H, int Kin, int rows_per_tile,
                            float eps, int *status) {
    constexpr int OPL = 8;            // outputs per lane
    constexpr int LPR = KOUT / OPL;   // lanes per output row
    constexpr int RPP = 32 / LPR;     // rows per gather pass
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint8_t *mine = smem + (size_t)warp * kBulkStages * kTileBytes;
    uint64_t *mb = reinterpret_cast<uint64_t *>(smem + kStagedWarps * kBulkStages * kTileBytes) +
                   warp * kBulkStages;
    if (lane == 0) {
        for (int s = 0; s < kBulkStages; ++s) sm100::mbar_init(&mb[s], 1);
        sm100::fence_mbar_init();
    }
    __syncwarp();
    const long long row_bytes = (long long)Kin * (long long)sizeof(T);
    const int sub = lane / LPR, cl = lane % LPR;
    const long long ntiles = (rows + rows_per_tile - 1) / rows_per_tile;
    const long long gw = (long long)blockIdx.x * kStagedWarps + warp;
    const long long nw = (long long)gridDim.x * kStagedWarps;
    const long long my_n = gw < ntiles ? (ntiles - gw + nw - 1) / nw : 0;  // this warp's tiles
    auto issue = [&](long long i) {  // lane 0: tile gw + i nw into slot i mod kBulkStages
        const long long r0 = (gw + i * nw) * rows_per_tile;
        const long long nrows = min((long long)rows_per_tile, rows - r0);
        const uint32_t bytes = (uint32_t)(nrows * row_bytes);
        uint64_t *bar = &mb[i % kBulkStages];
        sm100::fence_proxy_async_smem();  // earlier generic reads of the slot come first
        sm100::mbar_arrive_expect_tx(bar, bytes);
        sm100::bulk_load(mine + (i % kBulkStages) * kTileBytes, x + r0 * Kin, bytes, bar);
    };
    if (lane == 0)
        for (long long i = 0; i < my_n && i < kBulkStages; ++i) issue(i);
    bool bad = false, ok = true;
    long long i = 0;
    for (; i < my_n; ++i) {
        const int slot = (int)(i % kBulkStages);
        if (!sm100::mbar_wait(&mb[slot], (uint32_t)((i / kBulkStages) & 1), kBulkSpin)) {
            ok = false;
            break;
        }
        const T *ts = reinterpret_cast<const T *>(mine + slot * kTileBytes);
        const long long r0 = (gw + i * nw) * rows_per_tile;
        const int nrows = (int)min((long long)rows_per_tile, rows - r0);
        const int npass = (nrows + RPP - 1) / RPP;
        for (int p = 0; p < npass; ++p) {
            const int rr = p * RPP + sub;
            const bool valid = rr < nrows;
            float g[OPL];
            float ss = 0.f;
            if (valid) {
                const int h = (int)((r0 + rr) % H);
                const int4 *ip = reinterpret_cast<const int4 *>(idx + (size_t)h * KOUT) + 2 * cl;
                const int4 i0 = __ldg(ip), i1 = __ldg(ip + 1);
                const int c[OPL] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
                for (int e = 0; e < OPL; ++e) {
                    if ((unsigned)c[e] < (unsigned)Kin) {
                        g[e] = to_f32(ts[rr * Kin + c[e]]);
                    } else {
                        g[e] = 0.f;
                        bad = true;
                    }
                    ss = fmaf(g[e], g[e], ss);
                }
            } else {
#pragma unroll
                for (int e = 0; e < OPL; ++e) g[e] = 0.f;
            }
            ss = group_sum<T, LPR>(ss);
            const float inv = 1.f / fmaxf(sqrtf(ss), eps);
            if (valid) store8(y + (r0 + rr) * KOUT + cl * OPL, g, inv);
        }
        __syncwarp();  // every lane is done with this slot
        if (lane == 0 && i + kBulkStages < my_n) issue(i + kBulkStages);
    }
    if (!ok) {
        if (lane == 0 && status) atomicOr(status, kStatusTimeout);
        // copies still in flight must land before the CTA's shared memory goes away
        for (long long j = i; j < my_n && j < i + kBulkStages; ++j)
            sm100::mbar_wait(&mb[j % kBulkStages], (uint32_t)((j / kBulkStages) & 1), kBulkSpin);
    }
    if (bad && status) atomicOr(status, kStatusBounds);
}

template <typename T, int KOUT>
__global__ void __launch_bounds__(256)
    gather_normalize_kernel(const T *__restrict__ x, const int *__restrict__ idx,
                            T *__restrict__ y, long long rows, int H, int Kin, float eps,
                            int *status) {
    constexpr int PER = KOUT / 32;
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    bool bad = false;
    for (long long r0 = gw * kRowsPerWarp; r0 < rows; r0 += nw * kRowsPerWarp) {
        float v[kRowsPerWarp][PER];
        float ss[kRowsPerWarp];
#pragma unroll
        for (int u = 0; u < kRowsPerWarp; ++u) {
            const long long row = r0 + u;
            ss[u] = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                float val = 0.f;
                if (row < rows) {
                    const int h = (int)(row % H);
                    const int c = idx[h * KOUT + lane * PER + e];
                    if ((unsigned)c < (unsigned)Kin)
                        val = to_f32(x[row * Kin + c]);
                    else
                        bad = true;
                }
                v[u][e] = val;
                ss[u] = fmaf(val, val, ss[u]);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int u = 0; u < kRowsPerWarp; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], off);
#pragma unroll
        for (int u = 0; u < kRowsPerWarp; ++u) {
            const long long row = r0 + u;
            if (row >= rows) break;
            const float inv = 1.f / fmaxf(sqrtf(ss[u]), eps);
#pragma unroll
            for (int e = 0; e < PER; ++e)
                y[row * KOUT + lane * PER + e] = from_f32<T>(v[u][e] * inv);
        }
    }
    if (bad && status) atomicOr(status, kStatusBounds);
}

template <typename T, int KOUT>
cudaError_t launch_gn_t(const void *x, const int *idx, void *y, long long rows, int H, int Kin,
                        float eps, cudaStream_t stream) {
    const long long sms = sm_count() > 0 ? sm_count() : 152;
    const int row_bytes = Kin * (int)sizeof(T);
    if (row_bytes % 16 == 0 && row_bytes <= kTileBytes) {
        const int rpt = kTileBytes / row_bytes;
        const long long tiles = (rows + rpt - 1) / rpt;
        long long blocks = (tiles + kStagedWarps - 1) / kStagedWarps;
        if (blocks > sms * 3) blocks = sms * 3;  // 64 KB of slots: three CTAs per SM
        if (blocks < 1) blocks = 1;
        auto kern = gather_normalize_staged<T, KOUT>;
        static uintptr_t attr_set[64] = {};  // context the attributes were set in
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            return cudaErrorInvalidDevice;
        if (attr_set[dev] != context_key()) {
            const cudaError_t e = cudaFuncSetAttribute(
                kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStagedSmem);
            if (e != cudaSuccess) return e;
            attr_set[dev] = context_key();
        }
        kern<<<(unsigned)blocks, kStagedWarps * 32, kStagedSmem, stream>>>(
            static_cast<const T *>(x), idx, static_cast<T *>(y), rows, H, Kin, rpt, eps,
            device_status_ptr());
        return cudaGetLastError();
    }
    const long long warps = (rows + kRowsPerWarp - 1) / kRowsPerWarp;
    long long blocks = (warps + 7) / 8;
    if (blocks > sms * 16) blocks = sms * 16;
    if (blocks < 1) blocks = 1;
    gather_normalize_kernel<T, KOUT><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const T *>(x), idx, static_cast<T *>(y), rows, H, Kin, eps,
        device_status_ptr());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_normalize(const void *x, const int *idx, void *y, long long rows,
                                    int H, int Kin, int Kout, gdn_dtype dt, float eps,
                                    cudaStream_t stream) {
    const bool bf = dt == GDN_BF16;
    if (Kout == 64)
        return bf ? launch_gn_t<__nv_bfloat16, 64>(x, idx, y, rows, H, Kin, eps, stream)
                  : launch_gn_t<float, 64>(x, idx, y, rows, H, Kin, eps, stream);
    if (Kout == 32)
        return bf ? launch_gn_t<__nv_bfloat16, 32>(x, idx, y, rows, H, Kin, eps, stream)
                  : launch_gn_t<float, 32>(x, idx, y, rows, H, Kin, eps, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gdn
