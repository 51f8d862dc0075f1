// Internal declarations shared by the translation units of libgdn.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "gdn.h"

namespace gdn {

// Bits of the per-device status word (see gdn_get_last_device_status).
enum : int {
    kStatusTimeout = 1,
    kStatusBounds = 2,
    kStatusZeroState = 4,
    kStatusNotConverged = 8,
    kStatusRankDeficient = 16
};

// Chunk length of the chunkwise prefill.
constexpr int kChunk = 64;

// Debug builds (-DGDN_BOUNDS_CHECK) check the indices and coordinates the
// prefill kernels derive (segment ranges, TMA box coordinates, key-side block
// offsets, gate and gathered-row offsets) before using them: a failed check
// sets the bounds bit of the device status and the access is skipped (a
// skipped load then leaves its bounded wait to run out, so the call ends with
// the timeout bit as well).  Release builds compile every check away.
__device__ __forceinline__ bool bounds_ok(bool cond, int *status) {
#ifdef GDN_BOUNDS_CHECK
    if (!cond && status) atomicOr(status, kStatusBounds);
    return cond;
#else
    (void)cond;
    (void)status;
    return true;
#endif
}

// Address of the current device's status word (nullptr if the symbol lookup
// failed).  Kernels OR their bits into it.
int *device_status_ptr();

// Streaming multiprocessor count of the current device (cached).
int sm_count();

// Identifies the CUDA context current on the calling thread (0 if none is
// current yet).  Per-device caches of symbol addresses, kernel attributes,
// streams and events remember the context they were made in and are redone
// when another context is current (e.g. after cudaDeviceReset).
uintptr_t context_key();

// --- launchers (return the launch error, never synchronise) ---------------
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *alpha,
                          const float *beta, float *S, void *o, int B, int H, int K, int V,
                          gdn_dtype dt, cudaStream_t stream);

cudaError_t launch_state_rank(const float *S, int BH, int V, int K, float *fro2,
                              float *sigma1, float *er, int max_iter, float tol,
                              cudaStream_t stream);


// Tensor-core (tcgen05) chunked prefill: bf16 q/k/v, V = 128, K in {64, 128}.
// Long sequences on few heads run segment-parallel and need `workspace`.
//
// Processes tokens [0, T) of token tensors laid out as [B, Ts, H, *]
// (Ts >= T tokens per batch entry; alpha/beta [B, Ts, H]): Ts = T for a whole
// tensor, Ts > T for a window of a longer one.
cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *S0, void *o, float *ST, int B,
                              int T, int Ts, int H, int K, int V, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

// How the tensor-core prefill splits B*H sequences of T tokens into segments
// on a device with `nsm` SMs (nseg == 1: one CTA per whole sequence).
struct SegShape {
    int nseg;
    int seg_len;
    size_t workspace_bytes;
};
SegShape segment_shape(int BH, int T, int K, int nsm);

// Two-pass form of the tensor-core prefill: a key-side pass writes T', T'' and
// P of every chunk (prefill_prep_bytes) at byte offset prefill_prep_offset of
// the workspace, after the segment slots; launch_prefill_tc takes this form
// whenever workspace_bytes >= offset + bytes.
size_t prefill_prep_offset(const SegShape &sh);
size_t prefill_prep_bytes(long long BH, int T);
// Segment-parallel problems: the X buffer ([B, T, H, 128] bf16) right after
// the key-side operands, with which the two-pass form needs no second pass
// over the segments (0 for whole sequences).
size_t prefill_x_bytes(const SegShape &sh, long long BH, int T);

// The two-pass prefill from full-width q/k (K_in = 128) on a state pruned to
// 64 channels: the pruning prologue runs inside the key-side pass.  Workspace
// byte offsets of its parts (segment slots first, at 0).
struct GatheredLayout {
    size_t prep, qg, kg, x, total;  // x: the segments' X buffer (empty for whole sequences)
};
GatheredLayout gathered_layout(int B, int T, int H);
cudaError_t launch_prefill_gathered(const void *q_full, const void *k_full, const int *idx,
                                    const void *v, const float *alpha, const float *beta,
                                    const float *S0, void *o, float *ST, int B, int T, int H,
                                    void *workspace, size_t workspace_bytes, cudaStream_t stream);

// Pruning prologue: gather K_out of K_in channels per head and L2-normalise.
cudaError_t launch_gather_normalize(const void *x, const int *idx, void *y, long long rows,
                                    int H, int Kin, int Kout, gdn_dtype dt, float eps,
                                    cudaStream_t stream);

// Decode step reading full-width q/k and gathering + renormalising the kept
// channels in the kernel (idx [H, K], K_in the full width).
cudaError_t launch_decode_gathered(const void *q, const void *k, const int *idx, int Kin,
                                   const void *v, const float *alpha, const float *beta,
                                   float *S, void *o, int B, int H, int K, int V, gdn_dtype dt,
                                   float eps, cudaStream_t stream);

// Channel-gated rules (GDN / KDA / GDN2), token by token on the CUDA cores;
// also the prefill for float32 inputs and the (32, 32) variant (scalar gate).
// Tokens [0, T) of [B, Ts, H, *] tensors, as for the chunked prefill.
// The chunkwise tensor-core prefill of KDA / GDN2 (K = V = 128, bf16;
// gdn_gated_tc.cu): workspace bytes, and the two launches.
size_t prefill_gated_tc_workspace(int B, int T, int H, int gate);
cudaError_t launch_prefill_gated_tc(const void *q, const void *k, const void *v,
                                    const float *alpha, const float *beta, const float *bgate,
                                    const float *wgate, const float *S0, void *o, float *ST,
                                    int B, int T, int H, int gate, void *workspace,
                                    cudaStream_t stream);
cudaError_t launch_prefill_gated(const void *q, const void *k, const void *v,
                                 const float *alpha, const float *beta, const float *bg,
                                 const float *wg, const float *S0, void *o, float *ST, int B,
                                 int T, int Ts, int H, int K, int V, gdn_gate gate, gdn_dtype dt,
                                 cudaStream_t stream);
cudaError_t launch_decode_gated(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *bg, const float *wg, float *S,
                                void *o, int B, int H, int K, int V, gdn_gate gate, gdn_dtype dt,
                                cudaStream_t stream);

// Rank-r truncation (and singular values) of BH states [V, K] by one-sided Jacobi.
cudaError_t launch_state_truncate(float *S, int BH, int V, int K, int r, float *sigma,
                                  int max_sweeps, cudaStream_t stream);

// DRRQR channel selection: calibration Gram on the tensor cores (K = 128,
// bf16; workspace H * gram_splits * 64 KiB) and the per-head selection.
int gram_splits(int B, int T, int H);
cudaError_t launch_channel_gram(const void *k, const void *q, int B, int T, int H, float *G,
                                void *workspace, cudaStream_t stream);
size_t drrqr_select_smem(int n, int k);
cudaError_t launch_drrqr_select(const float *G, int H, int n, int k, float f, int max_swaps,
                                int *idx, float *rho, int *swaps, cudaStream_t stream);

// Prefill on host buffers, pipelined over windows of `window` tokens: byte
// offsets of one window slot's device buffers (two slots), the float32 state
// and the segment scratch inside the caller's device workspace.
struct HostLayout {
    size_t q, k, v, a, b, o, slot, state, seg, seg_bytes, total;
};
HostLayout host_layout(int B, int T, int H, int K, int V, gdn_dtype dt, int window);
cudaError_t launch_prefill_host(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *S0, void *o, float *ST, int B,
                                int T, int H, int K, int V, gdn_dtype dt, int window,
                                void *workspace, cudaStream_t stream);

// Programmatic dependent launch: a kernel launched this way may be scheduled
// while the previous kernel on the stream finishes; it must execute
// pdl_wait() before its first global-memory access (which then sees all of
// the previous kernel's writes) and may call pdl_trigger() to let its own
// successor be scheduled early.  (Used by the plain decode step.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Loads of the run dtype as float.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

}  // namespace gdn
