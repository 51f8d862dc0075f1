// C ABI of libgdn.so: host-side validation and dispatch (declared in gdn.h).
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "gdn_internal.cuh"

namespace gdn {

// Per-device status word.  Kernels OR kStatus* bits into it; the host reads
// and clears it in gdn_get_last_device_status.
static __device__ int g_device_status;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_ptr[kMaxDevices];
uintptr_t g_status_ctx[kMaxDevices];  // the context g_status_ptr was looked up in
int g_sm_count[kMaxDevices];

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}
}  // namespace

uintptr_t context_key() {
    // the driver entry point is fetched through the runtime, so the library
    // keeps no link-time dependency on libcuda (it loads on machines without
    // a driver; nothing here runs there)
    using GetCurrent = CUresult (*)(CUcontext *);
    static GetCurrent fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<GetCurrent>(p);
    }();
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return 0;
    return reinterpret_cast<uintptr_t>(ctx);
}

int *device_status_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    const uintptr_t ctx = context_key();
    if (!g_status_ptr[dev] || ctx == 0 || g_status_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
        g_status_ctx[dev] = context_key();  // current now that the lookup ran
    }
    return g_status_ptr[dev];
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace gdn

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_kv(int K, int V) {
    return (K == 32 && V == 32) || (K == 64 && V == 128) || (K == 128 && V == 128);
}

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return GDN_OK;
    if (e == cudaErrorInvalidValue) return GDN_ERR_INVALID_ARG;
    return GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int gdn_version(void) { return 100; }

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported (K, V) variant or device";
        case GDN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case GDN_ERR_CUDA: return "CUDA runtime or launch error";
        case GDN_ERR_TIMEOUT: return "device wait timed out";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_DEVICE_BOUNDS: return "device-side index check failed";
        case GDN_WARN_ZERO_STATE: return "warning: all-zero state (stable rank undefined, 0 returned)";
        case GDN_WARN_NOT_CONVERGED: return "warning: Jacobi sweeps stopped at max_sweeps before convergence";
        case GDN_WARN_RANK_DEFICIENT: return "warning: calibration matrix has rank < k (greedy choice kept, no swaps)";
        default: return "unknown status";
    }
}

size_t gdn_prefill_workspace_size(int B, int T, int H, int K, int V, gdn_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || V != 128 || (K != 128 && K != 64) || dtype != GDN_BF16)
        return 0;
    if ((long long)B * H > 0x7fffffffLL) return 0;
    return gdn::segment_shape(B * H, T, K, gdn::sm_count()).workspace_bytes;
}

size_t gdn_prefill_two_pass_workspace_size(int B, int T, int H, int K, int V, gdn_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || V != 128 || (K != 128 && K != 64) || dtype != GDN_BF16)
        return 0;
    if ((long long)B * H > 0x7fffffffLL) return 0;
    const gdn::SegShape sh = gdn::segment_shape(B * H, T, K, gdn::sm_count());
    return gdn::prefill_prep_offset(sh) + gdn::prefill_prep_bytes((long long)B * H, T) +
           gdn::prefill_x_bytes(sh, (long long)B * H, T);
}

namespace {
// T = 0: the final state is the start state (or zero).
int empty_prefill(const float *S0, float *S_T, int B, int H, int K, int V, cudaStream_t st) {
    if (!S_T) return GDN_OK;
    const size_t bytes = sizeof(float) * (size_t)B * H * V * K;
    cudaError_t e = S0 ? (S0 == S_T ? cudaSuccess
                                    : cudaMemcpyAsync(S_T, S0, bytes, cudaMemcpyDeviceToDevice, st))
                       : cudaMemsetAsync(S_T, 0, bytes, st);
    return from_cuda(e);
}

// Which gate arrays a gate needs (non-NULL) and forbids (NULL).
bool gates_match(gdn_gate gate, const float *beta, const float *b, const float *w) {
    if (gate == GDN_GATE_GDN2) return !beta && b && w;
    return beta && !b && !w;
}
bool valid_gate(int gate) {
    return gate == GDN_GATE_SCALAR || gate == GDN_GATE_KDA || gate == GDN_GATE_GDN2;
}
}  // namespace

int gdn_prefill(const void *q, const void *k, const void *v, const float *alpha,
                const float *beta, const float *S0, void *o, float *S_T, int B, int T, int H,
                int K, int V, gdn_dtype dtype, void *workspace, size_t workspace_bytes,
                void *stream) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if (!o && !S_T) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !beta)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, alpha, beta, S0, o, S_T};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    const size_t need = gdn_prefill_workspace_size(B, T, H, K, V, dtype);
    if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
    if ((long long)B * H == 0) return GDN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return empty_prefill(S0, S_T, B, H, K, V, st);
    // bf16 at V = 128 runs on the tensor cores; float32 mode and the small
    // (32, 32) variant run the token-by-token CUDA-core kernel (scalar gate).
    if (dtype == GDN_BF16 && V == 128 && (K == 128 || K == 64))
        return from_cuda(gdn::launch_prefill_tc(q, k, v, alpha, beta, S0, o, S_T, B, T, T, H, K, V,
                                                workspace, workspace_bytes, st));
    return from_cuda(gdn::launch_prefill_gated(q, k, v, alpha, beta, nullptr, nullptr, S0, o, S_T,
                                               B, T, T, H, K, V, GDN_GATE_SCALAR, dtype, st));
}

size_t gdn_prefill_gathered_workspace_size(int B, int T, int H, int K_in, int K, int V,
                                           gdn_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || K_in != 128 || K != 64 || V != 128 || dtype != GDN_BF16)
        return 0;
    if ((long long)B * H > 0x7fffffffLL) return 0;
    return gdn::gathered_layout(B, T, H).total;
}

int gdn_prefill_gathered(const void *q_full, const void *k_full, const int *idx, int K_in,
                         const void *v, const float *alpha, const float *beta, const float *S0,
                         void *o, float *S_T, int B, int T, int H, int K, int V, gdn_dtype dtype,
                         void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0 || K_in <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 || K_in != 128 || K != 64 || V != 128) return GDN_ERR_UNSUPPORTED;
    if (!o && !S_T) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q_full || !k_full || !idx || !v || !alpha || !beta)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q_full, k_full, idx, v, alpha, beta, S0, o, S_T, workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    if ((long long)B * H == 0) return GDN_OK;
    if ((long long)B * H > 0x7fffffffLL) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return empty_prefill(S0, S_T, B, H, K, V, st);
    const size_t need = gdn_prefill_gathered_workspace_size(B, T, H, K_in, K, V, dtype);
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    return from_cuda(gdn::launch_prefill_gathered(q_full, k_full, idx, v, alpha, beta, S0, o, S_T,
                                                  B, T, H, workspace, workspace_bytes, st));
}

int gdn_decode_step(const void *q, const void *k, const void *v, const float *alpha,
                    const float *beta, float *S, void *o, int B, int H, int K, int V,
                    gdn_dtype dtype, void *stream) {
    if (B < 0 || H < 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H == 0) return GDN_OK;
    if (!q || !k || !v || !alpha || !beta || !S || !o) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, alpha, beta, S, o};
    for (const void *p : ptrs)
        if (!aligned16(p)) return GDN_ERR_ALIGNMENT;
    return from_cuda(gdn::launch_decode(q, k, v, alpha, beta, S, o, B, H, K, V, dtype,
                                        static_cast<cudaStream_t>(stream)));
}

int gdn_gather_normalize(const void *x, const int *idx, void *y, long long N, int H, int K_in,
                         int K_out, gdn_dtype dtype, void *stream) {
    if (N < 0 || H < 1 || (K_out != 32 && K_out != 64) || K_in < K_out || K_in > 1024)
        return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (N == 0) return GDN_OK;
    if (!x || !idx || !y) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {x, idx, y};
    for (const void *p : ptrs)
        if (!aligned16(p)) return GDN_ERR_ALIGNMENT;
    if (N > (1LL << 40) / H) return GDN_ERR_INVALID_ARG;
    return from_cuda(gdn::launch_gather_normalize(x, idx, y, N * H, H, K_in, K_out, dtype, 1e-12f,
                                                  static_cast<cudaStream_t>(stream)));
}

int gdn_decode_step_gathered(const void *q_full, const void *k_full, const int *idx, int K_in,
                             const void *v, const float *alpha, const float *beta, float *S,
                             void *o, int B, int H, int K, int V, gdn_dtype dtype, void *stream) {
    if (B < 0 || H < 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if (K_in < K || K_in > 1024) return GDN_ERR_INVALID_ARG;
    if ((long long)B * H == 0) return GDN_OK;
    if (!q_full || !k_full || !idx || !v || !alpha || !beta || !S || !o) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q_full, k_full, idx, v, alpha, beta, S, o};
    for (const void *p : ptrs)
        if (!aligned16(p)) return GDN_ERR_ALIGNMENT;
    return from_cuda(gdn::launch_decode_gathered(q_full, k_full, idx, K_in, v, alpha, beta, S, o,
                                                 B, H, K, V, dtype, 1e-12f,
                                                 static_cast<cudaStream_t>(stream)));
}

int gdn_prefill_gated(const void *q, const void *k, const void *v, const float *alpha,
                      const float *beta, const float *b, const float *w, const float *S0,
                      void *o, float *S_T, int B, int T, int H, int K, int V, gdn_gate gate,
                      gdn_dtype dtype, void *stream) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!valid_gate(gate)) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if (!o && !S_T) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !gates_match(gate, beta, b, w)))
        return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, alpha, beta, b, w, S0, o, S_T};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    if ((long long)B * H == 0) return GDN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return empty_prefill(S0, S_T, B, H, K, V, st);
    return from_cuda(gdn::launch_prefill_gated(q, k, v, alpha, beta, b, w, S0, o, S_T, B, T, T,
                                               H, K, V, gate, dtype, st));
}

size_t gdn_prefill_gated_chunked_workspace_size(int B, int T, int H, int K, int V,
                                                gdn_gate gate, gdn_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || K != 128 || V != 128 || dtype != GDN_BF16) return 0;
    if (gate != GDN_GATE_KDA && gate != GDN_GATE_GDN2) return 0;
    if ((long long)B * H > 0x7fffffffLL) return 0;
    return gdn::prefill_gated_tc_workspace(B, T, H, gate);
}

int gdn_prefill_gated_chunked(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *b, const float *w, const float *S0,
                              void *o, float *S_T, int B, int T, int H, int K, int V,
                              gdn_gate gate, gdn_dtype dtype, void *workspace,
                              size_t workspace_bytes, void *stream) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!valid_gate(gate)) return GDN_ERR_INVALID_ARG;
    if (gate == GDN_GATE_SCALAR || dtype != GDN_BF16 || K != 128 || V != 128)
        return GDN_ERR_UNSUPPORTED;
    if (!o && !S_T) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !gates_match(gate, beta, b, w)))
        return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, alpha, beta, b, w, S0, o, S_T, workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    if ((long long)B * H == 0) return GDN_OK;
    if ((long long)B * H > 0x7fffffffLL) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return empty_prefill(S0, S_T, B, H, K, V, st);
    const size_t need = gdn_prefill_gated_chunked_workspace_size(B, T, H, K, V, gate, dtype);
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    return from_cuda(gdn::launch_prefill_gated_tc(q, k, v, alpha, beta, b, w, S0, o, S_T, B, T, H,
                                                  gate, workspace, st));
}

int gdn_decode_step_gated(const void *q, const void *k, const void *v, const float *alpha,
                          const float *beta, const float *b, const float *w, float *S, void *o,
                          int B, int H, int K, int V, gdn_gate gate, gdn_dtype dtype,
                          void *stream) {
    if (B < 0 || H < 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!valid_gate(gate)) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if ((long long)B * H == 0) return GDN_OK;
    if (!q || !k || !v || !alpha || !S || !o || !gates_match(gate, beta, b, w))
        return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, alpha, beta, b, w, S, o};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    if ((long long)B * H > 0x7fffffffLL) return GDN_ERR_INVALID_ARG;
    return from_cuda(gdn::launch_decode_gated(q, k, v, alpha, beta, b, w, S, o, B, H, K, V, gate,
                                              dtype, static_cast<cudaStream_t>(stream)));
}

int gdn_state_truncate(float *S, int BH, int V, int K, int r, float *sigma, int max_sweeps,
                       void *stream) {
    if (BH < 0 || r < 1 || max_sweeps < 1 || max_sweeps > 1000) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if (BH == 0) return GDN_OK;
    if (!S) return GDN_ERR_INVALID_ARG;
    if (!aligned16(S) || (sigma && !aligned16(sigma))) return GDN_ERR_ALIGNMENT;
    if (r >= (K < V ? K : V) && !sigma) return GDN_OK;  // nothing to cut, nothing asked
    return from_cuda(gdn::launch_state_truncate(S, BH, V, K, r, sigma, max_sweeps,
                                                static_cast<cudaStream_t>(stream)));
}

int gdn_prefill_truncated(const void *q, const void *k, const void *v, const float *alpha,
                          const float *beta, const float *S0, void *o, float *S_T, int B, int T,
                          int H, int K, int V, gdn_dtype dtype, int seg_len, int r,
                          int max_sweeps, void *workspace, size_t workspace_bytes,
                          void *stream) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if (seg_len < 1 || r < 1 || max_sweeps < 1 || max_sweeps > 1000) return GDN_ERR_INVALID_ARG;
    if (!S_T) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !beta)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, alpha, beta, S0, o, S_T};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    // windows are seg_len tokens long, the last one possibly shorter
    const int L = seg_len < T ? seg_len : T, tail = T % seg_len;
    size_t need = gdn_prefill_workspace_size(B, L, H, K, V, dtype);
    if (tail > 0) {
        const size_t need_tail = gdn_prefill_workspace_size(B, tail, H, K, V, dtype);
        if (need_tail > need) need = need_tail;
    }
    if (need > 0 && (!workspace || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
    if ((long long)B * H == 0) return GDN_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) return empty_prefill(S0, S_T, B, H, K, V, st);
    const size_t esz = dtype == GDN_BF16 ? 2 : 4;
    const bool tc = dtype == GDN_BF16 && V == 128 && (K == 128 || K == 64);
    const float *start = S0;
    for (int t0 = 0; t0 < T; t0 += seg_len) {
        const int n = T - t0 < seg_len ? T - t0 : seg_len;
        const size_t tok = (size_t)t0 * H;  // token-head offset of the window
        const char *qw = static_cast<const char *>(q) + tok * K * esz;
        const char *kw = static_cast<const char *>(k) + tok * K * esz;
        const char *vw = static_cast<const char *>(v) + tok * V * esz;
        char *ow = o ? static_cast<char *>(o) + tok * V * esz : nullptr;
        cudaError_t e = tc ? gdn::launch_prefill_tc(qw, kw, vw, alpha + tok, beta + tok, start, ow,
                                                    S_T, B, n, T, H, K, V, workspace,
                                                    workspace_bytes, st)
                           : gdn::launch_prefill_gated(qw, kw, vw, alpha + tok, beta + tok,
                                                       nullptr, nullptr, start, ow, S_T, B, n, T,
                                                       H, K, V, GDN_GATE_SCALAR, dtype, st);
        if (e != cudaSuccess) return from_cuda(e);
        start = S_T;
        if (t0 + n < T && r < (K < V ? K : V)) {
            e = gdn::launch_state_truncate(S_T, B * H, V, K, r, nullptr, max_sweeps, st);
            if (e != cudaSuccess) return from_cuda(e);
        }
    }
    return GDN_OK;
}

size_t gdn_channel_gram_workspace_size(int B, int T, int H, int K) {
    if (B <= 0 || T <= 0 || H <= 0 || K != 128) return 0;
    return (size_t)H * gdn::gram_splits(B, T, H) * 128 * 128 * sizeof(float);
}

int gdn_channel_gram(const void *k, const void *q, int B, int T, int H, int K, gdn_dtype dtype,
                     float *G, void *workspace, size_t workspace_bytes, void *stream) {
    if (B < 0 || T < 0 || H < 0) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (K != 128 || dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (H == 0) return GDN_OK;
    if (!G) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((long long)B * T == 0)
        return from_cuda(cudaMemsetAsync(G, 0, sizeof(float) * (size_t)H * K * K, st));
    if (!k || !q) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {k, q, G, workspace};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    if ((long long)B * ((T + 63) / 64) > 0x7fffffffLL || H > 65535) return GDN_ERR_INVALID_ARG;
    const size_t need = gdn_channel_gram_workspace_size(B, T, H, K);
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    return from_cuda(gdn::launch_channel_gram(k, q, B, T, H, G, workspace, st));
}

int gdn_drrqr_select(const float *G, int H, int n, int k, float f, int max_swaps, int *idx,
                     float *rho_max, int *swaps, void *stream) {
    if (H < 0 || n < 2 || n > 128 || k < 1 || k >= n) return GDN_ERR_INVALID_ARG;
    if (!(f >= 1.f) || !(f < 3.0e38f) || max_swaps < 0 || max_swaps > 100000)
        return GDN_ERR_INVALID_ARG;
    if (H == 0) return GDN_OK;
    if (!G || !idx) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {G, idx, rho_max, swaps};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_ALIGNMENT;
    return from_cuda(gdn::launch_drrqr_select(G, H, n, k, f, max_swaps, idx, rho_max, swaps,
                                              static_cast<cudaStream_t>(stream)));
}

size_t gdn_prefill_host_workspace_size(int B, int T, int H, int K, int V, gdn_dtype dtype,
                                       int window) {
    if (B <= 0 || T < 0 || H <= 0 || window < 1 || !supported_kv(K, V)) return 0;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return 0;
    if ((long long)B * H > 0x7fffffffLL) return 0;
    return gdn::host_layout(B, T, H, K, V, dtype, window).total;
}

int gdn_prefill_host(const void *q, const void *k, const void *v, const float *alpha,
                     const float *beta, const float *S0, void *o, float *S_T, int B, int T, int H,
                     int K, int V, gdn_dtype dtype, int window, void *workspace,
                     size_t workspace_bytes, void *stream) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0 || window < 1) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_FP32) return GDN_ERR_INVALID_ARG;
    if (!supported_kv(K, V)) return GDN_ERR_UNSUPPORTED;
    if (!o && !S_T) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !beta)) return GDN_ERR_INVALID_ARG;
    if ((long long)B * H == 0) return GDN_OK;
    const size_t need = gdn_prefill_host_workspace_size(B, T, H, K, V, dtype, window);
    if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GDN_ERR_ALIGNMENT;
    return from_cuda(gdn::launch_prefill_host(q, k, v, alpha, beta, S0, o, S_T, B, T, H, K, V,
                                              dtype, window, workspace,
                                              static_cast<cudaStream_t>(stream)));
}

int gdn_state_rank(const float *S, int BH, int V, int K, float *fro2, float *sigma1,
                   float *stable_rank, int max_iter, float tol, void *stream) {
    if (BH < 0 || V < 1 || K < 1 || V > 128 || K > 128) return GDN_ERR_INVALID_ARG;
    if (max_iter < 1 || !(tol >= 0.f)) return GDN_ERR_INVALID_ARG;
    if (BH == 0) return GDN_OK;
    if (!S || !fro2 || !sigma1 || !stable_rank) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {S, fro2, sigma1, stable_rank};
    for (const void *p : ptrs)
        if (!aligned16(p)) return GDN_ERR_ALIGNMENT;
    return from_cuda(gdn::launch_state_rank(S, BH, V, K, fro2, sigma1, stable_rank, max_iter,
                                            tol, static_cast<cudaStream_t>(stream)));
}

int gdn_get_last_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GDN_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, gdn::g_device_status, sizeof(int)) != cudaSuccess)
        return GDN_ERR_CUDA;
    const int zero = 0;
    if (word != 0 && cudaMemcpyToSymbol(gdn::g_device_status, &zero, sizeof(int)) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (word & gdn::kStatusTimeout) return GDN_ERR_TIMEOUT;
    if (word & gdn::kStatusBounds) return GDN_ERR_DEVICE_BOUNDS;
    if (word & gdn::kStatusNotConverged) return GDN_WARN_NOT_CONVERGED;
    if (word & gdn::kStatusRankDeficient) return GDN_WARN_RANK_DEFICIENT;
    if (word & gdn::kStatusZeroState) return GDN_WARN_ZERO_STATE;
    return GDN_OK;
}

}  // extern "C"
