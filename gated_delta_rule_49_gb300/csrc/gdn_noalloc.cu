// gdn_prefill_noalloc: gdn_prefill for callers that cannot allocate device
// memory.  The scratch that the segment-parallel prefill needs lives in one
// file-scope device array of fixed size instead of a caller-supplied buffer.
#include <mutex>

#include "gdn_internal.cuh"

namespace {

// Scratch for gdn_prefill_noalloc.  Every GPU that loads the library holds
// these 32 MiB until the process exits.  In host code `g_noalloc_scratch` is
// only a host-side stand-in for the symbol, never a device address: the
// address is looked up per device with cudaGetSymbolAddress below.  Under
// CUDA's default lazy module loading the array is only materialised on a
// device when the first call there looks its address up (a driver allocation
// that may synchronise); a caller that must not allocate after start-up makes
// one small call per device at start-up.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDev];
uintptr_t g_scratch_ctx[kMaxDev];  // the context the address belongs to

// Device address of the scratch array on the current device (looked up once
// per device and context, with that device current), or nullptr on failure.
void *scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    const uintptr_t ctx = gdn::context_key();
    if (!g_scratch_ptr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = gdn::context_key();  // current now that the lookup ran
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" size_t gdn_prefill_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

extern "C" int gdn_prefill_noalloc(const void *q, const void *k, const void *v,
                                   const float *alpha, const float *beta, const float *S0,
                                   void *o, float *S_T, int B, int T, int H, int K, int V,
                                   gdn_dtype dtype, void *stream) {
    const size_t need = gdn_prefill_workspace_size(B, T, H, K, V, dtype);
    if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;
    const size_t two_pass = gdn_prefill_two_pass_workspace_size(B, T, H, K, V, dtype);
    const bool use = need > 0 || (two_pass > 0 && two_pass <= kNoAllocScratchBytes);
    void *ws = nullptr;
    if (use) {
        ws = scratch_address();
        if (!ws) return GDN_ERR_CUDA;
    }
    // Every byte of the scratch that the prefill reads is written earlier in
    // the same call, so nothing has to be cleared between calls.
    return gdn_prefill(q, k, v, alpha, beta, S0, o, S_T, B, T, H, K, V, dtype, ws,
                       use ? kNoAllocScratchBytes : 0, stream);
}
