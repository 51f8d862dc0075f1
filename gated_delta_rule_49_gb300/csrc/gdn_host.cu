// Prefill on host-resident buffers: the runtime part that moves a step's
// inputs to the GPU and its results back while the recurrence runs.
//
// The sequence axis is cut into windows of `window` tokens.  For window w the
// host->device copy of q, k, v, alpha, beta (one strided 2-D copy per tensor,
// all batch entries at once) runs on an internal copy stream, the prefill of
// window w runs on the caller's stream from the state left by window w - 1
// (kept in device memory in float32), and the device->host copy of window w's
// outputs runs on a second internal copy stream.  Two window slots of device
// buffers alternate; events order every reuse:
//
//   h2d stream:      in(w)  ........ in(w+1) ...... in(w+2) [after compute(w)]
//   caller stream:   ...... compute(w) ....... compute(w+1) [after out(w-1)]
//   d2h stream:      .................. out(w) ......... out(w+1)
//
// so copies in both directions overlap the compute of neighbouring windows.
// With window a multiple of 64 the chunk boundaries are those of a single
// whole-sequence prefill and the results are identical to it.
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kMaxDev = 64;

struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t in_ready[2], in_free[2], out_ready[2], out_free[2], done, s0_ready;
    uintptr_t ctx = 0;  // the context the streams and events belong to (0: none yet)
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxDev];

cudaError_t pipe_for(int dev, HostPipe **out) {
    HostPipe &p = g_pipe[dev];
    // made once per device and context (a reset context invalidates the old
    // handles, which are then simply forgotten)
    if (p.ctx == 0 || p.ctx != context_key()) {
        p.ctx = 0;
        cudaError_t e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking);
        cudaEvent_t *evs[] = {&p.in_ready[0], &p.in_ready[1], &p.in_free[0], &p.in_free[1],
                              &p.out_ready[0], &p.out_ready[1], &p.out_free[0], &p.out_free[1],
                              &p.done, &p.s0_ready};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        p.ctx = context_key();
    }
    *out = &p;
    return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// Device bytes one window slot holds, and the whole workspace layout.
HostLayout host_layout(int B, int T, int H, int K, int V, gdn_dtype dt, int window) {
    HostLayout L{};
    const size_t esz = dt == GDN_BF16 ? 2 : 4;
    const size_t W = (size_t)window;
    L.q = 0;
    L.k = L.q + align256((size_t)B * W * H * K * esz);
    L.v = L.k + align256((size_t)B * W * H * K * esz);
    L.a = L.v + align256((size_t)B * W * H * V * esz);
    L.b = L.a + align256((size_t)B * W * H * 4);
    L.o = L.b + align256((size_t)B * W * H * 4);
    L.slot = L.o + align256((size_t)B * W * H * V * esz);
    L.state = 2 * L.slot;
    L.seg = L.state + align256((size_t)B * H * V * K * 4);
    L.seg_bytes = 0;
    if (dt == GDN_BF16 && V == 128 && (K == 128 || K == 64)) {
        const int tail = T % window;
        const int Ls[2] = {window < T ? window : T, tail};
        for (int n : Ls)
            if (n > 0) {
                const SegShape sh = segment_shape(B * H, n, K, sm_count());
                if (sh.workspace_bytes > L.seg_bytes) L.seg_bytes = sh.workspace_bytes;
            }
    }
    L.total = L.seg + align256(L.seg_bytes);
    return L;
}

cudaError_t launch_prefill_host(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *S0, void *o, float *ST, int B,
                                int T, int H, int K, int V, gdn_dtype dt, int window,
                                void *workspace, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pipe_mu);  // the internal streams and events
    HostPipe *P = nullptr;
    e = pipe_for(dev, &P);
    if (e != cudaSuccess) return e;
    const HostLayout L = host_layout(B, T, H, K, V, dt, window);
    char *ws = static_cast<char *>(workspace);
    float *Sdev = reinterpret_cast<float *>(ws + L.state);
    const size_t esz = dt == GDN_BF16 ? 2 : 4;
    const bool tc = dt == GDN_BF16 && V == 128 && (K == 128 || K == 64);
    const size_t sbytes = (size_t)B * H * V * K * 4;
#define GDN_TRY(x)                          \
    do {                                    \
        const cudaError_t e_ = (x);         \
        if (e_ != cudaSuccess) return e_;   \
    } while (0)

    // the caller's earlier work on `stream` comes first (it may have written
    // the host inputs through a device->host copy of its own)
    GDN_TRY(cudaEventRecord(P->done, stream));
    GDN_TRY(cudaStreamWaitEvent(P->h2d, P->done, 0));
    GDN_TRY(cudaStreamWaitEvent(P->d2h, P->done, 0));
    if (S0) {
        GDN_TRY(cudaMemcpyAsync(Sdev, S0, sbytes, cudaMemcpyHostToDevice, P->h2d));
        GDN_TRY(cudaEventRecord(P->s0_ready, P->h2d));
        GDN_TRY(cudaStreamWaitEvent(stream, P->s0_ready, 0));
    }
    if (T == 0 && !S0) GDN_TRY(cudaMemsetAsync(Sdev, 0, sbytes, stream));
    const int nwin = (T + window - 1) / window;
    for (int w = 0; w < nwin; ++w) {
        const int slot = w & 1;
        const int t0 = w * window;
        const int n = T - t0 < window ? T - t0 : window;
        char *base = ws + slot * L.slot;
        // ---- inputs of window w (the slot's previous prefill must be done) ----
        if (w >= 2) GDN_TRY(cudaStreamWaitEvent(P->h2d, P->in_free[slot], 0));
        struct Piece {
            size_t off;
            const void *src;
            size_t per_token;
        } in[] = {{L.q, q, (size_t)H * K * esz},
                  {L.k, k, (size_t)H * K * esz},
                  {L.v, v, (size_t)H * V * esz},
                  {L.a, alpha, (size_t)H * 4},
                  {L.b, beta, (size_t)H * 4}};
        for (const Piece &pc : in)
            GDN_TRY(cudaMemcpy2DAsync(base + pc.off, (size_t)window * pc.per_token,
                                      static_cast<const char *>(pc.src) + (size_t)t0 * pc.per_token,
                                      (size_t)T * pc.per_token, (size_t)n * pc.per_token, B,
                                      cudaMemcpyHostToDevice, P->h2d));
        GDN_TRY(cudaEventRecord(P->in_ready[slot], P->h2d));
        // ---- the recurrence over window w on the caller's stream ----
        GDN_TRY(cudaStreamWaitEvent(stream, P->in_ready[slot], 0));
        if (w >= 2 && o) GDN_TRY(cudaStreamWaitEvent(stream, P->out_free[slot], 0));
        const float *start = (w == 0) ? (S0 ? Sdev : nullptr) : Sdev;
        void *ow = o ? base + L.o : nullptr;
        if (tc)
            e = launch_prefill_tc(base + L.q, base + L.k, base + L.v,
                                  reinterpret_cast<const float *>(base + L.a),
                                  reinterpret_cast<const float *>(base + L.b), start, ow, Sdev, B,
                                  n, window, H, K, V, L.seg_bytes ? ws + L.seg : nullptr,
                                  L.seg_bytes, stream);
        else
            e = launch_prefill_gated(base + L.q, base + L.k, base + L.v,
                                     reinterpret_cast<const float *>(base + L.a),
                                     reinterpret_cast<const float *>(base + L.b), nullptr, nullptr,
                                     start, ow, Sdev, B, n, window, H, K, V, GDN_GATE_SCALAR, dt,
                                     stream);
        if (e != cudaSuccess) return e;
        GDN_TRY(cudaEventRecord(P->in_free[slot], stream));
        // ---- outputs of window w ----
        if (o) {
            GDN_TRY(cudaEventRecord(P->out_ready[slot], stream));
            GDN_TRY(cudaStreamWaitEvent(P->d2h, P->out_ready[slot], 0));
            const size_t per = (size_t)H * V * esz;
            GDN_TRY(cudaMemcpy2DAsync(static_cast<char *>(o) + (size_t)t0 * per, (size_t)T * per,
                                      base + L.o, (size_t)window * per, (size_t)n * per, B,
                                      cudaMemcpyDeviceToHost, P->d2h));
            GDN_TRY(cudaEventRecord(P->out_free[slot], P->d2h));
        }
    }
    // ---- final state, then the caller's stream waits for every copy ----
    GDN_TRY(cudaEventRecord(P->done, stream));
    GDN_TRY(cudaStreamWaitEvent(P->d2h, P->done, 0));
    if (ST) GDN_TRY(cudaMemcpyAsync(ST, Sdev, sbytes, cudaMemcpyDeviceToHost, P->d2h));
    GDN_TRY(cudaEventRecord(P->done, P->d2h));
    GDN_TRY(cudaStreamWaitEvent(stream, P->done, 0));
#undef GDN_TRY
    return cudaSuccess;
}

}  // namespace gdn
