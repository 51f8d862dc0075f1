/*
 * gdn.h -- C ABI of libgdn.so: the gated delta-rule recurrence on one GPU.
 *
 * The recurrence (per batch element b and head h, state S in R^{V x K}):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t
 *
 * equivalently: decay the old state first, form the error of its prediction
 * u_t = beta_t (v_t - alpha_t S_{t-1} k_t), write u_t k_t^T, then read with
 * the query.  Sources: "On State Reduction in Linear Attention" reading notes,
 * Sec. 2.1, Eqs. (1)-(2) (DeltaNet update in error-correction form, the read
 * o_t = S_t q_t, Gated DeltaNet's scalar decay) and "Linear Attention
 * Architectures" reading notes, Sec. 2.4, Eqs. 15-17 (decay before the error).
 * A channel-pruned state keeps d_k' of the key/query channels ("On State
 * Reduction" notes, Sec. 2.6): callers pass the gathered, re-normalised
 * q/k with K = d_k'.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller, dense and
 *    row-major, each 16-byte aligned (else GDN_ERR_ALIGNMENT).  The library
 *    never allocates device memory in these calls.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronise, except
 *    gdn_get_last_device_status.
 *  - Arguments are validated on the host before any launch; a rejected call
 *    launches nothing.  A failed launch returns GDN_ERR_CUDA.  No entry point
 *    calls exit(), traps or asserts on the device.
 *  - Supported (K, V) pairs: (32, 32), (64, 128), (128, 128); others return
 *    GDN_ERR_UNSUPPORTED.  K is d_k (or a pruned d_k'), V is d_v.
 *  - State tensors, alpha and beta are always float32; q, k, v and o are
 *    bf16 (GDN_BF16) or float32 (GDN_FP32).  Arithmetic is float32 with the
 *    state carried in float32; in GDN_BF16 mode at V = 128 the prefill runs
 *    the chunk form on the tensor cores (bf16 operands, float32 accumulation),
 *    otherwise it runs token by token on the CUDA cores.
 *  - alpha is expected in (0, 1] and beta in [0, 2); values are not checked.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad dtype, ... */
    GDN_ERR_UNSUPPORTED = -2,   /* (K, V) not a compiled variant, or no sm_103 device */
    GDN_ERR_ALIGNMENT = -3,     /* a pointer is not 16-byte aligned */
    GDN_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
    GDN_ERR_TIMEOUT = -5,       /* device status: a bounded wait in a kernel gave up */
    GDN_ERR_WORKSPACE = -6,     /* workspace missing or smaller than required */
    GDN_ERR_DEVICE_BOUNDS = -7, /* device status: a kernel's own index check failed */
    GDN_WARN_ZERO_STATE = 1,    /* device status: gdn_state_rank saw an all-zero state */
    GDN_WARN_NOT_CONVERGED = 2, /* device status: gdn_state_truncate hit max_sweeps */
    GDN_WARN_RANK_DEFICIENT = 3 /* device status: gdn_drrqr_select saw rank(M) < k */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_FP32 = 1 } gdn_dtype;

/*
 * gdn_prefill -- run the recurrence over T tokens of every (b, h) sequence.
 *
 *   q, k   [B, T, H, K] (dtype)      v  [B, T, H, V] (dtype)
 *   alpha, beta [B, T, H] float32    S0 [B, H, V, K] float32, or NULL = zero
 *   o      [B, T, H, V] (dtype), or NULL to skip the outputs
 *   S_T    [B, H, V, K] float32, or NULL to skip the final state; S_T may be
 *          the same pointer as S0 (in-place continuation)
 *
 * Chunkwise-parallel form with 64-token chunks: within a chunk the
 * pseudo-values u_t solve a unit lower-triangular system (the UT/WY
 * transform), the chunk-local products run as matrix products, and the
 * state is carried from chunk to chunk in float32.  Any T >= 0 is accepted
 * (a ragged last chunk is masked; T = 0 copies S0, or zero, into S_T).
 * B = 0 or H = 0 is a no-op.
 *
 * workspace: device scratch of at least gdn_prefill_workspace_size() bytes
 * (may be NULL when that size is 0); 256-byte aligned.  With at least
 * gdn_prefill_two_pass_workspace_size() bytes the bf16 tensor-core path runs
 * in two passes: first the state-independent part of every chunk (A, the
 * triangular inverse) for all chunks of all sequences at once, then the
 * state recurrence, which only loads those operands.  For whole sequences
 * the results are bit-identical to the one-pass form; only the speed
 * differs.  Segment-parallel problems (few, long sequences) take another
 * route there: every segment's outputs from a zero start and the map x of
 * its start state, then o += S_start x and the end state from the chain of
 * segment maps, instead of a second pass over the segments; those results
 * agree with the one-pass form to rounding (a bf16 step of o, the float32
 * chain of S_T).
 */
GDN_API int gdn_prefill(const void *q, const void *k, const void *v, const float *alpha,
                const float *beta, const float *S0, void *o, float *S_T, int B, int T, int H,
                int K, int V, gdn_dtype dtype, void *workspace, size_t workspace_bytes,
                void *stream);

/* Bytes of device workspace gdn_prefill needs for this problem (0 if none). */
GDN_API size_t gdn_prefill_workspace_size(int B, int T, int H, int K, int V, gdn_dtype dtype);

/* Bytes of device workspace with which gdn_prefill takes the two-pass form:
 * the segment scratch of gdn_prefill_workspace_size (rounded up to 256 bytes)
 * plus 16 KiB per 64-token chunk per (b, h) for the key-side operands, plus,
 * for segment-parallel problems, B*T*H*128 bf16 (rounded up to 256 bytes)
 * for the segments' maps x.  With the operands only (no x buffer) a
 * segment-parallel call that wants o runs the second pass like the one-pass
 * form.
 * 0 when the problem has no two-pass form (float32, or V != 128, or
 * K not in {64, 128}). */
GDN_API size_t gdn_prefill_two_pass_workspace_size(int B, int T, int H, int K, int V,
                                                   gdn_dtype dtype);

/*
 * gdn_prefill_noalloc -- gdn_prefill for callers that cannot allocate device
 * memory: for example a component that only receives device pointers from the
 * framework that owns the GPU's memory, or a server that reserves all of its
 * memory at start-up and must not call cudaMalloc afterwards (an allocation can
 * synchronise the device and its size is not known in advance).  The pages
 * have no counterpart; this is a deployment convenience of this library.
 *
 * Same arguments, results and errors as gdn_prefill, without the workspace:
 * the scratch that the segment-parallel path needs (see
 * gdn_prefill_workspace_size) comes from one 32 MiB array compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  A problem that needs more scratch than that returns
 * GDN_ERR_WORKSPACE before anything is launched.  Problems whose two-pass
 * workspace fits in the array take the two-pass form.  The call allocates
 * nothing.
 *
 *  - The first call on a device that needs scratch looks up the array's
 *    device address (cudaGetSymbolAddress) with that device current; make
 *    that first call before any stream capture.  Under CUDA's default lazy
 *    module loading that lookup is also when the driver materialises the
 *    array on the device (an allocation that may synchronise): a caller
 *    that must not allocate after start-up makes one small call per device
 *    at start-up.
 *  - The address is cached per device and per CUDA context (looked up again
 *    when another context is current, e.g. after cudaDeviceReset).
 *  - All calls on a device share the one array, and it keeps the contents of
 *    the last call.  Nothing needs clearing (each call writes every scratch
 *    value it reads), but calls that may overlap on the GPU -- on different
 *    streams, or from several host threads -- race on the scratch: order them
 *    on one stream or serialise them.
 */
GDN_API int gdn_prefill_noalloc(const void *q, const void *k, const void *v, const float *alpha,
                                const float *beta, const float *S0, void *o, float *S_T, int B,
                                int T, int H, int K, int V, gdn_dtype dtype, void *stream);

/* Scratch bytes available to gdn_prefill_noalloc (the size of its array). */
GDN_API size_t gdn_prefill_noalloc_max_workspace(void);

/*
 * gdn_prefill_gathered -- gdn_prefill on a channel-pruned state, from the
 * full-width q and k: the pruning prologue (the formula of
 * gdn_gather_normalize, below) runs inside the key-side pass of the two-pass
 * prefill, which loads the full-width q/k rows, keeps and renormalises
 * channels idx[h, :] on chip for its own products, and leaves the gathered
 * q', k' in the workspace for the state pass; there is no separate pass over
 * q and k ("On State Reduction" notes, Sec. 2.6 and Alg. 1: pruning is
 * deployed as a gather on the projection path).
 *
 *   q_full, k_full [B, T, H, K_in] bf16, K_in = 128
 *   idx            [H, K] int32 kept channels in [0, K_in), K = 64
 *   v, alpha, beta, S0, o, S_T: as for gdn_prefill with K = 64, V = 128
 *   workspace      >= gdn_prefill_gathered_workspace_size(B, T, H, K_in, K, V,
 *                  dtype) bytes, 16-byte aligned, caller-owned device memory
 *
 * Results are bit-identical to gdn_gather_normalize on q and k followed by
 * gdn_prefill with its two-pass workspace.  Other (K_in, K, V) or float32
 * return GDN_ERR_UNSUPPORTED; a missing or short workspace GDN_ERR_WORKSPACE.
 * An index outside [0, K_in) is not read: it contributes 0 and sets the
 * GDN_ERR_DEVICE_BOUNDS device status.
 */
GDN_API int gdn_prefill_gathered(const void *q_full, const void *k_full, const int *idx, int K_in,
                                 const void *v, const float *alpha, const float *beta,
                                 const float *S0, void *o, float *S_T, int B, int T, int H, int K,
                                 int V, gdn_dtype dtype, void *workspace, size_t workspace_bytes,
                                 void *stream);

/* Workspace bytes of gdn_prefill_gathered (0 for an unsupported shape). */
GDN_API size_t gdn_prefill_gathered_workspace_size(int B, int T, int H, int K_in, int K, int V,
                                                   gdn_dtype dtype);

/*
 * gdn_decode_step -- one token of the recurrence for every (b, h), with the
 * state updated in place:
 *
 *   q, k [B, H, K] (dtype)   v [B, H, V] (dtype)   alpha, beta [B, H] float32
 *   S    [B, H, V, K] float32, read once and written once
 *   o    [B, H, V] (dtype)
 *
 * Each value channel (row of S) is an independent system ("On State
 * Reduction" notes, Sec. 2.5), so a row is decayed, dotted with k and q,
 * corrected and written back in one pass.
 */
GDN_API int gdn_decode_step(const void *q, const void *k, const void *v, const float *alpha,
                    const float *beta, float *S, void *o, int B, int H, int K, int V,
                    gdn_dtype dtype, void *stream);

/*
 * gdn_gather_normalize -- the pruning prologue: keep d_k' of the d_k
 * key/query channels of every head and recompute the L2 normalisation on
 * the kept coordinates ("On State Reduction" notes, Sec. 2.6 and Alg. 1):
 *
 *     y[n, h, :] = x[n, h, idx[h, :]] / max(|x[n, h, idx[h, :]]|, 1e-12)
 *
 *   x   [N, H, K_in] (dtype), N = B * T rows per head (any scale: a full-width
 *       normalisation before this call changes nothing)
 *   idx [H, K_out] int32 channel indices in [0, K_in) (any order)
 *   y   [N, H, K_out] (dtype), K_out in {32, 64}, K_out <= K_in <= 1024
 *
 * An index outside [0, K_in) is not read; it contributes 0 and sets the
 * GDN_ERR_DEVICE_BOUNDS device status.  Use it to feed gdn_prefill the pruned
 * q and k from full-width projections.
 */
GDN_API int gdn_gather_normalize(const void *x, const int *idx, void *y, long long N, int H,
                                 int K_in, int K_out, gdn_dtype dtype, void *stream);

/*
 * gdn_decode_step_gathered -- gdn_decode_step on a channel-pruned state that
 * reads full-width q and k and applies the pruning prologue inside the step
 * (same formula as gdn_gather_normalize, no separate pass):
 *
 *   q_full, k_full [B, H, K_in] (dtype); idx [H, K] int32; K <= K_in <= 1024
 *   v [B, H, V]; alpha, beta [B, H]; S [B, H, V, K] updated in place; o [B, H, V]
 *
 * (K, V) as for gdn_decode_step.  Bad indices as for gdn_gather_normalize.
 */
GDN_API int gdn_decode_step_gathered(const void *q_full, const void *k_full, const int *idx,
                                     int K_in, const void *v, const float *alpha,
                                     const float *beta, float *S, void *o, int B, int H, int K,
                                     int V, gdn_dtype dtype, void *stream);

/*
 * gdn_prefill_host -- gdn_prefill on HOST-resident buffers (pinned host
 * memory for the copies to overlap; pageable memory works, serialised).
 * The sequence axis is cut into windows of `window` tokens; the host->device
 * copy of window w + 1, the prefill of window w (on `stream`, from the
 * float32 state left by window w - 1) and the device->host copy of window
 * w - 1's outputs run concurrently, on two internal copy streams and `stream`.
 *
 *   q, k, v, alpha, beta, S0, o, S_T: host pointers, same shapes and dtypes as
 *     gdn_prefill (S0 may be NULL; o or S_T may be NULL, not both)
 *   window: tokens per pipeline stage (>= 1; a multiple of 64 gives results
 *     identical to gdn_prefill on device copies of the same inputs)
 *   workspace: DEVICE memory of gdn_prefill_host_workspace_size(...) bytes,
 *     16-byte aligned (two window slots, the state and the prefill's scratch)
 *
 * Asynchronous with respect to the host like every call here: the host
 * buffers must stay valid, and the outputs are complete, once `stream` has
 * reached the point after this call (cudaStreamSynchronize(stream)).
 * Concurrent calls on one device are serialised while they enqueue.
 */
GDN_API size_t gdn_prefill_host_workspace_size(int B, int T, int H, int K, int V,
                                               gdn_dtype dtype, int window);
GDN_API int gdn_prefill_host(const void *q, const void *k, const void *v, const float *alpha,
                             const float *beta, const float *S0, void *o, float *S_T, int B,
                             int T, int H, int K, int V, gdn_dtype dtype, int window,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Gates of the channel-gated delta rules ("Linear Attention Architectures"
 * reading notes, Secs. 2.4-2.6).  Per token and head, S in R^{V x K}:
 *
 *   GDN_GATE_SCALAR  Gated DeltaNet: S <- a S; u = beta (v - S k)
 *                    alpha, beta [.., H]
 *   GDN_GATE_KDA     Kimi Delta Attention: the decay acts per key channel, on
 *                    the right of the state: S <- S diag(alpha); u = beta (v - S k)
 *                    alpha [.., H, K], beta [.., H]
 *   GDN_GATE_GDN2    Gated DeltaNet-2: separate erase (key side) and write
 *                    (value side) gates: S <- S diag(alpha); u = w (.) v - S (b (.) k)
 *                    alpha, b [.., H, K], w [.., H, V]
 *
 * then, for all three, S <- S + u k^T and o = S q (the write keeps the
 * original key on its right).  alpha = a 1 turns KDA into GDN; b = w = beta 1
 * turns GDN2 into KDA.
 */
typedef enum { GDN_GATE_SCALAR = 0, GDN_GATE_KDA = 1, GDN_GATE_GDN2 = 2 } gdn_gate;

/*
 * gdn_prefill_gated -- the recurrence over T tokens under any of the gates
 * above, token by token on the CUDA cores (value rows split across CTAs).
 *
 *   q, k [B, T, H, K], v [B, T, H, V] (dtype);  o [B, T, H, V] (dtype)
 *   alpha [B, T, H] (SCALAR) or [B, T, H, K] (KDA, GDN2), float32
 *   beta [B, T, H] float32 (SCALAR, KDA; must be NULL for GDN2)
 *   b [B, T, H, K], w [B, T, H, V] float32 (GDN2; must be NULL otherwise)
 *   S0 [B, H, V, K] float32 or NULL (zero state);  S_T [B, H, V, K] float32
 *
 * (K, V) as for gdn_prefill; any T >= 0 (T = 0 copies S0, or zeros, into
 * S_T).  o or S_T may be NULL (not both); S_T may alias S0.  Needs no
 * workspace.  Host validation as for gdn_prefill.
 */
GDN_API int gdn_prefill_gated(const void *q, const void *k, const void *v, const float *alpha,
                              const float *beta, const float *b, const float *w,
                              const float *S0, void *o, float *S_T, int B, int T, int H, int K,
                              int V, gdn_gate gate, gdn_dtype dtype, void *stream);

/*
 * gdn_prefill_gated_chunked -- gdn_prefill_gated for KDA and GDN2 in the
 * chunkwise form on the tensor cores: 64-token chunks, a key-side pass over
 * every chunk of every sequence at once (the per-channel gate prefix; the
 * intra-chunk products A and P with each 16-token row block's exponents
 * referred to its midpoint, so every factor stays below e^(8 max |log alpha|);
 * the triangular inverse; W), then one CTA per sequence carrying the float32
 * state ("Linear Attention Architectures" notes, Secs. 2.5-2.6; the
 * pseudo-value form of "On State Reduction" notes, Sec. 2.3).  Arguments as
 * for gdn_prefill_gated, plus
 *
 *   workspace  >= gdn_prefill_gated_chunked_workspace_size(...) bytes,
 *              16-byte aligned, caller-owned device memory (about 64.5 KiB
 *              per 64-token chunk per (b, h) for KDA, 80.5 KiB for GDN2)
 *   b, w       (GDN2) 16-byte aligned, like q, k and v
 *
 * For GDN2 the call forks one elementwise kernel (w (.) v into the
 * workspace) onto a stream of the library's own, one per device, and joins
 * it back into `stream` before the state pass: work on `stream` stays
 * ordered as usual, and stream capture records the fork and the join.
 *
 * Supported: gate KDA or GDN2, K = V = 128, bf16; anything else returns
 * GDN_ERR_UNSUPPORTED (gdn_prefill_gated covers it token by token).  The
 * operands of the tensor-core products are bf16 (float32 accumulation, the
 * inverse and the state in float32), so results agree with gdn_prefill_gated
 * to the bf16 operand rounding, not bit for bit.  o or S_T may be NULL (not
 * both); S_T may alias S0.  A missing or short workspace returns
 * GDN_ERR_WORKSPACE.
 */
GDN_API int gdn_prefill_gated_chunked(const void *q, const void *k, const void *v,
                                      const float *alpha, const float *beta, const float *b,
                                      const float *w, const float *S0, void *o, float *S_T,
                                      int B, int T, int H, int K, int V, gdn_gate gate,
                                      gdn_dtype dtype, void *workspace, size_t workspace_bytes,
                                      void *stream);

/* Workspace bytes of gdn_prefill_gated_chunked (0 where it has no form). */
GDN_API size_t gdn_prefill_gated_chunked_workspace_size(int B, int T, int H, int K, int V,
                                                        gdn_gate gate, gdn_dtype dtype);

/*
 * gdn_decode_step_gated -- one token of gdn_prefill_gated on a state updated
 * in place:  q, k [B, H, K]; v, o [B, H, V]; alpha [B, H] or [B, H, K];
 * beta [B, H]; b [B, H, K]; w [B, H, V]; S [B, H, V, K].  Which gates must be
 * given (and which must be NULL) as for gdn_prefill_gated.
 */
GDN_API int gdn_decode_step_gated(const void *q, const void *k, const void *v,
                                  const float *alpha, const float *beta, const float *b,
                                  const float *w, float *S, void *o, int B, int H, int K, int V,
                                  gdn_gate gate, gdn_dtype dtype, void *stream);

/*
 * gdn_state_rank -- stable rank of BH states ("On State Reduction" notes,
 * Sec. 2.2, Eq. (5)): er(S) = ||S||_F^2 / ||S||_2^2.
 *
 *   S [BH, V, K] float32 (1 <= V, K <= 128)
 *   fro2, sigma1, stable_rank [BH] float32 outputs: ||S||_F^2, sigma_1, er
 *
 * sigma_1^2 is the largest eigenvalue of S^T S by power iteration from the
 * fixed start x_j = 1 + j/K: the Rayleigh quotient is checked every 4
 * products of S^T S with the iterate, and the iteration stops when it changes
 * by at most tol (relative) between checks or after max_iter products
 * (max_iter >= 1, tol >= 0).  An all-zero state yields 0 in all three outputs
 * and sets the GDN_WARN_ZERO_STATE device status.
 */
GDN_API int gdn_state_rank(const float *S, int BH, int V, int K, float *fro2, float *sigma1,
                   float *stable_rank, int max_iter, float tol, void *stream);

/*
 * gdn_state_truncate -- rank-r truncation of BH states, in place ("How much
 * of a Gated DeltaNet state is used" blog, Sec. 3): each state is projected
 * onto its top-r left singular directions,
 *
 *     S <- U_r U_r^T S      (the best rank-r approximation of S),
 *
 * and, if `sigma` is given, its singular values are written in descending
 * order.
 *
 *   S     [BH, V, K] float32, (K, V) one of the supported variants
 *   r     >= 1; r >= min(V, K) leaves S unchanged
 *   sigma [BH, min(V, K)] float32 or NULL
 *   max_sweeps  1..1000 one-sided Jacobi sweeps (about 6-10 reach float32
 *         orthogonality); stopping there sets GDN_WARN_NOT_CONVERGED
 *
 * Where sigma_r == sigma_{r+1} the kept subspace is not unique; the result is
 * then one of the equally good truncations.
 */
GDN_API int gdn_state_truncate(float *S, int BH, int V, int K, int r, float *sigma,
                               int max_sweeps, void *stream);

/*
 * gdn_prefill_truncated -- the same blog section's experiment: the prefill
 * run in segments of seg_len tokens, the carried state truncated to rank r
 * (gdn_state_truncate) at every segment boundary inside the sequence.  The
 * final state S_T is not truncated, nor is S0.
 *
 * Arguments as for gdn_prefill, with S_T required (it carries the state
 * between segments; it may alias S0) and a workspace as
 * gdn_prefill_workspace_size reports for B, min(seg_len, T) and for the
 * last, shorter segment (0 for the usual shapes).  seg_len >= 1, r >= 1,
 * max_sweeps as for gdn_state_truncate.
 */
GDN_API int gdn_prefill_truncated(const void *q, const void *k, const void *v,
                                  const float *alpha, const float *beta, const float *S0,
                                  void *o, float *S_T, int B, int T, int H, int K, int V,
                                  gdn_dtype dtype, int seg_len, int r, int max_sweeps,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * DRRQR channel selection ("On State Reduction in Linear Attention" notes,
 * Sec. 2.8): pick d_k' = k of the d_k = n key/query channels of every head so
 * that the kept columns of the calibration matrix M_h = [K_cal; Q_cal]
 * (tokens as rows) form a well-conditioned basis.
 *
 * gdn_channel_gram -- G_h = K_h^T K_h + Q_h^T Q_h = M_h^T M_h (the QR's R
 *   satisfies R^T R = G), summed over the calibration tokens on the tensor
 *   cores:  k, q [B, T, H, 128] bf16 (the activations as the layer feeds them
 *   to the recurrence);  G [H, 128, 128] float32 output.  Needs a workspace of
 *   gdn_channel_gram_workspace_size(B, T, H, K) bytes.  Only K = 128 and bf16
 *   (GDN_ERR_UNSUPPORTED otherwise).  B * T = 0 gives G = 0.
 */
GDN_API size_t gdn_channel_gram_workspace_size(int B, int T, int H, int K);
GDN_API int gdn_channel_gram(const void *k, const void *q, int B, int T, int H, int K,
                             gdn_dtype dtype, float *G, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * gdn_drrqr_select -- per head, column-pivoted QR of M (through the pivoted
 *   Cholesky factorisation of G) for the initial permutation, then
 *   strong-RRQR swaps of a kept and a candidate channel while
 *   max rho_ij = sqrt(U_ij^2 + (gamma_j / omega_i)^2) > f, with U = A_k^{-1} B_k,
 *   omega_i = 1 / |row i of A_k^{-1}|, gamma_j = |column j of C_k|.
 *
 *   G [H, n, n] float32 (from gdn_channel_gram, or any symmetric PSD matrix)
 *   2 <= n <= 128, 1 <= k < n;  f >= 1;  0 <= max_swaps
 *   idx [H, k] int32 output: the kept channels in selection order
 *   rho_max [H] float32 (final max rho) and swaps [H] int32, each optional
 *
 * At the end every rho_ij <= f (unless max_swaps stopped it), which gives the
 * notes' bounds with c_f = sqrt(1 + f^2 k (n - k)).  If rank(M) < k (a pivot of
 * G below 1e-6 of its largest diagonal entry, i.e. sigma_k below about 1e-3
 * sigma_1) the greedy choice is returned without swaps and
 * GDN_WARN_RANK_DEFICIENT is set.
 * Computed in float32: near-ties (equal pivots or rho values) may be broken
 * differently from a float64 computation; any such result satisfies the same
 * stopping test to float32 accuracy.
 */
GDN_API int gdn_drrqr_select(const float *G, int H, int n, int k, float f, int max_swaps,
                             int *idx, float *rho_max, int *swaps, void *stream);

/*
 * gdn_get_last_device_status -- synchronise `stream`, then read and clear the
 * current device's status word.  Returns GDN_OK, GDN_ERR_TIMEOUT,
 * GDN_ERR_DEVICE_BOUNDS, GDN_WARN_NOT_CONVERGED, GDN_WARN_RANK_DEFICIENT or
 * GDN_WARN_ZERO_STATE (warnings
 * only when no error is set) or
 * GDN_ERR_CUDA if the synchronisation itself failed.
 */
GDN_API int gdn_get_last_device_status(void *stream);

/*
 * gdn_selftest_wait_timeout -- exercise the bounded wait that every mbarrier
 * wait of the tensor-core prefill goes through.  One thread of one CTA waits
 * on a shared-memory barrier that nothing ever completes, gives up after
 * limit_cycles SM clock cycles (1 <= limit_cycles <= 2^31), sets the timeout
 * bit of the device status word and returns; the context stays usable.
 * Asynchronous on `stream`; read the outcome with gdn_get_last_device_status
 * (GDN_ERR_TIMEOUT).  Meant for tests of the failure-detection path.
 */
GDN_API int gdn_selftest_wait_timeout(long long limit_cycles, void *stream);

/* Static, NUL-terminated description of a status code. */
GDN_API const char *gdn_status_string(int status);

/* Library ABI version (major * 100 + minor). */
GDN_API int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
